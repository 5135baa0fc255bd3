// warp_mma.cuh -- warp-level tensor-core helpers (ldmatrix, bf16 and tf32 mma.sync) shared by
// the kernels that stage small bf16 tiles in shared memory with padded rows.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace kla {
namespace wmma16 {

__device__ __forceinline__ uint32_t sptr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// bf16 pairs <-> fp32 (round to nearest even)
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float2 unpack2(uint32_t u) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(h);
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// One 16 x 8 tile of A B in fp32 shared memory (tf32 operands, fp32 accumulate): A rows
// [ar, ar+16) x columns [ac, ac+8*KS) of a matrix with pitch pa; B rows [br, br+8*KS) x columns
// [bc, bc+8) with pitch pb.
template <int KS>
__device__ __forceinline__ void tile_tf32(float (&acc)[4], const float *A, int pa, int ar, int ac, const float *Bm,
                                          int pb, int br, int bc, int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const float *a0 = A + (ar + g) * pa + ac + 8 * ks + q;
        const uint32_t a[4] = {tf32(a0[0]), tf32(a0[8 * pa]), tf32(a0[4]), tf32(a0[8 * pa + 4])};
        const float *b0 = Bm + (br + 8 * ks + q) * pb + bc + g;
        mma_tf32(acc, a, tf32(b0[0]), tf32(b0[4 * pb]));
    }
}
// Operand fragments of a 16 x 16 (A: rows x k) or 16 x 16 (B: k x two n8 tiles) block of a
// bf16 tile at shared address `t` with row pitch `pitch` elements. The suffix names how the
// tile stores the operand: _rk = [row][k] for A or [n][k] for B (no transpose); _kr = [k][row]
// for A or [k][n] for B (ldmatrix.trans).
__device__ __forceinline__ void frag_a_rk(uint32_t t, int pitch, int r0, int k0, int lane, uint32_t (&a)[4]) {
    const int m = lane >> 3;
    ldsm4(t + 2 * ((r0 + (lane & 7) + (m & 1) * 8) * pitch + k0 + (m >> 1) * 8), a);
}
__device__ __forceinline__ void frag_a_kr(uint32_t t, int pitch, int r0, int k0, int lane, uint32_t (&a)[4]) {
    const int m = lane >> 3;
    ldsm4t(t + 2 * ((k0 + (lane & 7) + (m >> 1) * 8) * pitch + r0 + (m & 1) * 8), a);
}
// b[0], b[1]: n-tile n0; b[2], b[3]: n-tile n0 + 8
__device__ __forceinline__ void frag_b_rk(uint32_t t, int pitch, int n0, int k0, int lane, uint32_t (&b)[4]) {
    const int m = lane >> 3;
    ldsm4(t + 2 * ((n0 + (lane & 7) + (m >> 1) * 8) * pitch + k0 + (m & 1) * 8), b);
}
__device__ __forceinline__ void frag_b_kr(uint32_t t, int pitch, int n0, int k0, int lane, uint32_t (&b)[4]) {
    const int m = lane >> 3;
    ldsm4t(t + 2 * ((k0 + (lane & 7) + (m & 1) * 8) * pitch + n0 + (m >> 1) * 8), b);
}
}  // namespace wmma16
}  // namespace kla
