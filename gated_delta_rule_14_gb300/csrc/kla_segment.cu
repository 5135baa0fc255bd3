// kla_segment.cu -- start states of the segments of a long sequence (sequence-parallel scan).
//
// The recurrence is affine in the state: over a segment, S_end = M S_start + Z, where Z is the
// segment's final state from S_start = 0 and M (d_k x d_k) its final state from S_start = I
// with v = 0 (every token applies S -> (D - beta k (D k)^T) S + beta k v^T; GeekNews,
// "Revisando las variantes de atencion lineal de la familia DeltaNet", section "Transicion
// diagonal-bajo rango"). Given Z_s and M_s of the segments of one chain, the true start states
// follow by a short serial pass:
//     S_start[1] = Z_0 (segment 0 already started from the true initial state),
//     S_start[s + 1] = M_s S_start[s] + Z_s.
// One CTA per (sequence, head) chain runs that pass in fp32; the 128 x 128 products are tiled
// through shared memory (M transposed so both operands are read as contiguous float4).
#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr int kLdA = kD + 4;   // padded row of M^T in shared memory

__global__ void __launch_bounds__(kThreads) seg_combine_kernel(const float *Z, const float *M, float *Sst,
                                                               int nseg) {
    extern __shared__ __align__(16) float csm[];
    float *At = csm;                 // M^T: [k][i], row stride kLdA
    float *X = csm + kD * kLdA;      // current start state [k][j]
    const int tid = threadIdx.x;
    const size_t chain = blockIdx.x;
    const size_t dd = static_cast<size_t>(kD) * kD;
    const float *Zc = Z + chain * nseg * dd, *Mc = M + chain * nseg * dd;
    float *Sc = Sst + chain * nseg * dd;

    for (int idx = tid; idx < kD * kD / 4; idx += kThreads) {   // S_start[1] = Z_0
        const float4 z = reinterpret_cast<const float4 *>(Zc)[idx];
        reinterpret_cast<float4 *>(X)[idx] = z;
        reinterpret_cast<float4 *>(Sc + dd)[idx] = z;
    }
    const int i0 = (tid >> 4) * 8, j0 = (tid & 15) * 8;
    for (int s = 1; s + 1 < nseg; ++s) {
        __syncthreads();
        const float *Ms = Mc + s * dd;
        for (int idx = tid; idx < kD * kD; idx += kThreads) {
            const int i = idx >> 7, k = idx & (kD - 1);
            At[k * kLdA + i] = Ms[idx];
        }
        __syncthreads();
        float acc[8][8];
        const float *Zs = Zc + s * dd;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float4 a = *reinterpret_cast<const float4 *>(Zs + (i0 + r) * kD + j0);
            const float4 b = *reinterpret_cast<const float4 *>(Zs + (i0 + r) * kD + j0 + 4);
            acc[r][0] = a.x; acc[r][1] = a.y; acc[r][2] = a.z; acc[r][3] = a.w;
            acc[r][4] = b.x; acc[r][5] = b.y; acc[r][6] = b.z; acc[r][7] = b.w;
        }
        for (int k = 0; k < kD; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(At + k * kLdA + i0);
            const float4 a1 = *reinterpret_cast<const float4 *>(At + k * kLdA + i0 + 4);
            const float4 x0 = *reinterpret_cast<const float4 *>(X + k * kD + j0);
            const float4 x1 = *reinterpret_cast<const float4 *>(X + k * kD + j0 + 4);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(av[r], xv[c], acc[r][c]);
        }
        __syncthreads();   // every read of X done before it is replaced
        float *Sn = Sc + (s + 1) * dd;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float4 a = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
            const float4 b = make_float4(acc[r][4], acc[r][5], acc[r][6], acc[r][7]);
            *reinterpret_cast<float4 *>(X + (i0 + r) * kD + j0) = a;
            *reinterpret_cast<float4 *>(X + (i0 + r) * kD + j0 + 4) = b;
            *reinterpret_cast<float4 *>(Sn + (i0 + r) * kD + j0) = a;
            *reinterpret_cast<float4 *>(Sn + (i0 + r) * kD + j0 + 4) = b;
        }
    }
}

}  // namespace

cudaError_t launch_seg_combine(const float *Z, const float *M, float *Sst, int chains, int nseg,
                               cudaStream_t stream) {
    const int smem = (kD * kLdA + kD * kD) * static_cast<int>(sizeof(float));
    cudaError_t e = cudaFuncSetAttribute(seg_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    seg_combine_kernel<<<chains, kThreads, smem, stream>>>(Z, M, Sst, nseg);
    return cudaGetLastError();
}

}  // namespace kla
