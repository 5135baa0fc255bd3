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
// The columns of the start states evolve independently (X <- M X + Z acts on each column of X
// alone), so every chain's pass is split over kSplit CTAs of kD / kSplit columns each; a CTA
// keeps its column block of X in shared memory, streams the transitions M_s into two padded
// buffers by cp.async (M_{s+1} lands while step s computes) and runs the short serial pass in
// fp32.
#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr int kD = 128;
constexpr int kSplit = 8;              // CTAs per chain
constexpr int kCols = kD / kSplit;     // columns of X per CTA (16)
constexpr int kThreads = 256;          // 128 rows x 16 columns: 8 outputs (one row, 8 columns) per thread
constexpr int kLdM = kD + 4;           // padded row of M in shared memory
constexpr int kSmemBytes = (2 * kD * kLdM + kD * kCols) * static_cast<int>(sizeof(float));

__device__ __forceinline__ void cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__global__ void __launch_bounds__(kThreads) seg_combine_kernel(const float *Z, const float *M, float *Sst,
                                                               int nseg) {
    extern __shared__ __align__(16) float csm[];
    float *Mb = csm;                     // two buffers of M_s: [i][k], row stride kLdM
    float *X = csm + 2 * kD * kLdM;      // this CTA's columns of the current start state: [k][kCols]
    const int tid = threadIdx.x;
    const size_t chain = blockIdx.x / kSplit;
    const int c0 = (blockIdx.x % kSplit) * kCols;
    const size_t dd = static_cast<size_t>(kD) * kD;
    const float *Zc = Z + chain * nseg * dd, *Mc = M + chain * nseg * dd;
    float *Sc = Sst + chain * nseg * dd;

    auto load_m = [&](int s, int buf) {   // M_s into buffer buf, 16-byte granules
        const float *Ms = Mc + s * dd;
        float *dst = Mb + buf * kD * kLdM;
        for (int idx = tid; idx < kD * kD / 4; idx += kThreads) {
            const int i = idx >> 5, q = idx & 31;
            cp16(dst + i * kLdM + 4 * q, Ms + i * kD + 4 * q);
        }
        cp_commit();
    };
    if (nseg > 2) load_m(1, 0);
    for (int idx = tid; idx < kD * kCols / 4; idx += kThreads) {   // S_start[1] = Z_0
        const int r = idx / (kCols / 4), q = idx % (kCols / 4);
        const float4 z = *reinterpret_cast<const float4 *>(Zc + r * kD + c0 + 4 * q);
        reinterpret_cast<float4 *>(X)[idx] = z;
        *reinterpret_cast<float4 *>(Sc + dd + r * kD + c0 + 4 * q) = z;
    }
    const int i0 = tid >> 1, j0 = (tid & 1) * 8;   // row i0, columns j0..j0+7 of the block
    for (int s = 1; s + 1 < nseg; ++s) {
        const int buf = (s - 1) & 1;
        // Z_s of this thread's outputs, requested before the waits
        const float *Zs = Zc + s * dd + i0 * kD + c0 + j0;
        const float4 za = *reinterpret_cast<const float4 *>(Zs);
        const float4 zb = *reinterpret_cast<const float4 *>(Zs + 4);
        if (s + 2 < nseg) {   // buffer buf ^ 1 was last read in step s - 1, before its closing barrier
            load_m(s + 1, buf ^ 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();   // M_s and X of the previous step are visible
        float acc[8] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
        const float *Mr = Mb + buf * kD * kLdM + i0 * kLdM;
#pragma unroll 2
        for (int k4 = 0; k4 < kD / 4; ++k4) {
            const float4 m = *reinterpret_cast<const float4 *>(Mr + 4 * k4);
            const float mv[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = 4 * k4 + u;
                const float4 x0 = *reinterpret_cast<const float4 *>(X + k * kCols + j0);
                const float4 x1 = *reinterpret_cast<const float4 *>(X + k * kCols + j0 + 4);
                acc[0] = fmaf(mv[u], x0.x, acc[0]); acc[1] = fmaf(mv[u], x0.y, acc[1]);
                acc[2] = fmaf(mv[u], x0.z, acc[2]); acc[3] = fmaf(mv[u], x0.w, acc[3]);
                acc[4] = fmaf(mv[u], x1.x, acc[4]); acc[5] = fmaf(mv[u], x1.y, acc[5]);
                acc[6] = fmaf(mv[u], x1.z, acc[6]); acc[7] = fmaf(mv[u], x1.w, acc[7]);
            }
        }
        __syncthreads();   // every read of X and of buffer buf is done before they are replaced
        float *Sn = Sc + (s + 1) * dd + i0 * kD + c0 + j0;
        const float4 a = make_float4(acc[0], acc[1], acc[2], acc[3]);
        const float4 b = make_float4(acc[4], acc[5], acc[6], acc[7]);
        *reinterpret_cast<float4 *>(X + i0 * kCols + j0) = a;
        *reinterpret_cast<float4 *>(X + i0 * kCols + j0 + 4) = b;
        *reinterpret_cast<float4 *>(Sn) = a;
        *reinterpret_cast<float4 *>(Sn + 4) = b;
    }
}

}  // namespace

cudaError_t launch_seg_combine(const float *Z, const float *M, float *Sst, int chains, int nseg,
                               cudaStream_t stream) {
    cudaError_t e =
        cudaFuncSetAttribute(seg_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    seg_combine_kernel<<<chains * kSplit, kThreads, kSmemBytes, stream>>>(Z, M, Sst, nseg);
    return cudaGetLastError();
}

}  // namespace kla
