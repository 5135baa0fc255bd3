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
// keeps its column block of X and the current M^T in shared memory and runs the short serial
// pass in fp32.
#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr int kD = 128;
constexpr int kSplit = 8;              // CTAs per chain
constexpr int kCols = kD / kSplit;     // columns of X per CTA (16)
constexpr int kThreads = 256;          // 128 rows x 16 columns: 8 outputs (one row, 8 columns) per thread
constexpr int kLdA = kD + 4;           // padded row of M^T in shared memory

__global__ void __launch_bounds__(kThreads) seg_combine_kernel(const float *Z, const float *M, float *Sst,
                                                               int nseg) {
    extern __shared__ __align__(16) float csm[];
    float *At = csm;                 // M^T: [k][i], row stride kLdA
    float *X = csm + kD * kLdA;      // this CTA's columns of the current start state: [k][kCols]
    const int tid = threadIdx.x;
    const size_t chain = blockIdx.x / kSplit;
    const int c0 = (blockIdx.x % kSplit) * kCols;
    const size_t dd = static_cast<size_t>(kD) * kD;
    const float *Zc = Z + chain * nseg * dd, *Mc = M + chain * nseg * dd;
    float *Sc = Sst + chain * nseg * dd;

    for (int idx = tid; idx < kD * kCols / 4; idx += kThreads) {   // S_start[1] = Z_0
        const int r = idx / (kCols / 4), q = idx % (kCols / 4);
        const float4 z = *reinterpret_cast<const float4 *>(Zc + r * kD + c0 + 4 * q);
        reinterpret_cast<float4 *>(X)[idx] = z;
        *reinterpret_cast<float4 *>(Sc + dd + r * kD + c0 + 4 * q) = z;
    }
    const int i0 = tid >> 1, j0 = (tid & 1) * 8;   // row i0, columns j0..j0+7 of the block
    for (int s = 1; s + 1 < nseg; ++s) {
        __syncthreads();
        const float *Ms = Mc + s * dd;
        for (int idx = tid; idx < kD * kD; idx += kThreads) {
            const int i = idx >> 7, k = idx & (kD - 1);
            At[k * kLdA + i] = Ms[idx];
        }
        __syncthreads();
        float acc[8];
        const float *Zs = Zc + s * dd + i0 * kD + c0 + j0;
        {
            const float4 a = *reinterpret_cast<const float4 *>(Zs);
            const float4 b = *reinterpret_cast<const float4 *>(Zs + 4);
            acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
            acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
        }
#pragma unroll 4
        for (int k = 0; k < kD; ++k) {
            const float a = At[k * kLdA + i0];
            const float4 x0 = *reinterpret_cast<const float4 *>(X + k * kCols + j0);
            const float4 x1 = *reinterpret_cast<const float4 *>(X + k * kCols + j0 + 4);
            acc[0] = fmaf(a, x0.x, acc[0]); acc[1] = fmaf(a, x0.y, acc[1]);
            acc[2] = fmaf(a, x0.z, acc[2]); acc[3] = fmaf(a, x0.w, acc[3]);
            acc[4] = fmaf(a, x1.x, acc[4]); acc[5] = fmaf(a, x1.y, acc[5]);
            acc[6] = fmaf(a, x1.z, acc[6]); acc[7] = fmaf(a, x1.w, acc[7]);
        }
        __syncthreads();   // every read of X done before it is replaced
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
    const int smem = (kD * kLdA + kD * kCols) * static_cast<int>(sizeof(float));
    cudaError_t e = cudaFuncSetAttribute(seg_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    seg_combine_kernel<<<chains * kSplit, kThreads, smem, stream>>>(Z, M, Sst, nseg);
    return cudaGetLastError();
}

}  // namespace kla
