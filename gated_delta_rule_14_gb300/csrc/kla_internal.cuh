// kla_internal.cuh -- shared declarations of the KLA CUDA library (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kla.h"

namespace kla {

// Device-side error bits, OR-ed into one word per device (see kla_device_status).
enum : unsigned {
    kErrTimeout = 1u,      // a bounded wait gave up
    kErrGateRange = 2u,    // per-channel log-decay outside the exact range of a factorised product
};

// Everything a chunk-forward launcher needs; pointers are device pointers.
struct ChunkArgs {
    const void *q, *k, *v;
    const float *alpha, *eta;
    float eps;
    const float *S0;
    void *o;
    float *S_T;
    int B, T, H, d_k, d_v, chunk;
    kla_dtype dtype;
    kla_gate gate;
    void *workspace;
    size_t workspace_bytes;
    unsigned *err;         // device error word
    cudaStream_t stream;
    int beta_raw;          // 1: beta = eta (KLA_BETA_RAW)
    float q_scale;         // o = S^T (q_scale q)
    int no_segments;       // 1: never split long sequences into parallel segments
    const unsigned *only;  // recurrent path: when set, only chains (b, h) with only[b * H + h] != 0 run
    int T_stride;          // tensor-core path, scalar gate: tokens between sequences in q/k/v/o/alpha/eta
                           // (0: T); a T-token slice of longer sequences when larger than T
};

struct DecodeArgs {
    const void *q, *k, *v;
    const float *alpha, *eta;
    float eps;
    float *S;
    void *o;
    int B, H, d_k, d_v;
    kla_dtype dtype;
    kla_gate gate;
    unsigned *err;         // device error word
    cudaStream_t stream;
    int beta_raw;          // 1: beta = eta (KLA_BETA_RAW)
    float q_scale;         // o = S^T (q_scale q)
};

// Backward pass: gradients of a loss given dL/do and dL/dS_T; every gradient is fp32.
struct BwdArgs {
    const void *q, *k, *v, *dO;
    const float *alpha, *eta;
    float eps;
    const float *S0, *dS_T;
    float *dq, *dk, *dv, *dalpha, *deta, *dS0;
    int B, T, H, d_k, d_v;
    kla_dtype dtype;
    kla_gate gate;
    int beta_raw;
    float q_scale;
    void *workspace;
    size_t workspace_bytes;
    cudaStream_t stream;
};

// kla_chunk_fwd_ex without the sequence-parallel segments: for callers that run several
// prefills side by side, where splitting each one would only add work. The workspace is optional
// (NULL, 0): with the per-channel gate and at least 4 * B * H bytes, chains outside the range of
// the factorised in-chunk products are rerun exactly, otherwise they are only reported.
kla_status chunk_fwd_nosplit(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                             float eps, const float *S0, void *o, float *S_T, int B, int T, int H, int d_k, int d_v,
                             int chunk, kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode, float q_scale,
                             void *workspace, size_t workspace_bytes, void *stream);

// The tensor-core prefill of tokens [t0, t0 + T) of every sequence (bf16, scalar gate, d_k = d_v = 128,
// chunk 64, no segments): q, k, v, o, alpha and eta point at token t0 of sequence 0 and successive
// sequences are T_stride tokens apart. The caller has validated the whole tensors; t0 is a
// multiple of 64, so the state carried from the previous slice enters at a chunk boundary.
kla_status chunk_fwd_slice(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                           float eps, const float *S0, void *o, float *S_T, int B, int T, int T_stride, int H,
                           kla_beta_mode beta_mode, float q_scale, void *stream);

// Every argument check of kla_chunk_fwd_ex except the workspace's (its errors, in its order).
kla_status check_chunk_fwd(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                           float eps, const float *S0, const void *o, const float *S_T, int B, int T, int H, int d_k,
                           int d_v, int chunk, kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode,
                           float q_scale);

// tcgen05 tensor-core chunk path: bf16, d_k = d_v = 128, chunk = 64.
bool chunk_tc_supports(const ChunkArgs &a);
cudaError_t launch_chunk_tc(const ChunkArgs &a);
// Device scratch the tensor-core path needs for these sizes: the segments' states when it splits
// long sequences into segments that run in parallel, and with the per-channel gate one flag per
// (sequence, head) chain whose gates leave the range of the factorised in-chunk products.
size_t chunk_tc_workspace_bytes(int B, int T, int H, kla_gate gate);
// Per-channel gate (fp32 [B, T, H, 128]): zeroes marks[B*H], then marks every (sequence, head)
// chain with a 64-token chunk whose gates, for some key channel, multiply to less than ~e^-78 over
// tokens 0-31 or 32-63 (the range of the in-chunk products factorised around token 31).
cudaError_t launch_gate_range(const float *alpha, int B, int T, int H, unsigned *marks, cudaStream_t stream);
// Start states of the segments of every chain: S_start[s+1] = M_s S_start[s] + Z_s.
cudaError_t launch_seg_combine(const float *Z, const float *M, float *Sst, int chains, int nseg,
                               cudaStream_t stream);
// backward pass (checkpoints every 8 tokens plus the residuals in the workspace).
size_t bwd_workspace_bytes(int B, int T, int H, int d_k, int d_v);
cudaError_t launch_bwd(const BwdArgs &a);
// The token-sequential fp32 backward (kla_bwd.cu) on every chain, or only on the chains with a
// nonzero mark in only[B*H]; its workspace is bwd_seq_workspace_bytes.
size_t bwd_seq_workspace_bytes(int B, int T, int H, int d_k, int d_v);
cudaError_t launch_bwd_seq(const BwdArgs &a, const unsigned *only);
// fused single-token decode step.
cudaError_t launch_decode(const DecodeArgs &a);
// Token-by-token recurrence with the state tile in registers: short sequences (multi-token
// decode, speculative verification, T <= kShortSeqMaxT) and every shape the tensor-core path
// does not take; any supported size and dtype, fp32 arithmetic.
constexpr int kShortSeqMaxT = 16;
// The chunk form of 9-16 tokens with the per-channel gate (bf16, d_k = d_v = 128, 16-byte
// aligned q, k, v, o, alpha and states): kla_tokens_ch.cu.
bool tokens_ch_supports(const ChunkArgs &a);
cudaError_t launch_tokens_ch(const ChunkArgs &a);
bool recurrent_preferred(const ChunkArgs &a);
cudaError_t launch_recurrent(const ChunkArgs &a);

// ------------------------------------------------------------------ device helpers
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// beta = eta / (||k||^2 + eps), 0 when the denominator is exactly zero; beta = eta in the
// raw mode (DeltaNet / Gated DeltaNet write strength).
__device__ __forceinline__ float kla_beta(float eta, float knorm2, float eps, int raw) {
    if (raw) return eta;
    const float den = knorm2 + eps;
    return den == 0.0f ? 0.0f : eta / den;
}

}  // namespace kla
