// kla_api.cu -- the C ABI declared in include/kla.h: host-side validation, dispatch to
// the CUDA kernels, and the device error word.
#include <mutex>

#include "kla_internal.cuh"

namespace kla {
// one bounded wait on a barrier phase that nothing completes (kla_selftest.cu)
cudaError_t launch_selftest_wait(unsigned *err, unsigned limit, cudaStream_t stream);
// several tokens per call on the pipelined decode tile walk (kla_decode.cu): T <= kShortSeqMaxT,
// d_k = 128, d_v a multiple of 32, 16-byte aligned q, k, v, states and per-channel gates
bool tokens_pipe_supports(const ChunkArgs &a);
cudaError_t launch_tokens_pipe(const ChunkArgs &a);
// backward paths: the chunkwise one (kla_bwd_chunk.cu) runs when it supports the call, with a
// workspace of its own size; the token-sequential one (kla_bwd.cu) otherwise
bool bwd_chunk_supports(const BwdArgs &a);
size_t bwd_chunk_workspace_bytes(int B, int T, int H, kla_gate gate);
}  // namespace kla

namespace {

// One error word per device; bounded device waits and range checks OR bits into it.
__device__ unsigned g_err_word;

constexpr int kMaxDevices = 64;
unsigned *g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mutex;

// Device address of g_err_word on the current device (looked up once per device).
cudaError_t err_word(unsigned **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_err_mutex);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_err_word);
        if (e != cudaSuccess) return e;
        g_err_ptr[dev] = static_cast<unsigned *>(p);
    }
    *out = g_err_ptr[dev];
    return cudaSuccess;
}

bool aligned(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }
bool aligned16(const void *p) { return aligned(p, 16); }
bool supported_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool supported_chunk(int c) { return c == 16 || c == 32 || c == 64; }

// `vec_align`: required alignment of q, k, v and o (16 for the chunk path, whose tiles may be
// moved by TMA; the element size for decode). alpha and eta are read as scalars.
// `ntok` = 0 (no tokens) allows the token tensors to be NULL.
kla_status check_common(const void *q, const void *k, const void *v, const float *alpha,
                        const float *eta, const void *o, int B, int H, int d_k, int d_v,
                        kla_dtype dtype, kla_gate gate, uintptr_t vec_align, size_t ntok) {
    if (ntok > 0 && (!q || !k || !v || !alpha || !eta || !o)) return KLA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || d_k < 1 || d_v < 1) return KLA_ERR_INVALID_ARG;
    if (dtype != KLA_DTYPE_F32 && dtype != KLA_DTYPE_BF16) return KLA_ERR_INVALID_ARG;
    if (gate != KLA_GATE_SCALAR && gate != KLA_GATE_CHANNEL) return KLA_ERR_INVALID_ARG;
    if (vec_align == 0) vec_align = dtype == KLA_DTYPE_BF16 ? 2 : 4;
    if (!aligned(q, vec_align) || !aligned(k, vec_align) || !aligned(v, vec_align) || !aligned(o, vec_align) ||
        !aligned(alpha, 4) || !aligned(eta, 4))
        return KLA_ERR_INVALID_ARG;
    if (!supported_d(d_k) || !supported_d(d_v)) return KLA_ERR_UNSUPPORTED;
    return KLA_OK;
}

// Step-size mode known and query scale finite.
bool valid_mode(kla_beta_mode m, float q_scale) {
    return (m == KLA_BETA_KACZMARZ || m == KLA_BETA_RAW) && q_scale == q_scale && q_scale - q_scale == 0.0f;
}

// [lo, hi) byte range of a buffer, for overlap checks.
struct Span {
    uintptr_t lo, hi;
};
Span span(const void *p, size_t bytes) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, a + bytes};
}
bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

}  // namespace

// The error word for launchers below the entry points (the backward's carries).
namespace kla {
cudaError_t device_error_word(unsigned **out) { return err_word(out); }
}  // namespace kla

extern "C" {

int kla_abi_version(void) { return 102; }

const char *kla_status_string(kla_status s) {
    switch (s) {
        case KLA_OK: return "KLA_OK";
        case KLA_ERR_INVALID_ARG: return "KLA_ERR_INVALID_ARG: bad pointer, size, alignment or workspace";
        case KLA_ERR_UNSUPPORTED: return "KLA_ERR_UNSUPPORTED: size or chunk not implemented";
        case KLA_ERR_CUDA: return "KLA_ERR_CUDA: a CUDA call or kernel launch failed";
        case KLA_ERR_TIMEOUT: return "KLA_ERR_TIMEOUT: a bounded device wait gave up";
    }
    return "KLA_ERR_UNKNOWN";
}

size_t kla_chunk_fwd_workspace_size(int B, int T, int H, int d_k, int d_v, int chunk, kla_dtype dtype,
                                    kla_gate gate) {
    if (B < 1 || H < 1 || T < 1) return 0;
    kla::ChunkArgs a{};
    a.B = B; a.T = T; a.H = H; a.d_k = d_k; a.d_v = d_v; a.chunk = chunk; a.dtype = dtype; a.gate = gate;
    if (kla::recurrent_preferred(a)) return 0;
    return kla::chunk_tc_supports(a) ? kla::chunk_tc_workspace_bytes(B, T, H, gate) : 0;
}

}  // extern "C"

// Every argument check of the chunk forward except the workspace's.
kla_status kla::check_chunk_fwd(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                                float eps, const float *S0, const void *o, const float *S_T, int B, int T, int H,
                                int d_k, int d_v, int chunk, kla_dtype dtype, kla_gate gate,
                                kla_beta_mode beta_mode, float q_scale) {
    if (T < 0) return KLA_ERR_INVALID_ARG;
    if (!valid_mode(beta_mode, q_scale)) return KLA_ERR_INVALID_ARG;
    kla_status st = check_common(q, k, v, alpha, eta, o, B, H, d_k, d_v, dtype, gate, 16,
                                 static_cast<size_t>(B) * T * H);
    if (st != KLA_OK) return st;
    if (!supported_chunk(chunk)) return KLA_ERR_UNSUPPORTED;
    if ((S0 && !aligned16(S0)) || (S_T && !aligned16(S_T))) return KLA_ERR_INVALID_ARG;
    if (!(eps == eps)) return KLA_ERR_INVALID_ARG;   // NaN stabiliser

    // The final state may alias S0 exactly but must not overlap anything else.
    const size_t esz = dtype == KLA_DTYPE_BF16 ? 2 : 4;
    const size_t ntok = static_cast<size_t>(B) * T * H;
    const size_t sbytes = static_cast<size_t>(B) * H * d_k * d_v * 4;
    if (S_T) {
        Span s = span(S_T, sbytes);
        const Span others[] = {span(q, ntok * d_k * esz), span(k, ntok * d_k * esz), span(v, ntok * d_v * esz),
                               span(o, ntok * d_v * esz),
                               span(alpha, ntok * (gate == KLA_GATE_CHANNEL ? d_k : 1) * 4),
                               span(eta, ntok * 4)};
        for (const Span &x : others)
            if (x.hi > x.lo && overlaps(s, x)) return KLA_ERR_INVALID_ARG;
        if (S0 && S0 != S_T && overlaps(s, span(S0, sbytes))) return KLA_ERR_INVALID_ARG;
    }
    return KLA_OK;
}

namespace {

kla_status chunk_fwd_impl(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                          float eps, const float *S0, void *o, float *S_T, int B, int T, int H, int d_k, int d_v,
                          int chunk, kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode, float q_scale,
                          void *workspace, size_t workspace_bytes, void *stream, int no_segments) {
    kla_status st = kla::check_chunk_fwd(q, k, v, alpha, eta, eps, S0, o, S_T, B, T, H, d_k, d_v, chunk, dtype,
                                         gate, beta_mode, q_scale);
    if (st != KLA_OK) return st;
    const size_t need = no_segments ? 0 : kla_chunk_fwd_workspace_size(B, T, H, d_k, d_v, chunk, dtype, gate);
    if (workspace_bytes < need || (need > 0 && !workspace)) return KLA_ERR_INVALID_ARG;
    const size_t sbytes = static_cast<size_t>(B) * H * d_k * d_v * 4;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (T == 0) {   // no tokens: the final state is the initial state
        if (!S_T) return KLA_OK;
        cudaError_t e = S0 ? (S0 == S_T ? cudaSuccess : cudaMemcpyAsync(S_T, S0, sbytes, cudaMemcpyDeviceToDevice, cs))
                           : cudaMemsetAsync(S_T, 0, sbytes, cs);
        return e == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
    }

    kla::ChunkArgs a{q, k, v, alpha, eta, eps, S0, o, S_T, B, T, H, d_k, d_v, chunk, dtype, gate,
                     workspace, workspace_bytes, nullptr, cs};
    a.beta_raw = beta_mode == KLA_BETA_RAW;
    a.q_scale = q_scale;
    a.no_segments = no_segments;
    if (err_word(&a.err) != cudaSuccess) return KLA_ERR_CUDA;
    cudaError_t e = !kla::recurrent_preferred(a)      ? kla::launch_chunk_tc(a)
                    : kla::tokens_pipe_supports(a) ? kla::launch_tokens_pipe(a)
                                                   : kla::launch_recurrent(a);
    return e == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

}  // namespace

kla_status kla::chunk_fwd_nosplit(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                                  float eps, const float *S0, void *o, float *S_T, int B, int T, int H, int d_k,
                                  int d_v, int chunk, kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode,
                                  float q_scale, void *workspace, size_t workspace_bytes, void *stream) {
    return chunk_fwd_impl(q, k, v, alpha, eta, eps, S0, o, S_T, B, T, H, d_k, d_v, chunk, dtype, gate, beta_mode,
                          q_scale, workspace, workspace_bytes, stream, 1);
}

kla_status kla::chunk_fwd_slice(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                                float eps, const float *S0, void *o, float *S_T, int B, int T, int T_stride, int H,
                                kla_beta_mode beta_mode, float q_scale, void *stream) {
    if (T < 1 || T_stride < T) return KLA_ERR_INVALID_ARG;
    kla::ChunkArgs a{q, k, v, alpha, eta, eps, S0, o, S_T, B, T, H, 128, 128, 64, KLA_DTYPE_BF16, KLA_GATE_SCALAR,
                     nullptr, 0, nullptr, static_cast<cudaStream_t>(stream)};
    a.beta_raw = beta_mode == KLA_BETA_RAW;
    a.q_scale = q_scale;
    a.no_segments = 1;
    a.T_stride = T_stride;
    if (err_word(&a.err) != cudaSuccess) return KLA_ERR_CUDA;
    return kla::launch_chunk_tc(a) == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

extern "C" {

kla_status kla_chunk_fwd_ex(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                            float eps, const float *S0, void *o, float *S_T, int B, int T, int H, int d_k, int d_v,
                            int chunk, kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode, float q_scale,
                            void *workspace, size_t workspace_bytes, void *stream) {
    return chunk_fwd_impl(q, k, v, alpha, eta, eps, S0, o, S_T, B, T, H, d_k, d_v, chunk, dtype, gate, beta_mode,
                          q_scale, workspace, workspace_bytes, stream, 0);
}

kla_status kla_chunk_fwd(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                         float eps, const float *S0, void *o, float *S_T, int B, int T, int H, int d_k, int d_v,
                         int chunk, kla_dtype dtype, kla_gate gate, void *workspace, size_t workspace_bytes,
                         void *stream) {
    return kla_chunk_fwd_ex(q, k, v, alpha, eta, eps, S0, o, S_T, B, T, H, d_k, d_v, chunk, dtype, gate,
                            KLA_BETA_KACZMARZ, 1.0f, workspace, workspace_bytes, stream);
}

kla_status kla_decode_step_ex(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                              float eps, float *S, void *o, int B, int H, int d_k, int d_v, kla_dtype dtype,
                              kla_gate gate, kla_beta_mode beta_mode, float q_scale, void *stream) {
    if (!valid_mode(beta_mode, q_scale)) return KLA_ERR_INVALID_ARG;
    kla_status st = check_common(q, k, v, alpha, eta, o, B, H, d_k, d_v, dtype, gate, 0, 1);
    if (st != KLA_OK) return st;
    if (!S || !aligned16(S)) return KLA_ERR_INVALID_ARG;
    if (!(eps == eps)) return KLA_ERR_INVALID_ARG;
    const size_t esz = dtype == KLA_DTYPE_BF16 ? 2 : 4;
    const size_t nh = static_cast<size_t>(B) * H;
    Span s = span(S, nh * d_k * d_v * 4);
    const Span others[] = {span(q, nh * d_k * esz), span(k, nh * d_k * esz), span(v, nh * d_v * esz),
                           span(o, nh * d_v * esz), span(alpha, nh * (gate == KLA_GATE_CHANNEL ? d_k : 1) * 4),
                           span(eta, nh * 4)};
    for (const Span &x : others)
        if (overlaps(s, x)) return KLA_ERR_INVALID_ARG;
    kla::DecodeArgs a{q, k, v, alpha, eta, eps, S, o, B, H, d_k, d_v, dtype, gate, nullptr,
                      static_cast<cudaStream_t>(stream)};
    a.beta_raw = beta_mode == KLA_BETA_RAW;
    a.q_scale = q_scale;
    if (err_word(&a.err) != cudaSuccess) return KLA_ERR_CUDA;
    return kla::launch_decode(a) == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

kla_status kla_decode_step(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                           float eps, float *S, void *o, int B, int H, int d_k, int d_v, kla_dtype dtype,
                           kla_gate gate, void *stream) {
    return kla_decode_step_ex(q, k, v, alpha, eta, eps, S, o, B, H, d_k, d_v, dtype, gate, KLA_BETA_KACZMARZ,
                              1.0f, stream);
}

size_t kla_chunk_bwd_workspace_size(int B, int T, int H, int d_k, int d_v) {
    return kla::bwd_workspace_bytes(B, T, H, d_k, d_v);
}

size_t kla_chunk_bwd_workspace_size_ex(int B, int T, int H, int d_k, int d_v, kla_dtype dtype, kla_gate gate) {
    const bool chunked = dtype == KLA_DTYPE_BF16 && (gate == KLA_GATE_SCALAR || gate == KLA_GATE_CHANNEL) &&
                         d_k == 128 && d_v == 128 && T > kla::kShortSeqMaxT && B >= 1 && H >= 1;
    return chunked ? kla::bwd_chunk_workspace_bytes(B, T, H, gate) : kla::bwd_seq_workspace_bytes(B, T, H, d_k, d_v);
}

kla_status kla_chunk_bwd(const void *q, const void *k, const void *v, const float *alpha, const float *eta,
                         float eps, const float *S0, const void *dO, const float *dS_T, float *dq, float *dk,
                         float *dv, float *dalpha, float *deta, float *dS0, int B, int T, int H, int d_k, int d_v,
                         kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode, float q_scale, void *workspace,
                         size_t workspace_bytes, void *stream) {
    if (T < 0) return KLA_ERR_INVALID_ARG;
    if (!valid_mode(beta_mode, q_scale)) return KLA_ERR_INVALID_ARG;
    const size_t ntok = static_cast<size_t>(B) * T * H;
    kla_status st = check_common(q, k, v, alpha, eta, dO, B, H, d_k, d_v, dtype, gate, 0, ntok);
    if (st != KLA_OK) return st;
    if (ntok > 0 && (!dq || !dk || !dv || !dalpha || !deta)) return KLA_ERR_INVALID_ARG;
    if (!aligned(dq, 4) || !aligned(dk, 4) || !aligned(dalpha, 4) || !aligned(deta, 4) || !aligned16(dv))
        return KLA_ERR_INVALID_ARG;
    if ((S0 && !aligned16(S0)) || (dS_T && !aligned16(dS_T)) || (dS0 && !aligned16(dS0))) return KLA_ERR_INVALID_ARG;
    if (!(eps == eps)) return KLA_ERR_INVALID_ARG;
    kla::BwdArgs a{q, k, v, dO, alpha, eta, eps, S0, dS_T, dq, dk, dv, dalpha, deta, dS0, B, T, H, d_k, d_v,
                   dtype, gate, beta_mode == KLA_BETA_RAW, q_scale, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream)};
    // the chunkwise path needs its own (smaller) workspace; any other call the token-sequential one's
    const size_t need = T > 0 && kla::bwd_chunk_supports(a) ? kla::bwd_chunk_workspace_bytes(B, T, H, gate)
                                                            : kla::bwd_seq_workspace_bytes(B, T, H, d_k, d_v);
    if (workspace_bytes < need || (need > 0 && (!workspace || !aligned16(workspace)))) return KLA_ERR_INVALID_ARG;

    const size_t esz = dtype == KLA_DTYPE_BF16 ? 2 : 4;
    const size_t sbytes = static_cast<size_t>(B) * H * d_k * d_v * 4;
    const size_t abytes = ntok * (gate == KLA_GATE_CHANNEL ? d_k : 1) * 4;
    const Span outs[] = {span(dq, ntok * d_k * 4), span(dk, ntok * d_k * 4), span(dv, ntok * d_v * 4),
                         span(dalpha, abytes), span(deta, ntok * 4), span(dS0, dS0 ? sbytes : 0),
                         span(workspace, need)};
    const Span ins[] = {span(q, ntok * d_k * esz), span(k, ntok * d_k * esz), span(v, ntok * d_v * esz),
                        span(dO, ntok * d_v * esz), span(alpha, abytes), span(eta, ntok * 4),
                        span(S0, S0 ? sbytes : 0), span(dS_T, dS_T ? sbytes : 0)};
    for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
        if (outs[i].hi <= outs[i].lo) continue;
        for (const Span &x : ins)
            if (x.hi > x.lo && overlaps(outs[i], x)) return KLA_ERR_INVALID_ARG;
        for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
            if (outs[j].hi > outs[j].lo && overlaps(outs[i], outs[j])) return KLA_ERR_INVALID_ARG;
    }

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (T == 0) {   // no tokens: dL/dS0 = dL/dS_T
        if (!dS0) return KLA_OK;
        cudaError_t e = dS_T ? cudaMemcpyAsync(dS0, dS_T, sbytes, cudaMemcpyDeviceToDevice, cs)
                             : cudaMemsetAsync(dS0, 0, sbytes, cs);
        return e == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
    }
    return kla::launch_bwd(a) == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

kla_status kla_selftest_wait_timeout(unsigned limit_polls, void *stream) {
    if (limit_polls < 1 || limit_polls > 100000) return KLA_ERR_INVALID_ARG;
    unsigned *err = nullptr;
    if (err_word(&err) != cudaSuccess) return KLA_ERR_CUDA;
    return kla::launch_selftest_wait(err, limit_polls, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KLA_OK
               : KLA_ERR_CUDA;
}

kla_status kla_device_status(void *stream) {
    unsigned *p = nullptr;
    if (err_word(&p) != cudaSuccess) return KLA_ERR_CUDA;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    unsigned h = 0;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return KLA_ERR_CUDA;
    if (cudaMemcpy(&h, p, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return KLA_ERR_CUDA;
    if (h) {
        const unsigned zero = 0;
        if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return KLA_ERR_CUDA;
    }
    if (h & kla::kErrTimeout) return KLA_ERR_TIMEOUT;
    if (h & kla::kErrGateRange) return KLA_ERR_INVALID_ARG;
    return KLA_OK;
}

}  // extern "C"
