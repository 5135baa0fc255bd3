// kla_host.cu -- prefill from and to host memory with the copies overlapped with the kernels.
//
// kla_chunk_fwd_host splits the work into parts and runs, for part i: the host-to-device copies of its inputs on an upload stream, the prefill on one of
// several compute streams once those copies have landed, and the device-to-host copies of its
// outputs on a download stream once the prefill is done (two streams per direction, parts
// alternating, so two copies of a direction can be in flight). Copies of part i+1 overlap the
// prefill of part i, and the two directions of the link overlap each other.
//
// Time parts (bf16, scalar gate, d_k = d_v = 128, chunk 64, at least one chunk per part): part i
// is a slice of 64-token chunks of every sequence (small slices first and last, large ones in
// between), copied with strided (2-D) copies; the slices
// run in order on one compute stream with the state carried in place between them (in S_T_d, or
// in the fixed scratch array of kla_chunk_fwd_noalloc when no final state is wanted), each on
// all (sequence, head) chains at once. The first upload and the last prefill and download, which
// nothing overlaps, are then a part's share of the copies and a few chunk steps.
//
// Batch parts (every other call): part i is a range of whole sequences (contiguous in every
// tensor); prefills of different parts may run at the same time on different SMs. The
// sequence-parallel segments would only add work next to other parts, except in the last part:
// nothing runs beside it but the remaining copies, and its prefill plus its download are the
// call's tail, so it takes the segments when they shorten it, with the fixed scratch array (the
// last parts of consecutive calls are ordered on it by an event). With the per-channel gate, the
// other parts' rerun marks live in the array's last MiB, one slot per compute stream.
//
// Streams and events are created once per device on the first call and kept for the life of
// the process. Calls are ordered after earlier work on the caller's stream and the caller's
// stream waits for the last copy, so the call behaves as if it ran on that stream; calls on one
// device are serialised by a host mutex while they enqueue their work.
#include <algorithm>
#include <mutex>

#include "kla_internal.cuh"

namespace kla {
// Device address of the fixed KLA_NOALLOC_SCRATCH_BYTES scratch array on the current device
// (kla_noalloc.cu).
cudaError_t noalloc_scratch(void **out);
}  // namespace kla

namespace {

constexpr int kMaxDevices = 64;
constexpr int kComputeStreams = 8;
constexpr int kCopyStreams = 2;    // per direction: parts alternate between them
constexpr int kMaxParts = 64;
// The last MiB of the fixed scratch array holds, per compute stream, the flags with which the
// per-channel-gate prefill of a part marks chains for its exact rerun (parts sharing a slot
// share a stream, so they run one after the other); the last part's segments use the rest.
constexpr size_t kFlagTail = size_t(1) << 20;
constexpr size_t kFlagSlot = kFlagTail / kComputeStreams;

struct HostPipe {
    bool ready = false;
    cudaStream_t h2d[kCopyStreams] = {}, d2h[kCopyStreams] = {}, comp[kComputeStreams] = {};
    cudaEvent_t start = nullptr, in_done[kMaxParts] = {}, out_ready[kMaxParts] = {};
    cudaEvent_t end[kCopyStreams] = {}, comp_done[kComputeStreams] = {};
    cudaEvent_t scratch_free = nullptr;   // the last part's use of the shared scratch has ended
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mutex[kMaxDevices];

cudaError_t init_pipe(HostPipe &p) {
    if (p.ready) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    const unsigned sf = cudaStreamNonBlocking, ef = cudaEventDisableTiming;
    for (int c = 0; c < kCopyStreams; ++c) {
        if ((e = cudaStreamCreateWithFlags(&p.h2d[c], sf)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&p.d2h[c], sf)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&p.end[c], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    for (auto &s : p.comp)
        if ((e = cudaStreamCreateWithFlags(&s, sf)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&p.start, ef)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&p.scratch_free, ef)) != cudaSuccess) return e;
    for (int i = 0; i < kMaxParts; ++i) {
        if ((e = cudaEventCreateWithFlags(&p.in_done[i], ef)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&p.out_ready[i], ef)) != cudaSuccess) return e;
    }
    for (auto &ev : p.comp_done)
        if ((e = cudaEventCreateWithFlags(&ev, ef)) != cudaSuccess) return e;
    p.ready = true;
    return cudaSuccess;
}

}  // namespace

extern "C" kla_status kla_chunk_fwd_host(const void *q_h, const void *k_h, const void *v_h, const float *alpha_h,
                                         const float *eta_h, const float *S0_h, void *o_h, float *S_T_h, void *q_d,
                                         void *k_d, void *v_d, float *alpha_d, float *eta_d, float *S0_d, void *o_d,
                                         float *S_T_d, float eps, int B, int T, int H, int d_k, int d_v, int chunk,
                                         kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode, float q_scale,
                                         int parts, void *stream) {
    const bool time_parts = dtype == KLA_DTYPE_BF16 && gate == KLA_GATE_SCALAR && d_k == 128 && d_v == 128 &&
                            chunk == 64 && T > 16 && parts >= 1 && parts <= T / 64 &&
                            (S_T_d || static_cast<size_t>(B) * H * d_k * d_v * 4 <=
                                          static_cast<size_t>(KLA_NOALLOC_SCRATCH_BYTES) - kFlagTail);
    if (B < 1 || T < 1 || H < 1 || parts < 1 || parts > (time_parts ? kMaxParts : std::min(B, kMaxParts)))
        return KLA_ERR_INVALID_ARG;
    if (!q_h || !k_h || !v_h || !alpha_h || !eta_h || !o_h || !q_d || !k_d || !v_d || !alpha_d || !eta_d || !o_d)
        return KLA_ERR_INVALID_ARG;
    if ((S0_h != nullptr) != (S0_d != nullptr) || (S_T_h != nullptr) != (S_T_d != nullptr)) return KLA_ERR_INVALID_ARG;
    if (dtype != KLA_DTYPE_F32 && dtype != KLA_DTYPE_BF16) return KLA_ERR_INVALID_ARG;
    if (gate != KLA_GATE_SCALAR && gate != KLA_GATE_CHANNEL) return KLA_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_pipe_mutex[dev]);
    HostPipe &P = g_pipe[dev];
    if (init_pipe(P) != cudaSuccess) return KLA_ERR_CUDA;

    const size_t esz = dtype == KLA_DTYPE_BF16 ? 2 : 4;
    const size_t tok_per_b = static_cast<size_t>(T) * H;           // (t, h) rows of one sequence
    const size_t qk_b = tok_per_b * d_k * esz, v_b = tok_per_b * d_v * esz;
    const size_t a_b = tok_per_b * (gate == KLA_GATE_CHANNEL ? d_k : 1) * 4, e_b = tok_per_b * 4;
    const size_t s_b = static_cast<size_t>(H) * d_k * d_v * 4;
    const int bp = (B + parts - 1) / parts;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    auto H2D = cudaMemcpyHostToDevice;
    auto D2H = cudaMemcpyDeviceToHost;
    auto at = [](const void *p, size_t off) { return static_cast<const char *>(p) + off; };
    auto atw = [](void *p, size_t off) { return static_cast<char *>(p) + off; };

    bool ok = cudaEventRecord(P.start, cs) == cudaSuccess;
    for (int c = 0; ok && c < kCopyStreams; ++c)
        ok = cudaStreamWaitEvent(P.h2d[c], P.start, 0) == cudaSuccess &&
             cudaStreamWaitEvent(P.d2h[c], P.start, 0) == cudaSuccess;
    for (int c = 0; ok && c < kComputeStreams; ++c) ok = cudaStreamWaitEvent(P.comp[c], P.start, 0) == cudaSuccess;
    kla_status st = KLA_OK;
    void *scratch = nullptr;   // device address of the fixed scratch array
    if (ok && kla::noalloc_scratch(&scratch) != cudaSuccess) ok = false;
    if (time_parts && ok) {
        st = kla::check_chunk_fwd(q_d, k_d, v_d, alpha_d, eta_d, eps, S0_d, o_d, S_T_d, B, T, H, d_k, d_v, chunk, dtype,
                                  gate, beta_mode, q_scale);
        // Slice sizes follow a triangle (weights 1, 2, .., 2, 1): the first upload and the last
        // prefill and download, which nothing overlaps, are a small slice each while the copies of
        // the large middle slices overlap the link's other direction and the prefills. Slice i
        // covers chunks [cb[i], cb[i + 1]), at least one each.
        const int nchunks = (T + 63) / 64;
        int cb[kMaxParts + 1];
        {
            long wsum = 0;
            for (int i = 0; i < parts; ++i) wsum += std::min(i + 1, parts - i);
            long acc = 0;
            cb[0] = 0;
            for (int i = 0; i < parts; ++i) {
                acc += std::min(i + 1, parts - i);
                const int want = static_cast<int>((acc * nchunks + wsum / 2) / wsum);
                cb[i + 1] = std::min(std::max(want, cb[i] + 1), nchunks - (parts - 1 - i));
            }
        }
        float *state = S_T_d ? S_T_d : static_cast<float *>(scratch);
        cudaStream_t comp = P.comp[0];
        if (st == KLA_OK && !S_T_d && cudaStreamWaitEvent(comp, P.scratch_free, 0) != cudaSuccess) st = KLA_ERR_CUDA;
        const size_t qrow = static_cast<size_t>(H) * d_k * esz, vrow = static_cast<size_t>(H) * d_v * esz,
                     arow = static_cast<size_t>(H) * 4;   // bytes per token of every sequence
        cudaStream_t down = P.d2h[0];
        for (int i = 0; st == KLA_OK && ok && i < parts; ++i) {
            const int t0 = 64 * cb[i], nt = std::min(T, 64 * cb[i + 1]) - t0;
            cudaStream_t up = P.h2d[i % kCopyStreams];
            down = P.d2h[i % kCopyStreams];
            auto in2d = [&](void *dst, const void *src, size_t row) {   // tokens [t0, t0 + nt) of every sequence
                return cudaMemcpy2DAsync(atw(dst, t0 * row), T * row, at(src, t0 * row), T * row, nt * row, B, H2D,
                                         up) == cudaSuccess;
            };
            ok = in2d(q_d, q_h, qrow) && in2d(k_d, k_h, qrow) && in2d(v_d, v_h, vrow) && in2d(alpha_d, alpha_h, arow) &&
                 in2d(eta_d, eta_h, arow) &&
                 (i > 0 || !S0_h || cudaMemcpyAsync(S0_d, S0_h, B * s_b, H2D, up) == cudaSuccess) &&
                 cudaEventRecord(P.in_done[i], up) == cudaSuccess && cudaStreamWaitEvent(comp, P.in_done[i], 0) == cudaSuccess;
            if (!ok) break;
            st = kla::chunk_fwd_slice(at(q_d, t0 * qrow), at(k_d, t0 * qrow), at(v_d, t0 * vrow),
                                      reinterpret_cast<const float *>(at(alpha_d, t0 * arow)),
                                      reinterpret_cast<const float *>(at(eta_d, t0 * arow)), eps, i == 0 ? S0_d : state,
                                      atw(o_d, t0 * vrow), state, B, nt, T, H, beta_mode, q_scale, comp);
            if (st != KLA_OK) break;
            ok = cudaEventRecord(P.out_ready[i], comp) == cudaSuccess &&
                 cudaStreamWaitEvent(down, P.out_ready[i], 0) == cudaSuccess &&
                 cudaMemcpy2DAsync(atw(o_h, t0 * vrow), T * vrow, at(o_d, t0 * vrow), T * vrow, nt * vrow, B, D2H,
                                   down) == cudaSuccess;
        }
        if (st == KLA_OK && ok && S_T_h) ok = cudaMemcpyAsync(S_T_h, S_T_d, B * s_b, D2H, down) == cudaSuccess;
        // recorded even after a failure part-way: the next user of the array waits for what was enqueued
        if (!S_T_d && cudaEventRecord(P.scratch_free, comp) != cudaSuccess) ok = false;
    }
    for (int i = 0; !time_parts && ok && i < parts; ++i) {
        const int b0 = i * bp, nb = std::min(bp, B - b0);
        if (nb <= 0) break;
        cudaStream_t up = P.h2d[i % kCopyStreams], down = P.d2h[i % kCopyStreams];
        // inputs of part i
        ok = cudaMemcpyAsync(atw(q_d, b0 * qk_b), at(q_h, b0 * qk_b), nb * qk_b, H2D, up) == cudaSuccess &&
             cudaMemcpyAsync(atw(k_d, b0 * qk_b), at(k_h, b0 * qk_b), nb * qk_b, H2D, up) == cudaSuccess &&
             cudaMemcpyAsync(atw(v_d, b0 * v_b), at(v_h, b0 * v_b), nb * v_b, H2D, up) == cudaSuccess &&
             cudaMemcpyAsync(atw(alpha_d, b0 * a_b), at(alpha_h, b0 * a_b), nb * a_b, H2D, up) == cudaSuccess &&
             cudaMemcpyAsync(atw(eta_d, b0 * e_b), at(eta_h, b0 * e_b), nb * e_b, H2D, up) == cudaSuccess &&
             (!S0_h || cudaMemcpyAsync(atw(S0_d, b0 * s_b), at(S0_h, b0 * s_b), nb * s_b, H2D, up) == cudaSuccess) &&
             cudaEventRecord(P.in_done[i], up) == cudaSuccess;
        if (!ok) break;
        // the prefill of part i
        cudaStream_t comp = P.comp[i % kComputeStreams];
        ok = cudaStreamWaitEvent(comp, P.in_done[i], 0) == cudaSuccess;
        if (!ok) break;
        const void *qp = at(q_d, b0 * qk_b), *kp = at(k_d, b0 * qk_b), *vp = at(v_d, b0 * v_b);
        const float *ap = reinterpret_cast<const float *>(at(alpha_d, b0 * a_b));
        const float *ep = reinterpret_cast<const float *>(at(eta_d, b0 * e_b));
        const float *s0p = S0_d ? reinterpret_cast<const float *>(at(S0_d, b0 * s_b)) : nullptr;
        float *stp = S_T_d ? reinterpret_cast<float *>(atw(S_T_d, b0 * s_b)) : nullptr;
        const size_t need = b0 + nb >= B ? kla_chunk_fwd_workspace_size(nb, T, H, d_k, d_v, chunk, dtype, gate) : 0;
        const size_t seg_room = static_cast<size_t>(KLA_NOALLOC_SCRATCH_BYTES) - kFlagTail;
        if (need > 0 && need <= seg_room) {   // the last part, segmented or with the per-channel flags
            if (cudaStreamWaitEvent(comp, P.scratch_free, 0) != cudaSuccess) {
                st = KLA_ERR_CUDA;
                break;
            }
            st = kla_chunk_fwd_ex(qp, kp, vp, ap, ep, eps, s0p, atw(o_d, b0 * v_b), stp, nb, T, H, d_k, d_v, chunk, dtype,
                                  gate, beta_mode, q_scale, scratch, seg_room, comp);
            // recorded even when the prefill failed part-way: kernels it did enqueue may still use
            // the array, and the next user of the array must wait for them
            ok = cudaEventRecord(P.scratch_free, comp) == cudaSuccess;
            if (st != KLA_OK || !ok) break;
        } else {
            void *slot = gate == KLA_GATE_CHANNEL
                             ? static_cast<char *>(scratch) + seg_room + (i % kComputeStreams) * kFlagSlot
                             : nullptr;
            st = kla::chunk_fwd_nosplit(qp, kp, vp, ap, ep, eps, s0p, atw(o_d, b0 * v_b), stp, nb, T, H, d_k, d_v, chunk,
                                        dtype, gate, beta_mode, q_scale, slot, slot ? kFlagSlot : 0, comp);
            if (st != KLA_OK) break;
        }
        ok = cudaEventRecord(P.out_ready[i], comp) == cudaSuccess &&
             cudaStreamWaitEvent(down, P.out_ready[i], 0) == cudaSuccess;
        if (!ok) break;
        // outputs of part i
        ok = cudaMemcpyAsync(atw(o_h, b0 * v_b), at(o_d, b0 * v_b), nb * v_b, D2H, down) == cudaSuccess &&
             (!S_T_h ||
              cudaMemcpyAsync(atw(S_T_h, b0 * s_b), at(S_T_d, b0 * s_b), nb * s_b, D2H, down) == cudaSuccess);
    }
    // the caller's stream continues after the last output copy (and after every compute stream,
    // so that an error part-way leaves no work of this call behind it)
    bool joined = true;
    for (int c = 0; joined && c < kCopyStreams; ++c)
        joined = cudaEventRecord(P.end[c], P.d2h[c]) == cudaSuccess && cudaStreamWaitEvent(cs, P.end[c], 0) == cudaSuccess;
    for (int c = 0; joined && c < kComputeStreams; ++c)
        joined = cudaEventRecord(P.comp_done[c], P.comp[c]) == cudaSuccess &&
                 cudaStreamWaitEvent(cs, P.comp_done[c], 0) == cudaSuccess;
    if (st != KLA_OK) return st;
    return ok && joined ? KLA_OK : KLA_ERR_CUDA;
}
