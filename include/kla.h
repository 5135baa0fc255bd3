/*
 * kla.h -- C ABI of the KLA gated delta-rule recurrence on NVIDIA GB300 (sm_103a).
 *
 * The operation (Gist.science, "Riepilogo Tecnico: Attenzione Lineare Kaczmarz
 * (KLA)", sections "Derivazione Teorica" and "La Regola di Aggiornamento KLA"):
 * for every sequence b and head h, a state S (d_k x d_v; rows are key channels,
 * columns value channels) is carried over tokens t = 0..T-1:
 *
 *     S~_t  = alpha_t (.) S_{t-1}                 forget (gate on the key rows)
 *     e_t   = v_t - S~_t^T k_t                     residual against the decayed state
 *     beta_t= eta_t / (||k_t||^2 + eps)            Kaczmarz step (0 if the denominator is 0)
 *     S_t   = S~_t + beta_t k_t e_t^T              write
 *     o_t   = S_t^T q_t                            read, after the write
 *
 * The _ex entry points add two options (GeekNews, "Revisando las variantes de
 * atencion lineal de la familia DeltaNet", sections "Gated DeltaNet: primero
 * olvidar todo el estado" and "Kimi Delta Attention"):
 * beta_t = eta_t itself, the write strength of DeltaNet and Gated DeltaNet
 * (KLA_BETA_RAW), and a query scale s on the read, o_t = S_t^T (s q_t)
 * (s = d_k^{-1/2} in Kimi Delta Attention).
 *
 * alpha_t is one scalar per (b, t, h) (Gated DeltaNet / KLA gate) or one value per
 * key channel (Kimi Delta Attention gate: GeekNews, "Revisando las variantes de
 * atencion lineal de la familia DeltaNet", section "Kimi Delta Attention"), in
 * which case row i of S is scaled by alpha_t[i].
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers to row-major, contiguous tensors.
 *    Alignment: the state (S0, S_T, S) 16 bytes; q, k, v, o 16 bytes for
 *    kla_chunk_fwd and their element size for kla_decode_step; alpha, eta 4 bytes.
 *    The caller allocates and owns every buffer; the library allocates no device
 *    memory and keeps no per-call state.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 *    the legacy default stream). A returned KLA_OK means the work was enqueued.
 *  - Argument errors are detected on the host before anything is launched and
 *    return KLA_ERR_INVALID_ARG or KLA_ERR_UNSUPPORTED; nothing is written then.
 *  - Device-side waits are bounded; a wait that gives up records a flag that
 *    kla_device_status() reports as KLA_ERR_TIMEOUT.
 *  - The library keeps a few per-device objects for the life of the process (streams and
 *    events of its own, the device addresses of its error word and scratch array, looked up
 *    on first use). cudaDeviceReset() destroys them: do not call into the library on a
 *    device after resetting it.
 *  - Supported sizes: d_k, d_v in {16, 32, 64, 128}; chunk in {16, 32, 64}.
 *    bf16 inputs with d_k = d_v = 128 and chunk = 64 run on the tensor-core
 *    (tcgen05) path; every other supported case runs on the fp32 CUDA-core path.
 */
#ifndef KLA_H
#define KLA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kla_status {
    KLA_OK = 0,
    KLA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, workspace too small */
    KLA_ERR_UNSUPPORTED = 2,   /* valid but not implemented size / chunk combination */
    KLA_ERR_CUDA = 3,          /* a CUDA runtime call or a launch failed */
    KLA_ERR_TIMEOUT = 4        /* a bounded device wait gave up (see kla_device_status) */
} kla_status;

typedef enum kla_dtype {
    KLA_DTYPE_F32 = 0,         /* q, k, v, o stored as IEEE fp32 */
    KLA_DTYPE_BF16 = 1         /* q, k, v, o stored as bfloat16 */
} kla_dtype;

typedef enum kla_gate {
    KLA_GATE_SCALAR = 0,       /* alpha [B, T, H]: one gate per token and head */
    KLA_GATE_CHANNEL = 1       /* alpha [B, T, H, d_k]: one gate per key channel */
} kla_gate;

typedef enum kla_beta_mode {
    KLA_BETA_KACZMARZ = 0,     /* beta = eta / (||k||^2 + eps): the KLA step */
    KLA_BETA_RAW = 1           /* beta = eta: DeltaNet / Gated DeltaNet write strength; eps unused */
} kla_beta_mode;

/*
 * Chunkwise prefill (GeekNews page above, section "KDA por chunks: reordenar la
 * recurrencia como multiplicaciones de matrices"; the KLA page, section
 * "Implementazione", for beta entering the chunk solver as a diagonal).
 * The result equals the token-by-token recurrence up to floating-point rounding.
 *
 *   q, k     [B, T, H, d_k]  dtype            read only
 *   v        [B, T, H, d_v]  dtype            read only
 *   alpha    fp32, [B, T, H] (KLA_GATE_SCALAR) or [B, T, H, d_k] (KLA_GATE_CHANNEL),
 *            values in (0, 1]; the log-decay is taken on the device
 *   eta      fp32 [B, T, H], any finite value (eta = 1 with eps = 0 is the exact projection)
 *   eps      stabiliser added to ||k||^2
 *   S0       fp32 [B, H, d_k, d_v] initial state, or NULL for zeros
 *   o        [B, T, H, d_v] dtype, written (rounded to nearest even for bf16)
 *   S_T      fp32 [B, H, d_k, d_v] final state, or NULL if not wanted; may be the same
 *            pointer as S0 (in-place continuation); must not overlap any other argument
 *   T        >= 0; T = 0 writes S_T = S0 (or zeros) and no outputs, and then q, k, v,
 *            alpha, eta and o may be NULL. T need not be a multiple of chunk; the last
 *            chunk is masked.
 *   chunk    tokens per chunk
 *   workspace, workspace_bytes: device scratch of at least
 *            kla_chunk_fwd_workspace_size(...) bytes (may be NULL when that size is 0); its
 *            contents need no initialisation and are unspecified after the call
 *
 * Per-key-channel gates on the tensor-core path: the in-chunk products are factorised
 * around the 32nd token of each chunk, which is exact as long as, for every key channel, the
 * product of the gates over tokens 0-31 and over tokens 32-63 of a chunk each stays above
 * e^-80 (the gates averaged over 32 tokens above about 0.082). The call first marks, in the
 * workspace, every (sequence, head) chain with a chunk near or outside that range (one pass over
 * alpha); the tensor-core kernel skips the marked chains and the same call reruns them on the
 * fp32 token-by-token path, so every alpha in (0, 1] gives valid results and KLA_OK. The marks
 * cost 4 bytes per chain of workspace. chunk = 16 or 32 runs the fp32 path throughout.
 *
 * Calls of 1 to 16 tokens (multi-token decode, speculative verification) ignore `chunk`: bf16
 * with d_k = d_v = 128 runs the call's tokens as one chunk on warp-level tensor cores from 5
 * tokens with the scalar gate and from 9 with the per-channel gate (when alpha is 16-byte
 * aligned; no in-call decay factor exceeds 1, so any gate in (0, 1] gives valid results), the
 * state rounded to bf16 as an operand as on the chunkwise path; other calls walk the
 * tokens in order on fp32 state tiles. A call's first j outputs are bit-identical to those of a
 * call with only its first j tokens when both token counts fall in the same one of the ranges
 * 1-4, 5-8 and 9-16 (bf16, scalar gate, d = 128), 1-8 and 9-16 (bf16, per-channel gate,
 * d = 128), always otherwise.
 */
kla_status kla_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *alpha, const float *eta, float eps,
                         const float *S0, void *o, float *S_T,
                         int B, int T, int H, int d_k, int d_v, int chunk,
                         kla_dtype dtype, kla_gate gate,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * kla_chunk_fwd with the step-size mode and the query scale chosen by the caller (see the top of
 * this file). kla_chunk_fwd(...) is kla_chunk_fwd_ex(..., KLA_BETA_KACZMARZ, 1.0f, ...).
 *   beta_mode  KLA_BETA_KACZMARZ or KLA_BETA_RAW; anything else is KLA_ERR_INVALID_ARG
 *   q_scale    finite scale s of the read o_t = S_t^T (s q_t); the state does not depend on it;
 *              a NaN or infinite value is KLA_ERR_INVALID_ARG
 * Arguments, layouts, workspace and errors are otherwise those of kla_chunk_fwd.
 */
kla_status kla_chunk_fwd_ex(const void *q, const void *k, const void *v,
                            const float *alpha, const float *eta, float eps,
                            const float *S0, void *o, float *S_T,
                            int B, int T, int H, int d_k, int d_v, int chunk,
                            kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode, float q_scale,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device scratch kla_chunk_fwd / kla_chunk_fwd_ex need for these sizes (0 if none):
 * the segments' states when a long sequence with few (sequence, head) chains is split into
 * segments, and with the per-channel gate on the tensor-core path the chains' rerun marks (4
 * bytes per chain). The step-size mode and the query scale do not change it. */
size_t kla_chunk_fwd_workspace_size(int B, int T, int H, int d_k, int d_v, int chunk,
                                    kla_dtype dtype, kla_gate gate);

/*
 * Chunkwise prefill that allocates nothing, for callers that cannot allocate device memory
 * (for example a runtime whose memory manager owns all device memory, or code that must not
 * allocate while work is in flight on its stream). The pages have no counterpart: it is a
 * deployment variant of kla_chunk_fwd with the same arguments, results and errors, minus the
 * workspace. The scratch that kla_chunk_fwd would take from the caller (the segments' states
 * when a long sequence with few (sequence, head) chains is split into segments, and the rerun
 * marks of the per-channel gate) comes instead from a fixed array of KLA_NOALLOC_SCRATCH_BYTES
 * inside the library's device image; every GPU that loads the library holds that array until
 * the process exits.
 *  - The arguments are checked first, exactly as kla_chunk_fwd checks them (same errors); a
 *    valid call whose scratch (kla_chunk_fwd_workspace_size) exceeds KLA_NOALLOC_SCRATCH_BYTES
 *    is then rejected with KLA_ERR_UNSUPPORTED, before anything is launched.
 *  - The first call on a device that needs scratch looks up the array's device address with
 *    that device current (a host-side runtime query, no allocation); make that first call
 *    before any stream capture.
 *  - All calls on a device share the array, and it keeps the last call's contents (each call
 *    writes every element it reads, so nothing needs clearing). Calls whose kernels may run at
 *    the same time on the GPU race on it: order them (one stream, or events).
 */
#define KLA_NOALLOC_SCRATCH_BYTES (24u << 20)
kla_status kla_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                 const float *alpha, const float *eta, float eps,
                                 const float *S0, void *o, float *S_T,
                                 int B, int T, int H, int d_k, int d_v, int chunk,
                                 kla_dtype dtype, kla_gate gate, void *stream);

/*
 * kla_chunk_fwd_ex from and to HOST memory, with the copies overlapped with the kernels: the
 * work is split into `parts` parts; part i's inputs go host -> device on one copy stream, its
 * prefill runs on a compute stream once they have landed, and its outputs go device -> host on a
 * second copy stream, so part i+1's copies overlap part i's prefill and both directions of the
 * link are busy at once. The pages have no counterpart: it
 * is the host-buffer form of kla_chunk_fwd_ex for callers whose tensors live in host memory.
 *   q_h .. S_T_h  host tensors in the layouts of kla_chunk_fwd; pinned (page-locked) memory is
 *                 needed for the copies to overlap anything (pageable memory still works, with
 *                 synchronous copies); S0_h and S_T_h may be NULL (zeros / not wanted)
 *   q_d .. S_T_d  device buffers of the same sizes, owned by the caller (S0_d / S_T_d NULL
 *                 exactly when S0_h / S_T_h are); their contents after the call are unspecified
 *                 except o_d and S_T_d, which hold the results
 *   parts         time parts: 1 .. min(64, T / 64); batch parts: 1 .. min(B, 64)
 * Time parts (bf16, scalar gate, d_k = d_v = 128, chunk 64, and parts <= T / 64; without a final
 * state also B * H * 64 KB <= 23 MiB): part i is the same slice of whole 64-token chunks of every
 * sequence (the last slice takes the remainder), copied with strided copies; the slices run in
 * order on one compute stream with the state carried between them in fp32, in S_T_d or, when no
 * final state is wanted, in the fixed array of kla_chunk_fwd_noalloc (ordered by the same event as
 * below); the results equal kla_chunk_fwd's bit for bit. Every other call takes batch parts.
 * Batch parts run whole sequences, except the last part when the sequence-parallel segments of
 * kla_chunk_fwd shorten it (long sequences, few chains per part): it then takes its scratch
 * from the fixed array of kla_chunk_fwd_noalloc (no allocation). With the per-channel gate,
 * every part's rerun marks (see kla_chunk_fwd) live in that array too: up to 32768 chains per
 * part; a part with more chains reports out-of-range gates through kla_device_status instead of
 * rerunning them. The last parts of host calls are ordered on that array by an event of the
 * library's; a kla_chunk_fwd_noalloc call whose kernels may run at the same time as a host call
 * must be ordered against it by the caller. The call is
 * asynchronous and ordered on `stream`: it starts after earlier work on `stream`, and work
 * enqueued on `stream` afterwards starts after its last copy. The library keeps two copy
 * streams, eight compute streams and a few events per device for the life of the process;
 * calls on one device are serialised by a host mutex while they enqueue. Argument errors as
 * for kla_chunk_fwd; T must be >= 1.
 */
kla_status kla_chunk_fwd_host(const void *q_h, const void *k_h, const void *v_h, const float *alpha_h,
                              const float *eta_h, const float *S0_h, void *o_h, float *S_T_h,
                              void *q_d, void *k_d, void *v_d, float *alpha_d, float *eta_d, float *S0_d,
                              void *o_d, float *S_T_d, float eps,
                              int B, int T, int H, int d_k, int d_v, int chunk,
                              kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode, float q_scale,
                              int parts, void *stream);

/*
 * One fused single-token step for B sequences (GeekNews page above, section
 * "Kernel Triton recurrente fusionado para decodificacion": forget, predict,
 * residual, outer-product write, read; the KLA step of the KLA page).
 * Each head's state is read once and written once.
 *
 *   q, k     [B, H, d_k] dtype;  v [B, H, d_v] dtype
 *   alpha    fp32 [B, H] or [B, H, d_k];  eta fp32 [B, H]
 *   S        fp32 [B, H, d_k, d_v], updated in place
 *   o        [B, H, d_v] dtype, written
 */
kla_status kla_decode_step(const void *q, const void *k, const void *v,
                           const float *alpha, const float *eta, float eps,
                           float *S, void *o,
                           int B, int H, int d_k, int d_v,
                           kla_dtype dtype, kla_gate gate, void *stream);

/* kla_decode_step with the step-size mode and the query scale of kla_chunk_fwd_ex. */
kla_status kla_decode_step_ex(const void *q, const void *k, const void *v,
                              const float *alpha, const float *eta, float eps,
                              float *S, void *o,
                              int B, int H, int d_k, int d_v,
                              kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode, float q_scale,
                              void *stream);

/*
 * Backward pass of kla_chunk_fwd_ex (training): the gradients of a scalar loss L with respect to
 * every input, given dO = dL/do and dS_T = dL/dS_T. The pages give no backward algebra; this is
 * the chain rule through the forward (the fp64 oracle of the tests, the chain rule through
 * forget, predict, residual, step size, write and read in reverse token order, is checked
 * against finite differences of the forward). Every gradient is written in fp32.
 *
 *   q, k, v, alpha, eta, eps, S0, dtype, gate, beta_mode, q_scale: as for kla_chunk_fwd_ex (the
 *            same values the forward ran with); q, k, v need only their element alignment here
 *   dO       [B, T, H, d_v] dtype                 dL/do (read only)
 *   dS_T     fp32 [B, H, d_k, d_v] or NULL (zero)  dL/dS_T (read only)
 *   dq, dk   fp32 [B, T, H, d_k]                   written
 *   dv       fp32 [B, T, H, d_v], 16-byte aligned  written
 *   dalpha   fp32, shaped like alpha               written (dL/dalpha, not dL/dlog alpha)
 *   deta     fp32 [B, T, H]                        written
 *   dS0      fp32 [B, H, d_k, d_v] or NULL         written when given (dL/dS0)
 *   workspace, workspace_bytes: 16-byte aligned device scratch of at least
 *            kla_chunk_bwd_workspace_size(...) bytes (enough for either path), or of
 *            kla_chunk_bwd_workspace_size_ex(...) bytes when q, k, v and dO are 16-byte aligned
 * Outputs must not overlap each other or any input. T = 0 writes dS0 = dS_T (or zeros) only.
 * Supported sizes: d_k, d_v in {16, 32, 64, 128}. Two paths:
 *   - bf16, d_k = d_v = 128, T > 16, 16-byte aligned q, k, v, dO, either gate: chunkwise (64-token
 *     chunks) on the tensor cores, bf16 operands with fp32 accumulation and fp32 carried states
 *     (relative L2 error ~3e-3 against fp64); the chunk-state carries of long sequences with few
 *     (sequence, head) chains run as a sequence-parallel scan; alpha must be > 0 (dalpha is formed
 *     from dL/dlog alpha). With the per-channel gate the in-chunk decays are factorised around
 *     the 32nd token of each chunk, as in kla_chunk_fwd: the call first marks, in the workspace,
 *     the (sequence, head) chains with a chunk near or outside that range, the chunkwise kernels
 *     skip them and the same call runs them on the token-by-token path below, so every alpha in
 *     (0, 1] gives valid gradients;
 *   - every other call: token by token in fp32, one CTA per (sequence, head), so the time grows
 *     with T and not with B * H.
 */
kla_status kla_chunk_bwd(const void *q, const void *k, const void *v,
                         const float *alpha, const float *eta, float eps, const float *S0,
                         const void *dO, const float *dS_T,
                         float *dq, float *dk, float *dv, float *dalpha, float *deta, float *dS0,
                         int B, int T, int H, int d_k, int d_v,
                         kla_dtype dtype, kla_gate gate, kla_beta_mode beta_mode, float q_scale,
                         void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device scratch kla_chunk_bwd needs for these sizes on either path (0 when T = 0). */
size_t kla_chunk_bwd_workspace_size(int B, int T, int H, int d_k, int d_v);

/*
 * Bytes of device scratch kla_chunk_bwd needs for these sizes, dtype and gate when q, k, v and dO
 * are 16-byte aligned: with the scalar gate the chunkwise path's records (~129 KB per 64-token
 * chunk of every chain) when it applies; with the per-channel gate on the chunkwise path, 4 bytes
 * per chain for the range marks (256-byte aligned) and room for the larger of its records (~161 KB
 * per chunk) and the token-sequential path's checkpoints (which rerun the marked chains); else
 * the token-sequential path's. Like kla_chunk_fwd_workspace_size, it may query the current
 * device's SM count (the segment plan of long sequences).
 */
size_t kla_chunk_bwd_workspace_size_ex(int B, int T, int H, int d_k, int d_v, kla_dtype dtype, kla_gate gate);

/*
 * Synchronises `stream`, then reads and clears the device-side error flags that
 * bounded waits and range checks of earlier calls on this device may have set.
 * Returns KLA_OK, KLA_ERR_TIMEOUT, KLA_ERR_INVALID_ARG (a per-channel gate outside
 * the exact range of the tensor-core path) or KLA_ERR_CUDA.
 */
kla_status kla_device_status(void *stream);

/*
 * Self-test of the failure path (no counterpart on the pages): launches one thread that waits,
 * with the bounded wait every kernel of the library uses, on a barrier phase that nothing
 * completes. After `limit_polls` polls of at most 20 us each (1 .. 100000, i.e. at most 2 s) the
 * wait gives up and records a time-out, exactly as a stuck wait inside a real kernel would; no
 * fault, trap or hang is involved and the context stays usable. The next kla_device_status()
 * on the stream returns KLA_ERR_TIMEOUT (and clears the flag). KLA_ERR_INVALID_ARG for a limit
 * out of range.
 */
kla_status kla_selftest_wait_timeout(unsigned limit_polls, void *stream);

/* Static, human-readable name of a status code. */
const char *kla_status_string(kla_status status);

/* ABI version of this header (major * 100 + minor). */
int kla_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KLA_H */
