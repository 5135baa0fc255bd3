// kla_chunk_tc.cu -- tensor-core (tcgen05) chunkwise KLA prefill for sm_103a.
//
// Scope: bf16 q/k/v/o, d_k = d_v = 128, chunk C = 64, fp32 state; scalar gate (one alpha per
// token and head) or per-key-channel gate (one alpha per token, head and key channel).
//
// Algebra (GeekNews, "Revisando las variantes de atencion lineal de la familia DeltaNet",
// section "KDA por chunks"; KLA page, section "Implementazione": beta enters only as the
// diagonal of the chunk solver). Per chunk, with incoming state S (d_k x d_v), in-chunk
// inclusive log-decay prefix G, beta_i = eta_i / (||k_i||^2 + eps):
//   R   = strict_lower(beta_i e^{G_i-G_j} k_i.k_j),   T = (I + R)^{-1}       (UT transform)
//   W   = T diag(beta e^{G}) K,   U = T diag(beta) V                         (pseudo-keys/values)
//   E   = U - W S
//   O   = diag(e^{G}) Q S + A E,  A = lower(e^{G_i-G_j} q_i.k_j)
//   S' <- e^{G_end} S + (diag(e^{G_end - G}) K)^T E
//
// One CTA per (sequence, head) walks its chunks in order. Every large product runs on the
// 5th-generation tensor cores in the transposed orientation that puts 128 rows (d_k or d_v)
// on the TMEM lanes:
//   [K;Q] K^T            -> TMEM  (KK^T | QK^T)           M=128 N=64  K=128
//   K^T (T diag(beta e^G))^T, V^T (T diag(beta))^T -> W^T, U^T        M=128 N=64  K=64
//   S^T W^T, S^T Q^T     -> (W S)^T, (Q S)^T              M=128 N=64  K=128
//   E^T_s K              -> (K_end^T E)^T                  M=128 N=128 K=64
//   E^T A^T              -> (A E)^T                        M=128 N=64  K=64
// Operands are bf16 in 128-byte-swizzled shared memory (q/k/v tiles arrive by TMA, derived
// tiles are written by the threads), accumulators are fp32 in tensor memory.
//
// Two warp groups share the SM:
//  * state group (warps 0-7): owns S^T in fp32 registers (thread = one value channel, 64 key
//    channels) and runs the chain of chunk c: S^T W^T and S^T Q^T, E, E^T K and E^T A^T, the
//    state update, the output tile and its TMA store;
//  * operand group (warps 8-15): meanwhile builds the state-independent operands of chunk
//    c+1: gates, norms, [K;Q] K^T, R and A, T = (I + R)^{-1}, W^T and U^T.
// The 64 x 64 unit-lower inverse T is computed in fp32, in place over R: 16 x 16 diagonal
// blocks by substitution, then two levels of block merging (16 -> 32 -> 64) on warp-level tf32
// MMAs. The groups hand over through mbarriers that alternate strictly (no wait can alias a
// phase two steps back): `ready` (operands of chunk c are complete), `freed` (the state group
// has consumed the single-buffered W^T tile and U^T of chunk c), `done[c&1]` (the gate vectors
// of chunk c+2 are written). The q/k stage of chunk c is refilled with chunk c+2 as soon as
// the products reading its Q and K tiles have completed; its landing (`full`) also orders the
// reuse of chunk c's A tile. The v tile is single-buffered: it takes chunk c+1 as soon as the
// U^T product of chunk c has read it. Per-channel gate: K_end alternates between two buffers,
// so the operand group's scaled tiles of chunk c+1 do not wait for E^T K_end of chunk c.
// Every tcgen05.mma is issued by one elected lane inside a warp-uniform branch.
#include <cuda.h>

#include <algorithm>

#include <mutex>

#include "kla_internal.cuh"
#include "sm103_ptx.cuh"

namespace kla {
namespace {

using namespace ptx;

constexpr int kC = 64;          // chunk
constexpr int kD = 128;         // d_k = d_v
constexpr int kGroup = 256;     // threads per warp group
constexpr int kThreads = 2 * kGroup;
constexpr uint32_t kBarState = 1, kBarOperand = 2;   // named barriers of the two groups
constexpr uint32_t kBarPair0 = 3;                     // 3..6: warp pairs of the operand group (solve)
constexpr float kMinLogGate = -80.0f;
constexpr float kSafeDecay = -80.0f;   // chunk decay above which e^{-G_j} is representable
constexpr uint32_t kWaitLimit = 100000;   // x 20 us: a stuck wait gives up after ~2 s

// ---- shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_QK = 0;                        // 2 stages x 32 KB: [blk0: K rows | Q rows][blk1 ...]
constexpr uint32_t QK_STAGE = 32768;
constexpr uint32_t OFF_V = OFF_QK + 2 * QK_STAGE;     // 16 KB: v tile [blk0: 64 rows][blk1: 64 rows], refilled
                                                      // as soon as the U^T product has read it
constexpr uint32_t OFF_KE1 = OFF_V + 16384;           // 16 KB: per-channel gate: K_end of odd chunks
constexpr uint32_t OFF_AQK = OFF_KE1 + 16384;         // 2 x 8 KB: A (query rows) bf16, K-major
constexpr uint32_t OFF_WT = OFF_AQK + 2 * 8192;       // 16 KB: T_K | T_V bf16 for the W^T/U^T MMAs, then W^T bf16
constexpr uint32_t OFF_ST = OFF_WT + 16384;           // 32 KB: S^T bf16, K-major, 2 blocks of 128 rows
constexpr uint32_t OFF_ET = OFF_ST + 32768;           // 16 KB: E^T bf16
constexpr uint32_t OFF_ETS = OFF_ET + 16384;          // 16 KB: E^T diag(e^{G_end-G}) bf16, then O staging
                                                      // (per-channel gate: K_end of even chunks)
constexpr uint32_t OFF_R = OFF_ETS + 16384;           // 16 KB: R fp32, overwritten in place by T = (I + R)^{-1}
constexpr uint32_t OFF_XS = OFF_R + 16384;            // 7 KB: solve scratch
constexpr uint32_t OFF_SMALL = OFF_XS + 7168;         // per-chunk vectors + barriers
constexpr uint32_t SMALL_BYTES = 10240;
constexpr uint32_t SMEM_BYTES = OFF_SMALL + SMALL_BYTES + 1024;   // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory");

// ---- tensor memory columns (512 allocated)
constexpr uint32_t TM_A = 0;      // [KK^T ; QK^T]     64 cols
constexpr uint32_t TM_W = 64;     // W^T               64
constexpr uint32_t TM_U = 128;    // U^T               64
constexpr uint32_t TM_1A = 192;   // (W S)^T           64
constexpr uint32_t TM_1B = 256;   // (Q S)^T           64
constexpr uint32_t TM_3 = 320;    // (A E)^T           64
constexpr uint32_t TM_2 = 384;    // (K_end^T E)^T     128


struct ChunkVec {          // per-chunk vectors (three buffers, by chunk index mod 3)
    float G[kC];           // inclusive prefix of log-gates
    float beta[kC];
    float eG[kC];          // e^{G_i}
    float enG[kC];         // e^{-G_i} (valid when `safe`)
    float eEnd[kC];        // e^{G_end - G_i}
    float eta[kC];
    int safe;              // G_end >= kSafeDecay: e^{G_i - G_j} = e^{G_i} e^{-G_j} without overflow
    int pad[3];
};
// Per-key-channel vectors of one chunk (per-channel gate only), double-buffered by parity.
// r = kRef is the in-chunk reference token: every factor e^{G_i - G_r} or e^{G_r - G_i} spans
// at most 32 tokens of decay.
constexpr int kRef = 31;
static_assert(kRef == kC / 2 - 1, "the per-channel products split the chunk into two halves of 32 tokens");
struct ChanVec {
    float eGr[kD];         // e^{G_r}: scales the state operand
    float gam[kD];         // e^{G_end}: decay of the state over the chunk
    float F[kD];           // e^{G_end - G_r}
};
struct Small {
    ChunkVec v[3];                 // chunk c uses buffer c % 3: the vectors of chunk c+2 can be
    ChanVec ch[3];                 // written while chunks c and c+1 are still in use
    uint64_t full[2];              // q/k stage landed (TMA), by chunk parity
    uint64_t fullv;                // v tile landed (TMA), once per chunk
    uint64_t m2k[2];               // per-channel gate: E^T K_end of chunk c done (its K_end buffer c & 1 is free)
    uint64_t mA, mW, m1, m2, mO;   // tcgen05.commit of the five MMA groups
    uint64_t ready, freed;         // operand group -> state group, state group -> operand group
    uint64_t done[2];              // gate vectors of chunk c+2 written, by the parity of c
    uint32_t tmem_base;
    volatile int abort;
};
static_assert(sizeof(Small) <= SMALL_BYTES, "small area");

// Initial state and final state addressing. A launch covers `seg_count` segments of every
// (sequence, head) chain, starting at segment `seg_begin`; segment s spans tokens
// [s * seg_len, min(T, (s + 1) * seg_len)). A whole-sequence call is one segment.
enum : int {
    kS0Chain = 0,      // S0 + bh * d^2 for the chain's first segment, zeros for later segments (NULL: zeros)
    kS0Segment = 1,    // S0 + (bh * nseg + s) * d^2
    kS0Identity = 2,   // the identity (the transition of a segment is its final state from S0 = I, v = 0)
    kSTLast = 0,       // S_T + bh * d^2, written by the chain's last segment only (NULL: not written)
    kSTSegment = 1,    // S_T + (bh * nseg + s) * d^2
};
struct TcParams {
    const float *alpha, *eta;   // alpha: [B,T,H] (scalar gate) or [B,T,H,d_k] (per-channel gate)
    float eps;
    const float *S0;
    float *S_T;
    int B, T, H;
    int seg_len, seg_begin, seg_count, nseg;   // segments (seg_len a multiple of the chunk)
    int s0_mode, st_mode;
    int zero_v;    // treat v as zero (U = 0): the transition run of a segment
    int no_out;    // 0: write o; 1: no output; 2: only the chain's first segment writes o
    unsigned *err;
    int beta_raw;  // 1: beta = eta
    float q_scale; // o = S^T (q_scale q)
    const unsigned *rescue;   // per-channel gate: [B*H] marks of chains rerun exactly (skipped here), or NULL
    int Ts;                   // tokens between sequences in alpha and eta (T, or more for a slice)
};

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }
// fp32 64 x 64 matrices in shared memory, rows of 64 with the float4 groups of each 32-column
// half permuted by the row (keeps row-vector stores and the mma fragment loads conflict-free).
__device__ __forceinline__ int fidx(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }

__device__ __forceinline__ void st_v4_f32(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}
__device__ __forceinline__ void st_bf16x8(uint32_t addr, const float *x) {
    st_shared_v4(addr, pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}
__device__ __forceinline__ void st_bf16x8u(uint32_t addr, const uint32_t *x) {
    st_shared_v4(addr, pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                 pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                 pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                 pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
}

template <bool kCh>   // per-key-channel gate
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const TcParams p) {
    // a chain marked for the exact rerun is skipped entirely (its S0 stays as it is)
    if (p.rescue && p.rescue[blockIdx.x / p.seg_count] != 0u) return;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the shared array itself so that every access below
    // stays a shared-memory access (no generic addressing)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    Small &sm = *reinterpret_cast<Small *>(smem + OFF_SMALL);
    float *Rm = reinterpret_cast<float *>(smem + OFF_R);    // R, swizzled fp32 [64][64]
    float *Tm = Rm;                                         // T replaces R block by block
    float *Xs = reinterpret_cast<float *>(smem + OFF_XS);   // solve scratch
    __shared__ int abort_snap[2];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = warp >> 3;                  // 0: state group, 1: operand group
    const int gw = warp & 7, gtid = tid & (kGroup - 1);
    const int half = gw >> 2;
    const int row = (warp & 3) * 32 + lane;     // TMEM lane of this thread
    const int g8 = lane >> 2, t4 = lane & 3;    // mma.sync fragment coordinates
    const int bh = blockIdx.x / p.seg_count;
    const int seg = p.seg_begin + static_cast<int>(blockIdx.x) % p.seg_count;
    const int b = bh / p.H, h = bh % p.H;
    const int t_begin = seg * p.seg_len, t_end = min(p.T, t_begin + p.seg_len);
    const int nchunks = (t_end - t_begin + kC - 1) / kC;
    const bool write_out = p.no_out == 0 || (p.no_out == 2 && seg == 0);

    const uint32_t bar_full0 = smem_u32(&sm.full[0]);
    const uint32_t bar_A = smem_u32(&sm.mA), bar_W = smem_u32(&sm.mW);
    const uint32_t bar_1 = smem_u32(&sm.m1), bar_2 = smem_u32(&sm.m2), bar_o = smem_u32(&sm.mO);
    const uint32_t bar_ready = smem_u32(&sm.ready), bar_freed = smem_u32(&sm.freed);
    const uint32_t bar_done0 = smem_u32(&sm.done[0]);
    const uint32_t bar_fullv = smem_u32(&sm.fullv), bar_m2k0 = smem_u32(&sm.m2k[0]);

    if (tid == 0) {
        mbar_init(bar_full0, 1);
        mbar_init(bar_full0 + 8, 1);
        mbar_init(bar_A, 1);
        mbar_init(bar_W, 1);
        mbar_init(bar_1, 1);
        mbar_init(bar_2, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_ready, 1);
        mbar_init(bar_freed, 1);
        mbar_init(bar_done0, 1);
        mbar_init(bar_done0 + 8, 1);
        mbar_init(bar_fullv, 1);
        mbar_init(bar_m2k0, 1);
        mbar_init(bar_m2k0 + 8, 1);
        sm.abort = 0;
        abort_snap[0] = abort_snap[1] = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_o);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&sm.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;
    const uint32_t tlane = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);

    const uint32_t id_qk = idesc_bf16(128, 64, 0, 0);     // K-major x K-major, N=64
    const uint32_t id_w = idesc_bf16(128, 64, 1, 0);      // MN-major A, K-major B
    const uint32_t id_1a = idesc_bf16(128, 64, 0, 1);     // K-major A, MN-major B
    const uint32_t id_2 = idesc_bf16(128, 128, 0, 1);     // N=128, MN-major B

    auto qk_of = [&](int c) { return sbase + OFF_QK + (c & 1) * QK_STAGE; };
    auto v_of = [&](int) { return sbase + OFF_V; };
    auto ke_of = [&](int c) { return sbase + ((c & 1) ? OFF_KE1 : OFF_ETS); };   // per-channel gate: K_end
    auto aqk_of = [&](int c) { return sbase + OFF_AQK + (c & 1) * 8192; };

    auto issue_loads = [&](int c) {   // q and k tiles of chunk c; one thread
        const uint32_t bar = bar_full0 + 8 * (c & 1);
        const uint32_t qk = qk_of(c);
        mbar_arrive_expect_tx(bar, 4 * 8192);
        const int t0 = t_begin + c * kC;
        tma_load_4d(qk + 0, &tm_k, bar, 0, h, t0, b);
        tma_load_4d(qk + 8192, &tm_q, bar, 0, h, t0, b);
        tma_load_4d(qk + 16384, &tm_k, bar, 64, h, t0, b);
        tma_load_4d(qk + 24576, &tm_q, bar, 64, h, t0, b);
    };
    auto issue_v = [&](int c) {   // v tile of chunk c; one thread
        const uint32_t vv = v_of(c);
        mbar_arrive_expect_tx(bar_fullv, 2 * 8192);
        const int t0 = t_begin + c * kC;
        tma_load_4d(vv + 0, &tm_v, bar_fullv, 0, h, t0, b);
        tma_load_4d(vv + 8192, &tm_v, bar_fullv, 64, h, t0, b);
    };
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!mbar_wait_bounded(bar, parity, kWaitLimit)) sm.abort = 1;
    };
    const uint32_t gbar = grp == 0 ? kBarState : kBarOperand;
    auto gsync = [&]() { named_sync(gbar, kGroup); };
    // Uniform per-group abort decision: one thread snapshots the flag before a group barrier.
    auto group_aborted = [&]() {
        if (gtid == 0) abort_snap[grp] = sm.abort;
        gsync();
        return abort_snap[grp] != 0;
    };

    if (tid == 0) {
        issue_loads(0);
        if (nchunks > 1) issue_loads(1);
        if (!p.zero_v) issue_v(0);
    }

    // Per-token gate vectors (G, e^{G}, e^{-G}, e^{G_end - G}, eta) of a chunk are computed by
    // warp 0 of the state group two chunks ahead, from gates it prefetched into registers (two
    // tokens per lane), and handed to the operand group through `done`.
    float a_nx[2] = {1.f, 1.f}, e_nx[2] = {0.f, 0.f};
    auto load_gates = [&](int c) {
        if (warp == 0 && c < nchunks) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = t_begin + c * kC + 2 * lane + u;
                const bool ok = t < t_end;
                const size_t tok = (static_cast<size_t>(b) * p.Ts + t) * p.H + h;
                a_nx[u] = (ok && !kCh) ? p.alpha[tok] : 1.f;
                e_nx[u] = ok ? p.eta[tok] : 0.f;
            }
        }
    };
    auto gate_vec = [&](int c) {   // warp 0 only
        if (c >= nchunks) return;
        ChunkVec &cv = sm.v[c % 3];
        const float g0 = fmaxf(__logf(a_nx[0]), kMinLogGate), g1 = fmaxf(__logf(a_nx[1]), kMinLogGate);
        float s = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        const float gend = __shfl_sync(0xffffffffu, s, 31);
        const float G0 = s - g1, G1 = s;
        cv.G[2 * lane] = G0;
        cv.G[2 * lane + 1] = G1;
        cv.eG[2 * lane] = __expf(G0);
        cv.eG[2 * lane + 1] = __expf(G1);
        cv.enG[2 * lane] = __expf(-G0);
        cv.enG[2 * lane + 1] = __expf(-G1);
        cv.eEnd[2 * lane] = __expf(gend - G0);
        cv.eEnd[2 * lane + 1] = __expf(gend - G1);
        cv.eta[2 * lane] = e_nx[0];
        cv.eta[2 * lane + 1] = e_nx[1];
        if (lane == 0) cv.safe = kCh ? 1 : (gend >= kSafeDecay);
    };
    if (warp == 0) {   // chunks 0 and 1 before the groups split; chunk 2 prefetched
        load_gates(0);
        gate_vec(0);
        load_gates(1);
        gate_vec(1);
        load_gates(2);
    }
    __syncthreads();

    // ===================================================================== operand group
    // Per-channel gates (per-channel gate only): thread = (8-channel group cg, token half th,
    // 4-token sub-range sb of the half): lanes sb = lane % 8 of one warp share (cg, th), so the
    // running products of the gates across a half are shuffle scans over those 8 lanes. A thread
    // holds its 4 x 8 gates of the next chunk; the loads are issued a chunk ahead and left
    // untouched until their first use (`chgate`), so the thread does not wait for them. Tokens
    // past the end load the last token's gate and read as 1, and gates are clamped to e^-80 like
    // the log-gates.
    const int csb = lane & 7, cgth = gw * 4 + (lane >> 3);
    const int ccg = cgth & 15, cth = cgth >> 4;
    float ga[kCh ? 4 : 1][kCh ? 8 : 1];
    auto load_chgates = [&](int c) {
        if constexpr (kCh) {
            if (grp == 1 && c < nchunks) {
                // the 4 tokens are consecutive rows: one base address and a row stride (tokens past
                // the end reread the last row)
                const int t = t_begin + c * kC + 32 * cth + 4 * csb, tl = min(t, t_end - 1);
                const float *g0 = p.alpha + ((static_cast<size_t>(b) * p.Ts + tl) * p.H + h) * kD + 8 * ccg;
                const size_t rs = static_cast<size_t>(p.H) * kD;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float *gu = g0 + (t + u < t_end ? u : t_end - 1 - tl) * rs;
#pragma unroll
                    for (int j = 0; j < 8; ++j) ga[u][j] = gu[j];
                }
            }
        }
    };
    // gate of token u of this thread's sub-range, channel j of its group; inb[u]: token u is inside the
    // sequence (formed once per chunk)
    auto chgate = [&](const bool (&inb)[4], int u, int j) { return inb[u] ? fmaxf(ga[u][j], 1.8e-35f) : 1.f; };
    auto in_bounds = [&](int c, bool (&inb)[4]) {
#pragma unroll
        for (int u = 0; u < 4; ++u) inb[u] = t_begin + c * kC + 32 * cth + 4 * csb + u < t_end;
    };

    // (a) gates, norms, beta and the decay tables; issue [K;Q] K^T.
    auto op_front = [&](int c) {
        ChunkVec &cv = sm.v[c % 3];
        const uint32_t qk = qk_of(c);
        if (c >= 2) wait(bar_done0 + 8 * (c & 1), ((c - 2) >> 1) & 1);   // gate vectors of chunk c
        // per-channel: products of the gates over each half of the chunk; `ex` is the product over
        // the sub-ranges between this thread's and the reference token (before it in half 1, after
        // it in half 0), `tot` over the whole half
        float ex[kCh ? 8 : 1];
        bool inb[4];
        if constexpr (kCh) {
            in_bounds(c, inb);
            bool low = false;
            float tot[8];
            // the scan runs towards the reference token: from lane csb - off (half 1) or csb + off
            // (half 0) of the 8-lane group, one indexed shuffle a step
            const int dir = cth ? -1 : 1;
            const int src1 = (csb + dir) & 7, src2 = (csb + 2 * dir) & 7, src4 = (csb + 4 * dir) & 7;
            const bool in1 = cth ? csb >= 1 : csb + 1 < 8, in2 = cth ? csb >= 2 : csb + 2 < 8,
                       in4 = cth ? csb >= 4 : csb + 4 < 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float l = 1.f;
#pragma unroll
                for (int u = 0; u < 4; ++u) l *= chgate(inb, u, j);
                float sc = l;   // inclusive scan towards the reference token
                float y = __shfl_sync(0xffffffffu, sc, src1, 8);
                if (in1) sc *= y;
                y = __shfl_sync(0xffffffffu, sc, src2, 8);
                if (in2) sc *= y;
                y = __shfl_sync(0xffffffffu, sc, src4, 8);
                if (in4) sc *= y;
                const float nb = __shfl_sync(0xffffffffu, sc, src1, 8);
                ex[j] = in1 ? nb : 1.f;
                tot[j] = __shfl_sync(0xffffffffu, sc, cth ? 7 : 0, 8);
                low |= tot[j] < 1.8e-35f;
            }
            ChanVec &chv = sm.ch[c % 3];
            if (csb == 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) (cth ? chv.F : chv.eGr)[8 * ccg + j] = tot[j];   // e^{G_end-G_r} | e^{G_r}
                if (low) atomicOr(p.err, kErrGateRange);   // no flag array: the range error is reported
            }
        }
        wait(bar_full0 + 8 * (c & 1), (c >> 1) & 1);
        if (!kCh && gw == 0) {   // scalar gate: [K;Q] K^T needs only the tiles; issue it first
            tc_fence_after();
            if (elect_one()) {
                const uint64_t dq = sw128_desc(qk, 16, 1024);
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                    mma_bf16(tbase + TM_A, desc_add(dq, off), desc_add(dq, off), id_qk, s);
                }
                mma_commit(bar_A);
            }
            __syncwarp();
        }
        // ||k_i||^2: 4 threads per key row, 32 channels each
        float n2 = 0.f;
        {
            const int i = gtid >> 2, part = gtid & 3;
            const uint32_t base = qk + (part >> 1) * 16384;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 x = ld_shared_v4(base + sw128_off(i, (part & 1) * 64 + 16 * j));
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float lo = bf16lo(w[u]), hi = bf16hi(w[u]);
                    n2 = fmaf(lo, lo, n2);
                    n2 = fmaf(hi, hi, n2);
                }
            }
            n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
            n2 += __shfl_xor_sync(0xffffffffu, n2, 2);
        }
        gsync();   // eta of this chunk visible
        if ((gtid & 3) == 0) cv.beta[gtid >> 2] = kla_beta(cv.eta[gtid >> 2], n2, p.eps, p.beta_raw);
        uint32_t kb_stride = 16384, kb_base = qk;   // B operand of [K;Q] K^T: raw K rows
        if constexpr (kCh) {
            // Scaled tiles with reference token r: K_r = K e^{G-G_r}, Q_r = Q e^{G-G_r} (in place),
            // K_m = K e^{G_r-G} (B of [K_r;Q_r] K_m^T, over the R area) and K_end = K e^{G_end-G}
            // (B of E^T K_end, over the E^T_s area, free once E^T K_end of chunk c-1 has run).
            ChanVec &chv = sm.ch[c % 3];
            float Fv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) Fv[j] = chv.F[8 * ccg + j];
            if (cth == 0 && csb == 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) chv.gam[8 * ccg + j] = chv.eGr[8 * ccg + j] * Fv[j];   // e^{G_end}
            }
            // K_end of this chunk goes to buffer c & 1: E^T K_end of chunk c-2 must have read it
            if (c >= 2) wait(bar_m2k0 + 8 * (c & 1), ((c - 2) >> 1) & 1);
            const uint32_t blk = ccg >> 3, colb = (ccg & 7) * 16;
            const uint32_t Kt = qk + blk * 16384, Qt = Kt + 8192;
            const uint32_t Km = sbase + OFF_R + blk * 8192, Ke = ke_of(c) + blk * 8192;
            float run[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) run[j] = ex[j];
#pragma unroll
            for (int step = 0; step < 4; ++step) {
                // half 1: tokens ascending from the reference, run = e^{G_i - G_r}; half 0: tokens
                // descending towards the chunk start, run = e^{G_r - G_i} (the factors scale bf16
                // operands: the fast reciprocal's 2 ulp are far below bf16's)
                const int u = cth ? step : 3 - step;
                const int i = 32 * cth + 4 * csb + u;
                float fr[8], fm[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (cth) {
                        run[j] *= chgate(inb, u, j);
                        fr[j] = run[j];
                        fm[j] = __fdividef(1.f, run[j]);
                    } else {
                        fm[j] = run[j];
                        fr[j] = __fdividef(1.f, run[j]);
                        run[j] *= chgate(inb, u, j);
                    }
                }
                const uint32_t off = sw128_off(i, colb);
                const uint4 kx = ld_shared_v4(Kt + off), qx = ld_shared_v4(Qt + off);
                const uint32_t kw[4] = {kx.x, kx.y, kx.z, kx.w}, qw[4] = {qx.x, qx.y, qx.z, qx.w};
                uint32_t o1[4], o2[4], o3[4], o4[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {   // channel pairs, on packed fp32 multiplies
                    const float2 k2 = make_float2(bf16lo(kw[w]), bf16hi(kw[w]));
                    const float2 q2 = make_float2(bf16lo(qw[w]), bf16hi(qw[w]));
                    const float2 fr2 = make_float2(fr[2 * w], fr[2 * w + 1]), fm2 = make_float2(fm[2 * w], fm[2 * w + 1]);
                    const float2 a = __fmul2_rn(k2, fr2), bq = __fmul2_rn(q2, fr2), m = __fmul2_rn(k2, fm2),
                                 e = __fmul2_rn(m, make_float2(Fv[2 * w], Fv[2 * w + 1]));   // K_m e^{G_end-G_r}
                    o1[w] = pack_bf16(a.x, a.y);
                    o2[w] = pack_bf16(bq.x, bq.y);
                    o3[w] = pack_bf16(m.x, m.y);
                    o4[w] = pack_bf16(e.x, e.y);
                }
                st_shared_v4(Kt + off, o1[0], o1[1], o1[2], o1[3]);
                st_shared_v4(Qt + off, o2[0], o2[1], o2[2], o2[3]);
                st_shared_v4(Km + off, o3[0], o3[1], o3[2], o3[3]);
                st_shared_v4(Ke + off, o4[0], o4[1], o4[2], o4[3]);
            }
            load_chgates(c + 1);
            fence_proxy_async_smem();
            gsync();
            kb_stride = 8192;
            kb_base = sbase + OFF_R;
        }
        if (kCh && gw == 0) {
            tc_fence_after();
            if (elect_one()) {
                const uint64_t dq = sw128_desc(qk, 16, 1024), dkb = sw128_desc(kb_base, 16, 1024);
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                    const uint32_t boff = (s >> 2) * kb_stride + (s & 3) * 32;
                    mma_bf16(tbase + TM_A, desc_add(dq, off), desc_add(dkb, boff), id_qk, s);
                }
                mma_commit(bar_A);
            }
            __syncwarp();
        }
    };

    // W^T = K^T T_K^T and U^T = V^T T_V^T of chunk c (scalar gate); per-channel gate: W_r^T =
    // K_r^T T_V^T (the factor e^{G_r} of W is carried by the state operand instead).
    auto issue_wu = [&](int c) {   // one thread
        tc_fence_after();
        const uint32_t qk = qk_of(c), vv = v_of(c);
        const uint32_t tw = sbase + OFF_WT + (kCh ? 8192 : 0);
        const uint64_t dk = sw128_desc(qk, 16384, 1024), dtw = sw128_desc(tw, 16, 1024);
#pragma unroll
        for (int s = 0; s < 4; ++s) mma_bf16(tbase + TM_W, desc_add(dk, s * 2048), desc_add(dtw, s * 32), id_w, s);
        if (!p.zero_v) {
            if (!mbar_wait_bounded(bar_fullv, c & 1, kWaitLimit)) sm.abort = 1;   // v tile of chunk c
            const uint64_t dv = sw128_desc(vv, 8192, 1024), dtv = sw128_desc(sbase + OFF_WT + 8192, 16, 1024);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tbase + TM_U, desc_add(dv, s * 2048), desc_add(dtv, s * 32), id_w, s);
        }
        mma_commit(bar_W);
    };
    // (b) R and A from [KK^T; QK^T]; T = (I + R)^{-1}; T_K, T_V; issue W^T, U^T.
    auto op_mid = [&](int c) {
        ChunkVec &cv = sm.v[c % 3];
        gsync();   // beta of this chunk visible
        wait(bar_A, c & 1);
        tc_fence_after();
        {
            // two passes of 16 columns keep the live registers low
            const int i = row & (kC - 1);
            const bool key_row = row < kC;
            const float scale = key_row ? cv.beta[i] : 1.f;
            const bool safe = cv.safe != 0;
            const float ei = cv.eG[i] * scale, Gi = cv.G[i];
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
                uint32_t v[16];
                tmem_ld16(tlane + TM_A + 32 * half + 16 * pc, v);
                tmem_ld_wait();
                const int j0 = 32 * half + 16 * pc;
                float x[16];
                if (kCh) {   // the decay is inside the scaled operands
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        const bool keep = key_row ? (j < i) : (j <= i);
                        x[jj] = keep ? scale * __uint_as_float(v[jj]) : 0.f;
                    }
                } else if (safe) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float4 en = *reinterpret_cast<const float4 *>(&cv.enG[j0 + 4 * q4]);
                        const float e4[4] = {en.x, en.y, en.z, en.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int jj = 4 * q4 + u, j = j0 + jj;
                            const bool keep = key_row ? (j < i) : (j <= i);
                            x[jj] = keep ? ei * e4[u] * __uint_as_float(v[jj]) : 0.f;
                        }
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        const bool keep = key_row ? (j < i) : (j <= i);
                        x[jj] = keep ? scale * __expf(Gi - cv.G[j]) * __uint_as_float(v[jj]) : 0.f;
                    }
                }
                if (key_row) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        st_v4_f32(Rm + fidx(i, j0 + 4 * q4), x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
                } else {
                    const uint32_t base = aqk_of(c);
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch)
                        st_bf16x8(base + sw128_off(i, half * 64 + pc * 32 + ch * 16), x + 8 * ch);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        gsync();
        // ---- diagonal 16x16 blocks (one per warp pair): right-looking substitution in steps of
        // 4 rows. Lane = (row group r4 = lane / 8, column l = 8 (warp & 1) + lane % 8); the lanes of
        // row group jb finalise their 4 rows, broadcast them by shuffle, and the lanes below update.
        {
            const int o = 16 * (gw >> 1);
            const int l = 8 * (gw & 1) + (lane & 7), r4 = lane >> 3;
            float acc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[u] = (4 * r4 + u == l) ? 1.f : 0.f;
#pragma unroll
            for (int jb = 0; jb < 4; ++jb) {
                if (r4 == jb) {   // 4 x 4 substitution on the diagonal sub-block
#pragma unroll
                    for (int u = 1; u < 4; ++u) {
                        const float4 rr = *reinterpret_cast<const float4 *>(Rm + fidx(o + 4 * jb + u, o + 4 * jb));
                        const float rv[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
                        for (int v2 = 0; v2 < u; ++v2) acc[u] = fmaf(-rv[v2], acc[v2], acc[u]);
                    }
                }
                float xb[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) xb[u] = __shfl_sync(0xffffffffu, acc[u], jb * 8 + (lane & 7));
                if (r4 > jb) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 rr = *reinterpret_cast<const float4 *>(Rm + fidx(o + 4 * r4 + u, o + 4 * jb));
                        acc[u] = fmaf(-rr.x, xb[0], acc[u]);
                        acc[u] = fmaf(-rr.y, xb[1], acc[u]);
                        acc[u] = fmaf(-rr.z, xb[2], acc[u]);
                        acc[u] = fmaf(-rr.w, xb[3], acc[u]);
                    }
                }
            }
            // both warps of the pair have read this block of R: replace it by the block of T
            named_sync(kBarPair0 + (gw >> 1), 64);
#pragma unroll
            for (int u = 0; u < 4; ++u) Tm[fidx(o + 4 * r4 + u, o + l)] = acc[u];
        }
        gsync();
        // ---- merge 16 -> 32: T_{2p+1,2p} = -T_{2p+1,2p+1} (R_{2p+1,2p} T_{2p,2p}) (warps 0-3, tf32 mma)
        if (gw < 4) {
            const int pp = gw >> 1, nt = gw & 1;
            const int r0 = 16 * (2 * pp + 1), c0 = 16 * (2 * pp);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const uint32_t a[4] = {to_tf32(Rm[fidx(r0 + g8, c0 + 8 * ks + t4)]),
                                       to_tf32(Rm[fidx(r0 + g8 + 8, c0 + 8 * ks + t4)]),
                                       to_tf32(Rm[fidx(r0 + g8, c0 + 8 * ks + t4 + 4)]),
                                       to_tf32(Rm[fidx(r0 + g8 + 8, c0 + 8 * ks + t4 + 4)])};
                const uint32_t bb[2] = {to_tf32(Tm[fidx(c0 + 8 * ks + t4, c0 + 8 * nt + g8)]),
                                        to_tf32(Tm[fidx(c0 + 8 * ks + t4 + 4, c0 + 8 * nt + g8)])};
                mma_tf32_16x8x8(d, a, bb);
            }
            float *X = Xs + gw * 128;   // 16 x 8, row stride 8
            X[g8 * 8 + 2 * t4] = d[0];
            X[g8 * 8 + 2 * t4 + 1] = d[1];
            X[(g8 + 8) * 8 + 2 * t4] = d[2];
            X[(g8 + 8) * 8 + 2 * t4 + 1] = d[3];
            __syncwarp();
            float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const uint32_t a[4] = {to_tf32(Tm[fidx(r0 + g8, r0 + 8 * ks + t4)]),
                                       to_tf32(Tm[fidx(r0 + g8 + 8, r0 + 8 * ks + t4)]),
                                       to_tf32(Tm[fidx(r0 + g8, r0 + 8 * ks + t4 + 4)]),
                                       to_tf32(Tm[fidx(r0 + g8 + 8, r0 + 8 * ks + t4 + 4)])};
                const uint32_t bb[2] = {to_tf32(X[(8 * ks + t4) * 8 + g8]), to_tf32(X[(8 * ks + t4 + 4) * 8 + g8])};
                mma_tf32_16x8x8(e, a, bb);
            }
            const int cc = c0 + 8 * nt + 2 * t4;
            named_sync(kBarPair0 + pp, 64);   // both warps of the pair have read R_{r0,c0}
            Tm[fidx(r0 + g8, cc)] = -e[0];
            Tm[fidx(r0 + g8, cc + 1)] = -e[1];
            Tm[fidx(r0 + g8 + 8, cc)] = -e[2];
            Tm[fidx(r0 + g8 + 8, cc + 1)] = -e[3];
        }
        gsync();
        // ---- merge 32 -> 64: T_{32:,0:32} = -T_{32:,32:} (R_{32:,0:32} T_{0:32,0:32}) (8 warps)
        {
            const int mt = gw >> 2, nt = gw & 3;
            float *X2 = Xs + 512;   // 32 x 32, row stride 40
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                if (ks < nt) continue;   // T_{0:32,0:32} is lower triangular
                const int ra = 32 + 16 * mt;
                const uint32_t a[4] = {to_tf32(Rm[fidx(ra + g8, 8 * ks + t4)]),
                                       to_tf32(Rm[fidx(ra + g8 + 8, 8 * ks + t4)]),
                                       to_tf32(Rm[fidx(ra + g8, 8 * ks + t4 + 4)]),
                                       to_tf32(Rm[fidx(ra + g8 + 8, 8 * ks + t4 + 4)])};
                const uint32_t bb[2] = {to_tf32(Tm[fidx(8 * ks + t4, 8 * nt + g8)]),
                                        to_tf32(Tm[fidx(8 * ks + t4 + 4, 8 * nt + g8)])};
                mma_tf32_16x8x8(d, a, bb);
            }
            const int rr = 16 * mt + g8, cc = 8 * nt + 2 * t4;
            X2[rr * 40 + cc] = d[0];
            X2[rr * 40 + cc + 1] = d[1];
            X2[(rr + 8) * 40 + cc] = d[2];
            X2[(rr + 8) * 40 + cc + 1] = d[3];
            gsync();
            float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                if (ks > 2 * mt + 1) continue;   // T_{32:,32:} is lower triangular
                const int ra = 32 + 16 * mt;
                const uint32_t a[4] = {to_tf32(Tm[fidx(ra + g8, 32 + 8 * ks + t4)]),
                                       to_tf32(Tm[fidx(ra + g8 + 8, 32 + 8 * ks + t4)]),
                                       to_tf32(Tm[fidx(ra + g8, 32 + 8 * ks + t4 + 4)]),
                                       to_tf32(Tm[fidx(ra + g8 + 8, 32 + 8 * ks + t4 + 4)])};
                const uint32_t bb[2] = {to_tf32(X2[(8 * ks + t4) * 40 + 8 * nt + g8]),
                                        to_tf32(X2[(8 * ks + t4 + 4) * 40 + 8 * nt + g8])};
                mma_tf32_16x8x8(e, a, bb);
            }
            const int ro = 32 + rr;
            Tm[fidx(ro, cc)] = -e[0];
            Tm[fidx(ro, cc + 1)] = -e[1];
            Tm[fidx(ro + 8, cc)] = -e[2];
            Tm[fidx(ro + 8, cc + 1)] = -e[3];
        }
        gsync();
        // ---- T_K = T diag(beta e^G), T_V = T diag(beta): bf16 K-major (rows n, k contiguous)
        {
            const int n = gtid >> 2, kq = gtid & 3;
            float tk[16], tv[16];
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
                const int k0 = 16 * kq + 4 * u4;
                const float4 t = *reinterpret_cast<const float4 *>(Tm + fidx(n, k0));
                const float4 bt = *reinterpret_cast<const float4 *>(&cv.beta[k0]);
                const float4 eg = *reinterpret_cast<const float4 *>(&cv.eG[k0]);
                const float tt[4] = {t.x, t.y, t.z, t.w}, b4[4] = {bt.x, bt.y, bt.z, bt.w};
                const float g4[4] = {eg.x, eg.y, eg.z, eg.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float val = (k0 + u <= n) ? tt[u] : 0.f;
                    tv[4 * u4 + u] = val * b4[u];
                    tk[4 * u4 + u] = tv[4 * u4 + u] * g4[u];
                }
            }
            // T_K/T_V go to the W^T tile area: wait until the state group has consumed W^T and U^T
            // of chunk c-1 (and so the W^T/U^T MMAs of chunk c-1 have read their T_K/T_V)
            if (c >= 1) wait(bar_freed, (c - 1) & 1);
            const uint32_t bk = sbase + OFF_WT, bv = sbase + OFF_WT + 8192;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const uint32_t off = sw128_off(n, 32 * kq + 16 * hh);
                st_bf16x8(bk + off, tk + 8 * hh);
                st_bf16x8(bv + off, tv + 8 * hh);
            }
        }
        fence_proxy_async_smem();
        gsync();
        if (gw == 0) {
            tc_fence_after();
            if (elect_one()) {
                issue_wu(c);
                mbar_arrive(bar_ready);   // A, gate vectors and tiles of chunk c written; W^T/U^T in flight
            }
            __syncwarp();
        }
    };


    // ======================================================================= state group
    // S^T: this thread owns value channel m = row, key channels [64*half, 64*half + 64).
    float s_reg[64];
    if (grp == 0) {
        const float *S0 = nullptr;
        if (p.s0_mode == kS0Segment) S0 = p.S0 + (static_cast<size_t>(bh) * p.nseg + seg) * kD * kD;
        else if (p.s0_mode == kS0Chain && p.S0 && seg == 0) S0 = p.S0 + static_cast<size_t>(bh) * kD * kD;
        const bool ident = p.s0_mode == kS0Identity;
#pragma unroll
        for (int kk = 0; kk < 64; ++kk)
            s_reg[kk] = S0 ? S0[(64 * half + kk) * kD + row] : ((ident && 64 * half + kk == row) ? 1.f : 0.f);
    }

    // (c') W^T = K^T T_K^T and U^T = V^T T_V^T of chunk c, issued by the state group (which
    // waits for them next) so that the operand group moves on to chunk c+1 at once. Per-channel
    // gate: W_r^T = K_r^T T_V^T (the factor e^{G_r} of W is carried by the state operand).
    // (d) S^T -> bf16 operand; issue S^T W^T.
    auto st_issue1 = [&](int c) {
        load_gates(c + 2);   // warp 0: gates of chunk c+2, turned into vectors at the end of chunk c
        // W^T of chunk c -> bf16 MN-major B operand (rows k, 64 tokens per row), over the T area
        wait(bar_W, c & 1);
        tc_fence_after();
        // U^T of chunk c is computed: the v tile takes chunk c+1
        if (warp == 0) {
            if (!p.zero_v && c + 1 < nchunks && elect_one()) issue_v(c + 1);
            __syncwarp();
        }
        {
            uint32_t v[32];
            tmem_ld32(tlane + TM_W + 32 * half, v);
            tmem_ld_wait();
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                st_bf16x8u(sbase + OFF_WT + sw128_off(row, half * 64 + ch * 16), v + 8 * ch);
        }
        const uint32_t base = sbase + OFF_ST + half * 16384;
        if constexpr (kCh) {   // state operand S^T diag(e^{G_r}) (per key channel)
            const float *eGr = sm.ch[c % 3].eGr + 64 * half;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const float4 a = *reinterpret_cast<const float4 *>(eGr + 8 * ch);
                const float4 bq = *reinterpret_cast<const float4 *>(eGr + 8 * ch + 4);
                const float x[8] = {s_reg[8 * ch] * a.x,     s_reg[8 * ch + 1] * a.y, s_reg[8 * ch + 2] * a.z,
                                    s_reg[8 * ch + 3] * a.w, s_reg[8 * ch + 4] * bq.x, s_reg[8 * ch + 5] * bq.y,
                                    s_reg[8 * ch + 6] * bq.z, s_reg[8 * ch + 7] * bq.w};
                st_bf16x8(base + sw128_off(row, ch * 16), x);
            }
        } else {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) st_bf16x8(base + sw128_off(row, ch * 16), s_reg + 8 * ch);
        }
        fence_proxy_async_smem();
        if (gtid == 0) tma_store_wait_read_all();   // the previous output staging is free again
        gsync();
        if (gw == 0) {
            tc_fence_after();
            if (elect_one()) {
                const uint64_t dst = sw128_desc(sbase + OFF_ST, 16, 1024),
                               dwt = sw128_desc(sbase + OFF_WT, 16384, 1024);
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t aoff = (s >> 2) * 16384 + (s & 3) * 32;
                    mma_bf16(tbase + TM_1A, desc_add(dst, aoff), desc_add(dwt, s * 2048), id_1a, s);
                }
                mma_commit(bar_1);
            }
            __syncwarp();
        }
    };

    // (e) E^T = U^T - (W S)^T and E^T diag(e^{G_end-G}); release W^T and U^T; issue E^T_s K
    // and E^T A^T.
    auto st_issue2 = [&](int c) {
        const ChunkVec &cv = sm.v[c % 3];
        wait(bar_1, c & 1);
        tc_fence_after();
#pragma unroll
        for (int pc = 0; pc < 2; ++pc) {
            uint32_t u[16], w[16];
            tmem_ld16(tlane + TM_U + 32 * half + 16 * pc, u);
            tmem_ld16(tlane + TM_1A + 32 * half + 16 * pc, w);
            tmem_ld_wait();
            float e[16], es[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                e[jj] = (p.zero_v ? 0.f : __uint_as_float(u[jj])) - __uint_as_float(w[jj]);
                es[jj] = e[jj] * cv.eEnd[32 * half + 16 * pc + jj];
            }
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                const uint32_t off = sw128_off(row, half * 64 + pc * 32 + ch * 16);
                st_bf16x8(sbase + OFF_ET + off, e + 8 * ch);
                if (!kCh) st_bf16x8(sbase + OFF_ETS + off, es + 8 * ch);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        gsync();
        // warp 0 issues the product the state update waits for, warp 1 the output products, so
        // neither issue sequence waits behind the other
        if (gw == 0) {
            tc_fence_after();
            if (elect_one()) {
                mbar_arrive(bar_freed);   // W^T read by the finished S^T W^T, U^T loaded by every thread
                // scalar gate: (E^T diag(e^{G_end-G})) K; per-channel gate: E^T K_end (K_end over the
                // E^T_s area, 64-row blocks)
                const uint32_t a2 = sbase + (kCh ? OFF_ET : OFF_ETS);
                const uint32_t b2 = kCh ? ke_of(c) : qk_of(c), lbo2 = kCh ? 8192 : 16384;
                const uint64_t da2 = sw128_desc(a2, 16, 1024), db2 = sw128_desc(b2, lbo2, 1024);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tbase + TM_2, desc_add(da2, s * 32), desc_add(db2, s * 2048), id_2, s);
                mma_commit(bar_2);
                if (kCh) mma_commit(bar_m2k0 + 8 * (c & 1));   // the K_end buffer of chunk c is free
            }
            __syncwarp();
        } else if (gw == 1) {
            tc_fence_after();
            if (elect_one()) {
                if (write_out) {     // the output products: S^T Q^T and E^T A^T
                    const uint64_t dst = sw128_desc(sbase + OFF_ST, 16, 1024),
                                   dqq = sw128_desc(qk_of(c) + 8192, 16, 1024);
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                        mma_bf16(tbase + TM_1B, desc_add(dst, off), desc_add(dqq, off), id_qk, s);
                    }
                    const uint64_t det = sw128_desc(sbase + OFF_ET, 16, 1024), daq = sw128_desc(aqk_of(c), 16, 1024);
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_bf16(tbase + TM_3, desc_add(det, s * 32), desc_add(daq, s * 32), id_qk, s);
                }
                mma_commit(bar_o);
            }
            __syncwarp();
        }
    };

    // (f) S^T <- e^{G_end} S^T + (K_end^T E)^T; O^T = e^{G} (Q S)^T + (A E)^T -> TMA store;
    // retire chunk c and prefetch chunk c+2 into its stage.
    auto st_finish = [&](int c) {
        const ChunkVec &cv = sm.v[c % 3];
        if (warp == 0) {   // gate vectors of chunk c+2 into the buffer of chunk c-1 (retired)
            gate_vec(c + 2);
            __threadfence_block();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_done0 + 8 * (c & 1));
        }
        wait(bar_2, c & 1);
        tc_fence_after();
        {
            const float gam = cv.eG[kC - 1];
            const float *gch = sm.ch[c % 3].gam + 64 * half;
            // 32 columns per wait; 16 with the per-channel gate, whose decay vector needs the registers
            constexpr int kW = kCh ? 16 : 32;
#pragma unroll
            for (int hh = 0; hh < 64 / kW; ++hh) {
                uint32_t v[kW];
                if constexpr (kW == 32) tmem_ld32(tlane + TM_2 + 64 * half + 32 * hh, v);
                else tmem_ld16(tlane + TM_2 + 64 * half + 16 * hh, v);
                tmem_ld_wait();
#pragma unroll
                for (int kk = 0; kk < kW; ++kk) {
                    const float gk = kCh ? gch[kW * hh + kk] : gam;
                    s_reg[kW * hh + kk] = fmaf(gk, s_reg[kW * hh + kk], __uint_as_float(v[kk]));
                }
            }
        }
        wait(bar_o, c & 1);
        tc_fence_after();
        // Q and K of chunk c have been read by the finished products: refill the stage with chunk c+2
        if (warp == 0) {
            if (c + 2 < nchunks && elect_one()) issue_loads(c + 2);
            __syncwarp();
        }
        if (write_out) {
            // Pair value channels (m, m^1) so each lane stores two channels as one bf16x2:
            // within each group of 16 tokens, even lanes keep tokens 0-7, odd lanes 8-15.
            const bool odd = lane & 1;
            const int m0 = row & ~1;
            uint8_t *stg = smem + (kCh ? OFF_ET : OFF_ETS) + (m0 >> 6) * 8192 + (m0 & 63) * 2;
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
                uint32_t qs[16], ae[16];
                tmem_ld16(tlane + TM_1B + 32 * half + 16 * pc, qs);
                tmem_ld16(tlane + TM_3 + 32 * half + 16 * pc, ae);
                tmem_ld_wait();
                float o[16];   // s (e^G Q S + A E)
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    o[jj] = p.q_scale * fmaf(kCh ? 1.f : cv.eG[32 * half + 16 * pc + jj], __uint_as_float(qs[jj]),
                                             __uint_as_float(ae[jj]));
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const float mine = odd ? o[jj + 8] : o[jj];
                    const float send = odd ? o[jj] : o[jj + 8];
                    const float other = __shfl_xor_sync(0xffffffffu, send, 1);
                    const int n = 32 * half + 16 * pc + jj + (odd ? 8 : 0);
                    const uint32_t pr = odd ? pack_bf16(other, mine) : pack_bf16(mine, other);
                    *reinterpret_cast<uint32_t *>(stg + n * 128) = pr;
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        gsync();
        if (gtid == 0) {
            const int t0 = t_begin + c * kC;
            const uint32_t stg0 = sbase + (kCh ? OFF_ET : OFF_ETS);
            if (write_out) {
                tma_store_4d(&tm_o, stg0, 0, h, t0, b);
                tma_store_4d(&tm_o, stg0 + 8192, 64, h, t0, b);
                tma_store_commit();
            }
        }
    };

    // ================================================================== schedule
    if (grp == 1) {
        load_chgates(0);
        for (int c = 0; c < nchunks; ++c) {
            if (group_aborted()) break;
            op_front(c);
            op_mid(c);
        }
    } else {
        for (int c = 0; c < nchunks; ++c) {
            wait(bar_ready, c & 1);
            if (group_aborted()) break;
            tc_fence_after();
            st_issue1(c);
            st_issue2(c);
            st_finish(c);
        }
    }
    __syncthreads();

    if (sm.abort && tid == 0) atomicOr(p.err, kErrTimeout);
    if (tid == 0) tma_store_wait_all();
    float *ST = nullptr;
    if (p.S_T && p.st_mode == kSTSegment) ST = p.S_T + (static_cast<size_t>(bh) * p.nseg + seg) * kD * kD;
    else if (p.S_T && seg == p.nseg - 1) ST = p.S_T + static_cast<size_t>(bh) * kD * kD;
    if (grp == 0 && ST && !sm.abort) {
#pragma unroll
        for (int kk = 0; kk < 64; ++kk) ST[(64 * half + kk) * kD + row] = s_reg[kk];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// Per-channel gate: marks the (sequence, head) chains with a chunk whose gates, for some key
// channel, multiply to less than e^-78 over tokens 0-31 or 32-63 of the chunk (a margin inside
// the e^-80 limit of the factorised in-chunk products, with the same per-token clamp and tokens
// past the end counted as 1). One CTA of 128 threads (one per key channel) per (chunk, head,
// sequence); coalesced reads of 128 consecutive gates per token.
__global__ void __launch_bounds__(kD) gate_range_kernel(const float *alpha, int T, int H, unsigned *marks) {
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, k = threadIdx.x;
    const float kLow = 1.3e-34f;   // ~ e^-78
    bool low = false;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float prod = 1.f;
        const int t0 = c * kC + 32 * half, t1 = min(T, t0 + 32);
        for (int t = t0; t < t1; ++t)
            prod *= fmaxf(alpha[((static_cast<size_t>(b) * T + t) * H + h) * kD + k], 1.8e-35f);
        low |= prod < kLow;
    }
    if (__syncthreads_or(low) && k == 0) marks[static_cast<size_t>(b) * H + h] = 1u;
}

// ---------------------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// [B, T, H, 128] bf16 tensor (sequences Ts >= T tokens apart: a T-token slice of longer ones);
// box = 64 channels x 64 tokens of one (b, h).
bool make_map(CUtensorMap *m, const void *base, int B, int T, int H, bool swizzle, int Ts) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(H) * kD * 2,
                                   static_cast<cuuint64_t>(Ts) * H * kD * 2};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kC), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Number of segments a chain of `nchunks` chunks is split into, chosen to minimise the
// wall time in chunk-steps when each CTA occupies one SM: pass 1 runs the value run of
// segments 0..n-2 and the transition run of segments 1..n-2, pass 3 reruns segments 1..n-1.
int plan_segments(int B, int T, int H) {
    const int chains = B * H, nchunks = (T + kC - 1) / kC;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0)
        return 1;
    auto waves = [&](long ctas) { return (ctas + sms - 1) / sms; };
    const double base = static_cast<double>(waves(chains)) * nchunks;
    double best = 0.8 * base;   // only split when it saves a fifth or more
    int best_n = 1;
    for (int n = 2; n <= 64; ++n) {
        const int L = (nchunks + n - 1) / n;   // chunks per segment
        if (L < 8) break;
        const int nn = (nchunks + L - 1) / L;
        if (nn < 2) continue;
        const double cost = static_cast<double>(waves(static_cast<long>(chains) * ((nn - 1) + (nn - 2))) +
                                                waves(static_cast<long>(chains) * (nn - 1))) * L;
        if (cost < best) {
            best = cost;
            best_n = n;
        }
    }
    return best_n;
}

struct SegPlan {
    int nseg, seg_len;   // seg_len in tokens, a multiple of the chunk
};

// When the CTAs of pass 1a and pass 1b of the segment scan fit on the SMs together (the plan
// above then counts them as one wave), pass 1b runs on a second stream, concurrently with pass
// 1a (measured on B = 1, H = 16, T = 4096: 0.268 -> 0.208 ms); when they need two waves anyway,
// both stay on the caller's stream, which measured 2-4 % faster than interleaving them. One
// stream and two events per device, created on first use; the mutex keeps a call's fork and join
// records from interleaving with another thread's.
struct AuxStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxAuxDevices = 64;
AuxStream g_aux[kMaxAuxDevices];
std::mutex g_aux_mutex[kMaxAuxDevices];
SegPlan make_plan(int B, int T, int H) {
    const int n = plan_segments(B, T, H);
    if (n <= 1) return {1, ((T + kC - 1) / kC) * kC};
    const int nchunks = (T + kC - 1) / kC, L = (nchunks + n - 1) / n;
    return {(nchunks + L - 1) / L, L * kC};
}

// Segment states (Z, M and the start states, each [chains][nseg][d][d] fp32) when the sequence is
// split; then, with the per-channel gate, one flag per chain (256-byte aligned).
size_t seg_workspace_bytes(int B, int T, int H) {
    const SegPlan pl = make_plan(B, T, H);
    if (pl.nseg <= 1) return 0;
    return 3ull * B * H * pl.nseg * kD * kD * sizeof(float);
}
size_t rescue_flag_bytes(int B, int H) { return (static_cast<size_t>(B) * H * sizeof(unsigned) + 255) & ~size_t(255); }

// Per-channel gate: rerun, on the exact fp32 recurrence, the chains gate_range_kernel marked (the
// tensor-core kernel skipped them); every other CTA of the launch returns at once.
cudaError_t launch_rescue(const ChunkArgs &a, const unsigned *flags) {
    ChunkArgs r = a;
    r.only = flags;
    return launch_recurrent(r);
}

}  // namespace

cudaError_t launch_gate_range(const float *alpha, int B, int T, int H, unsigned *marks, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(marks, 0, static_cast<size_t>(B) * H * sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
    if (T < 1) return cudaSuccess;
    gate_range_kernel<<<dim3((T + kC - 1) / kC, H, B), kD, 0, stream>>>(alpha, T, H, marks);
    return cudaGetLastError();
}

size_t chunk_tc_workspace_bytes(int B, int T, int H, kla_gate gate) {
    return seg_workspace_bytes(B, T, H) + (gate == KLA_GATE_CHANNEL ? rescue_flag_bytes(B, H) : 0);
}

bool chunk_tc_supports(const ChunkArgs &a) {
    return a.dtype == KLA_DTYPE_BF16 && a.d_k == kD && a.d_v == kD && a.chunk == kC && a.T > 0;
}

cudaError_t launch_chunk_tc(const ChunkArgs &a) {
    CUtensorMap mq, mk, mv, mo;
    const int Ts = a.T_stride > 0 ? a.T_stride : a.T;
    // a slice of longer sequences: scalar gate, one segment (the range check, the rerun and the
    // segment plan index whole sequences)
    if (Ts != a.T && (Ts < a.T || a.gate != KLA_GATE_SCALAR || !a.no_segments)) return cudaErrorInvalidValue;
    if (!make_map(&mq, a.q, a.B, a.T, a.H, true, Ts) || !make_map(&mk, a.k, a.B, a.T, a.H, true, Ts) ||
        !make_map(&mv, a.v, a.B, a.T, a.H, true, Ts) || !make_map(&mo, a.o, a.B, a.T, a.H, false, Ts))
        return cudaErrorInvalidValue;
    auto kern = a.gate == KLA_GATE_CHANNEL ? chunk_tc_kernel<true> : chunk_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    const int chains = a.B * a.H;
    const SegPlan pl = a.no_segments ? SegPlan{1, ((a.T + kC - 1) / kC) * kC} : make_plan(a.B, a.T, a.H);
    const size_t seg_bytes = pl.nseg <= 1 ? 0 : seg_workspace_bytes(a.B, a.T, a.H);
    // Per-channel gate with a workspace: chains whose gates leave the range of the factorised
    // products are marked first (marks after the segment states), skipped by the tensor-core
    // launches and rerun exactly after them. Without a workspace they are only reported.
    unsigned *flags = nullptr;
    if (a.gate == KLA_GATE_CHANNEL && a.workspace && a.workspace_bytes >= seg_bytes + rescue_flag_bytes(a.B, a.H)) {
        flags = reinterpret_cast<unsigned *>(static_cast<char *>(a.workspace) + seg_bytes);
        if ((e = launch_gate_range(a.alpha, a.B, a.T, a.H, flags, a.stream)) != cudaSuccess) return e;
    }
    TcParams p{a.alpha, a.eta, a.eps, a.S0, a.S_T, a.B, a.T, a.H, pl.seg_len, 0, 1, pl.nseg,
               kS0Chain, kSTLast, 0, 0, a.err, a.beta_raw, a.q_scale, flags, Ts};
    if (pl.nseg <= 1) {
        kern<<<chains, kThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, mo, p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        return flags ? launch_rescue(a, flags) : cudaSuccess;
    }
    // Sequence-parallel scan over segments (workspace: Z | M | start states, each
    // [chains][nseg][d][d] fp32).
    if (!a.workspace || a.workspace_bytes < seg_bytes) return cudaErrorInvalidValue;
    const size_t part = static_cast<size_t>(chains) * pl.nseg * kD * kD;
    float *Z = static_cast<float *>(a.workspace), *M = Z + part, *Sst = M + part;
    // pass 1a: segments 0..n-2 from the true start (segment 0) or zero; segment 0 writes its outputs
    TcParams p1 = p;
    p1.seg_begin = 0;
    p1.seg_count = pl.nseg - 1;
    p1.S_T = Z;
    p1.st_mode = kSTSegment;
    p1.no_out = 2;
    // pass 1b: transitions of segments 1..n-2 (start from I, v = 0, no outputs)
    TcParams p2 = p;
    p2.seg_begin = 1;
    p2.seg_count = pl.nseg - 2;
    p2.S0 = nullptr;
    p2.s0_mode = kS0Identity;
    p2.S_T = M;
    p2.st_mode = kSTSegment;
    p2.zero_v = 1;
    p2.no_out = 1;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const bool one_wave = static_cast<long>(chains) * (p1.seg_count + p2.seg_count) <= sms;
    if (pl.nseg <= 2 || !one_wave) {
        kern<<<chains * p1.seg_count, kThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, mo, p1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (pl.nseg > 2) {
            kern<<<chains * p2.seg_count, kThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, mo, p2);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    } else {   // pass 1b on the auxiliary stream, between a fork and a join on the caller's stream
        if (dev < 0 || dev >= kMaxAuxDevices) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(g_aux_mutex[dev]);
        AuxStream &ax = g_aux[dev];
        if (!ax.s) {
            if ((e = cudaStreamCreateWithFlags(&ax.s, cudaStreamNonBlocking)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&ax.fork, cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&ax.join, cudaEventDisableTiming)) != cudaSuccess)
                return e;
        }
        if ((e = cudaEventRecord(ax.fork, a.stream)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(ax.s, ax.fork, 0)) != cudaSuccess)
            return e;
        kern<<<chains * p1.seg_count, kThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, mo, p1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        kern<<<chains * p2.seg_count, kThreads, SMEM_BYTES, ax.s>>>(mq, mk, mv, mo, p2);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = cudaEventRecord(ax.join, ax.s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(a.stream, ax.join, 0)) != cudaSuccess)
            return e;
    }
    // pass 2: start states of segments 1..n-1
    if ((e = launch_seg_combine(Z, M, Sst, chains, pl.nseg, a.stream)) != cudaSuccess) return e;
    // pass 3: segments 1..n-1 from their true start states; the last one writes S_T
    TcParams p3 = p;
    p3.seg_begin = 1;
    p3.seg_count = pl.nseg - 1;
    p3.S0 = Sst;
    p3.s0_mode = kS0Segment;
    kern<<<chains * p3.seg_count, kThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, mo, p3);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return flags ? launch_rescue(a, flags) : cudaSuccess;
}

}  // namespace kla
