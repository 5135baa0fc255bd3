// kla_chunk_tc.cu -- tensor-core (tcgen05) chunkwise KLA prefill for sm_103a.
//
// Scope: bf16 q/k/v/o, d_k = d_v = 128, chunk C = 64, scalar gate, fp32 state.
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
// One CTA per (sequence, head) walks its chunks in order; it is one SM's worth of work and the
// grid is B*H CTAs. Every product runs on the 5th-generation tensor cores in the transposed
// orientation that puts 128 rows (d_k or d_v) on the TMEM lanes:
//   [K;Q] K^T            -> TMEM  (KK^T | QK^T)           M=128 N=64  K=128
//   K^T (T diag(beta e^G))^T, V^T (T diag(beta))^T -> W^T, U^T        M=128 N=64  K=64
//   S^T W^T, S^T Q^T     -> (W S)^T, (Q S)^T              M=128 N=64  K=128
//   E^T_s K              -> (K_end^T E)^T                  M=128 N=128 K=64
//   E^T A^T              -> (A E)^T                        M=128 N=64  K=64
// Operands are bf16 in 128-byte-swizzled shared memory (q/k/v tiles arrive by TMA, derived
// tiles are written by the threads), accumulators are fp32 in tensor memory. The 64 x 64
// unit-triangular inverse is computed in fp32 on the CUDA cores (16 x 16 diagonal blocks by
// substitution, then block forward substitution). The state S^T lives in registers in fp32
// (thread = one value channel, 64 key channels), and is re-rounded to bf16 only as an MMA
// operand, never as the carried state.
#include <cuda.h>

#include <algorithm>

#include "kla_internal.cuh"
#include "sm103_ptx.cuh"

namespace kla {
namespace {

using namespace ptx;

constexpr int kC = 64;          // chunk
constexpr int kD = 128;         // d_k = d_v
constexpr int kThreads = 256;
constexpr float kMinLogGate = -80.0f;
constexpr uint32_t kWaitLimit = 1u << 24;

// ---- shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_QK = 0;                       // 2 stages x 32 KB: [blk0: K rows 0-63 | Q rows 0-63][blk1 ...]
constexpr uint32_t QK_STAGE = 32768;
constexpr uint32_t OFF_V = OFF_QK + 2 * QK_STAGE;    // 2 stages x 16 KB: [blk0: 64 rows][blk1: 64 rows]
constexpr uint32_t V_STAGE = 16384;
constexpr uint32_t OFF_AQK = OFF_V + 2 * V_STAGE;    // 8 KB: A (query rows) bf16, K-major
constexpr uint32_t OFF_X = OFF_AQK + 8192;           // 17 KB: R fp32 [64][65], then T_K | T_V bf16 tiles
constexpr uint32_t OFF_Y = OFF_X + 17408;            // 17 KB: T fp32 [64][65], then W^T bf16 tile
constexpr uint32_t OFF_ST = OFF_Y + 17408;           // 32 KB: S^T bf16, K-major, 2 blocks of 128 rows
constexpr uint32_t OFF_ET = OFF_ST + 32768;          // 16 KB: E^T bf16 (also fp32 scratch of the solve)
constexpr uint32_t OFF_ETS = OFF_ET + 16384;         // 16 KB: E^T diag(e^{G_end-G}) bf16, then O staging
constexpr uint32_t OFF_SMALL = OFF_ETS + 16384;      // small vectors + barriers
constexpr uint32_t SMEM_BYTES = OFF_SMALL + 2048 + 1024;   // + alignment slack

// ---- tensor memory columns (512 allocated)
constexpr uint32_t TM_A = 0;      // [KK^T ; QK^T]     64 cols
constexpr uint32_t TM_W = 64;     // W^T               64
constexpr uint32_t TM_U = 128;    // U^T               64
constexpr uint32_t TM_1A = 192;   // (W S)^T           64
constexpr uint32_t TM_1B = 256;   // (Q S)^T           64
constexpr uint32_t TM_3 = 320;    // (A E)^T           64
constexpr uint32_t TM_2 = 384;    // (K_end^T E)^T     128

constexpr uint32_t kTileBytes = 4 * 8192 + 2 * 8192;   // q, k, v chunk tiles per stage

struct Small {
    float G[kC];
    float beta[kC];
    float expG[kC];
    float expEnd[kC];
    float eta[kC];
    uint64_t full[2];
    uint64_t mA, mW, m1, m2;
    uint32_t tmem_base;
    volatile int abort;
};
static_assert(sizeof(Small) <= 2048, "small area");

struct TcParams {
    const float *alpha, *eta;
    float eps;
    const float *S0;
    float *S_T;
    int B, T, H;
    unsigned *err;
};

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    Small &sm = *reinterpret_cast<Small *>(smem + OFF_SMALL);
    float *Rm = reinterpret_cast<float *>(smem + OFF_X);    // [64][65]
    float *Tm = reinterpret_cast<float *>(smem + OFF_Y);    // [64][65]
    float *Xs = reinterpret_cast<float *>(smem + OFF_ET);   // solve scratch [3][16][16]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;        // TMEM lane of this thread
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int nchunks = (p.T + kC - 1) / kC;

    const uint32_t bar_full0 = smem_u32(&sm.full[0]);
    const uint32_t bar_A = smem_u32(&sm.mA), bar_W = smem_u32(&sm.mW);
    const uint32_t bar_1 = smem_u32(&sm.m1), bar_2 = smem_u32(&sm.m2);

    if (tid == 0) {
        mbar_init(bar_full0, 1);
        mbar_init(bar_full0 + 8, 1);
        mbar_init(bar_A, 1);
        mbar_init(bar_W, 1);
        mbar_init(bar_1, 1);
        mbar_init(bar_2, 1);
        sm.abort = 0;
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
    const uint32_t tlane = tbase + (static_cast<uint32_t>(quarter * 32) << 16);

    auto issue_loads = [&](int c) {   // thread 0 only
        const int st = c & 1;
        const uint32_t bar = bar_full0 + 8 * st;
        const uint32_t qk = sbase + OFF_QK + st * QK_STAGE;
        const uint32_t vv = sbase + OFF_V + st * V_STAGE;
        mbar_arrive_expect_tx(bar, kTileBytes);
        const int t0 = c * kC;
        tma_load_4d(qk + 0, &tm_k, bar, 0, h, t0, b);
        tma_load_4d(qk + 8192, &tm_q, bar, 0, h, t0, b);
        tma_load_4d(qk + 16384, &tm_k, bar, 64, h, t0, b);
        tma_load_4d(qk + 24576, &tm_q, bar, 64, h, t0, b);
        tma_load_4d(vv + 0, &tm_v, bar, 0, h, t0, b);
        tma_load_4d(vv + 8192, &tm_v, bar, 64, h, t0, b);
    };
    if (tid == 0) {
        issue_loads(0);
        if (nchunks > 1) issue_loads(1);
    }

    // State S^T: this thread owns value channel m = row, key channels [64*half, 64*half + 64).
    float s_reg[64];
    {
        const int m = row;
        const float *S0 = p.S0 ? p.S0 + static_cast<size_t>(bh) * kD * kD : nullptr;
#pragma unroll
        for (int kk = 0; kk < 64; ++kk) s_reg[kk] = S0 ? S0[(64 * half + kk) * kD + m] : 0.f;
    }

    // Gates of the next chunk, prefetched by warp 0 (two tokens per lane).
    float a_nx[2] = {1.f, 1.f}, e_nx[2] = {0.f, 0.f};
    auto load_gates = [&](int c) {
        if (warp == 0 && c < nchunks) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = c * kC + 2 * lane + u;
                const bool ok = t < p.T;
                const size_t tok = (static_cast<size_t>(b) * p.T + t) * p.H + h;
                a_nx[u] = ok ? p.alpha[tok] : 1.f;
                e_nx[u] = ok ? p.eta[tok] : 0.f;
            }
        }
    };
    load_gates(0);

    const uint32_t id_qk = idesc_bf16(128, 64, 0, 0);     // K-major x K-major, N=64
    const uint32_t id_w = idesc_bf16(128, 64, 1, 0);      // MN-major A, K-major B
    const uint32_t id_1a = idesc_bf16(128, 64, 0, 1);     // K-major A, MN-major B
    const uint32_t id_2 = idesc_bf16(128, 128, 0, 1);     // N=128, MN-major B

    for (int c = 0; c < nchunks; ++c) {
        const int st = c & 1;
        const uint32_t ph = c & 1;
        const uint32_t qk = sbase + OFF_QK + st * QK_STAGE;
        const uint32_t vv = sbase + OFF_V + st * V_STAGE;

        // ---- (1) gates: log-decay prefix, eta; prefetch the next chunk's gates
        if (warp == 0) {
            const float g0 = fmaxf(__logf(a_nx[0]), kMinLogGate), g1 = fmaxf(__logf(a_nx[1]), kMinLogGate);
            const float e0 = e_nx[0], e1 = e_nx[1];
            float s = g0 + g1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += y;
            }
            sm.G[2 * lane + 1] = s;
            sm.G[2 * lane] = s - g1;
            sm.eta[2 * lane] = e0;
            sm.eta[2 * lane + 1] = e1;
        }
        load_gates(c + 1);
        if (tid == 0) tma_store_wait_read_all();   // previous chunk's O staging is free again

        // ---- (2) S^T as a bf16 K-major operand (block = half, row = m)
        {
            const uint32_t base = sbase + OFF_ST + half * 16384;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                st_shared_v4(base + sw128_off(row, ch * 16), pack_bf16(s_reg[8 * ch + 0], s_reg[8 * ch + 1]),
                             pack_bf16(s_reg[8 * ch + 2], s_reg[8 * ch + 3]),
                             pack_bf16(s_reg[8 * ch + 4], s_reg[8 * ch + 5]),
                             pack_bf16(s_reg[8 * ch + 6], s_reg[8 * ch + 7]));
            }
        }

        // ---- wait for this chunk's q/k/v tiles
        if (!mbar_wait_bounded(bar_full0 + 8 * st, (c >> 1) & 1, kWaitLimit)) sm.abort = 1;

        // ---- (3) ||k_i||^2: 4 threads per key row, 32 channels each
        float n2 = 0.f;
        {
            const int i = tid >> 2, part = tid & 3;
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
        __syncthreads();   // #1: G, eta visible
        if (sm.abort) break;
        if ((tid & 3) == 0) {
            const int i = tid >> 2;
            const float G = sm.G[i];
            sm.beta[i] = kla_beta(sm.eta[i], n2, p.eps);
            sm.expG[i] = __expf(G);
            sm.expEnd[i] = __expf(sm.G[kC - 1] - G);
        }
        fence_proxy_async_smem();   // S^T tile -> tensor core
        __syncthreads();            // #2

        // ---- (4) [K;Q] K^T and S^T Q^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                mma_bf16(tbase + TM_A, sw128_desc(qk + off, 16, 1024), sw128_desc(qk + off, 16, 1024), id_qk, s);
            }
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                mma_bf16(tbase + TM_1B, sw128_desc(sbase + OFF_ST + off, 16, 1024),
                         sw128_desc(qk + 8192 + off, 16, 1024), id_qk, s);
            }
            mma_commit(bar_A);
        }
        if (!mbar_wait_bounded(bar_A, ph, kWaitLimit)) sm.abort = 1;
        tc_fence_after();

        // ---- (5) R (key rows) and A (query rows)
        {
            uint32_t v[32];
            tmem_ld32(tlane + TM_A + 32 * half, v);
            tmem_ld_wait();
            if (row < kC) {
                const int i = row;
                const float Gi = sm.G[i], bi = sm.beta[i];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = 32 * half + jj;
                    const float r = (j < i) ? bi * __expf(Gi - sm.G[j]) * __uint_as_float(v[jj]) : 0.f;
                    Rm[i * 65 + j] = r;
                }
            } else {
                const int i = row - kC;
                const float Gi = sm.G[i];
                float a[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = 32 * half + jj;
                    a[jj] = (j <= i) ? __expf(Gi - sm.G[j]) * __uint_as_float(v[jj]) : 0.f;
                }
                const uint32_t base = sbase + OFF_AQK;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    st_shared_v4(base + sw128_off(i, half * 64 + ch * 16), pack_bf16(a[8 * ch], a[8 * ch + 1]),
                                 pack_bf16(a[8 * ch + 2], a[8 * ch + 3]), pack_bf16(a[8 * ch + 4], a[8 * ch + 5]),
                                 pack_bf16(a[8 * ch + 6], a[8 * ch + 7]));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();   // #3
        if (sm.abort) break;

        // ---- (6) T = (I + R)^{-1}, fp32. Diagonal 16x16 blocks by substitution (warps 0-3).
        if (warp < 4 && lane < 16) {
            const int o = 16 * warp;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float acc = (i == lane) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < i; ++j) acc = fmaf(-Rm[(o + i) * 65 + o + j], x[j], acc);
                x[i] = acc;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Tm[(o + i) * 65 + o + lane] = x[i];
        }
        __syncthreads();
        // Off-diagonal blocks, by distance d from the diagonal:
        //   X_ba = sum_{x=a}^{b-1} R_bx T_xa ;  T_ba = -T_bb X_ba
#pragma unroll 1
        for (int d = 1; d < 4; ++d) {
            const int nblk = 4 - d;
            for (int idx = tid; idx < nblk * 256; idx += kThreads) {
                const int blk = idx >> 8, i = (idx >> 4) & 15, j = idx & 15;
                const int bb = blk + d, aa = blk;
                float acc = 0.f;
                for (int x = aa; x < bb; ++x)
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        acc = fmaf(Rm[(16 * bb + i) * 65 + 16 * x + u], Tm[(16 * x + u) * 65 + 16 * aa + j], acc);
                Xs[idx] = acc;
            }
            __syncthreads();
            for (int idx = tid; idx < nblk * 256; idx += kThreads) {
                const int blk = idx >> 8, i = (idx >> 4) & 15, j = idx & 15;
                const int bb = blk + d, aa = blk;
                float acc = 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    if (u <= i) acc = fmaf(Tm[(16 * bb + i) * 65 + 16 * bb + u], Xs[(blk << 8) + (u << 4) + j], acc);
                Tm[(16 * bb + i) * 65 + 16 * aa + j] = -acc;
            }
            __syncthreads();
        }

        // ---- (7) T_K = T diag(beta e^G), T_V = T diag(beta): bf16 K-major (rows n, k contiguous)
        {
            const int n = tid >> 2, kq = tid & 3;
            float tk[16], tv[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int k = 16 * kq + u;
                const float t = (k <= n) ? Tm[n * 65 + k] : 0.f;
                tv[u] = t * sm.beta[k];
                tk[u] = tv[u] * sm.expG[k];
            }
            const uint32_t bk = sbase + OFF_X, bv = sbase + OFF_X + 8192;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const uint32_t off = sw128_off(n, 32 * kq + 16 * hh);
                const float *a = tk + 8 * hh, *e = tv + 8 * hh;
                st_shared_v4(bk + off, pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]),
                             pack_bf16(a[6], a[7]));
                st_shared_v4(bv + off, pack_bf16(e[0], e[1]), pack_bf16(e[2], e[3]), pack_bf16(e[4], e[5]),
                             pack_bf16(e[6], e[7]));
            }
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- (8) W^T = K^T T_K^T, U^T = V^T T_V^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                mma_bf16(tbase + TM_W, sw128_desc(qk + s * 2048, 16384, 1024),
                         sw128_desc(sbase + OFF_X + s * 32, 16, 1024), id_w, s);
            }
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                mma_bf16(tbase + TM_U, sw128_desc(vv + s * 2048, 8192, 1024),
                         sw128_desc(sbase + OFF_X + 8192 + s * 32, 16, 1024), id_w, s);
            }
            mma_commit(bar_W);
        }
        if (!mbar_wait_bounded(bar_W, ph, kWaitLimit)) sm.abort = 1;
        tc_fence_after();

        // ---- (9) W^T -> bf16, MN-major B operand (rows k, 64 tokens per row)
        {
            uint32_t v[32];
            tmem_ld32(tlane + TM_W + 32 * half, v);
            tmem_ld_wait();
            const uint32_t base = sbase + OFF_Y;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                st_shared_v4(base + sw128_off(row, half * 64 + ch * 16),
                             pack_bf16(__uint_as_float(v[8 * ch]), __uint_as_float(v[8 * ch + 1])),
                             pack_bf16(__uint_as_float(v[8 * ch + 2]), __uint_as_float(v[8 * ch + 3])),
                             pack_bf16(__uint_as_float(v[8 * ch + 4]), __uint_as_float(v[8 * ch + 5])),
                             pack_bf16(__uint_as_float(v[8 * ch + 6]), __uint_as_float(v[8 * ch + 7])));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (sm.abort) break;

        // ---- (10) (W S)^T = S^T W^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t aoff = (s >> 2) * 16384 + (s & 3) * 32;
                mma_bf16(tbase + TM_1A, sw128_desc(sbase + OFF_ST + aoff, 16, 1024),
                         sw128_desc(sbase + OFF_Y + s * 2048, 16384, 1024), id_1a, s);
            }
            mma_commit(bar_1);
        }
        if (!mbar_wait_bounded(bar_1, ph, kWaitLimit)) sm.abort = 1;
        tc_fence_after();

        // ---- (11) E^T = U^T - (W S)^T, and E^T diag(e^{G_end - G})
        {
            uint32_t u[32], w[32];
            tmem_ld32(tlane + TM_U + 32 * half, u);
            tmem_ld32(tlane + TM_1A + 32 * half, w);
            tmem_ld_wait();
            float e[32], es[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                e[jj] = __uint_as_float(u[jj]) - __uint_as_float(w[jj]);
                es[jj] = e[jj] * sm.expEnd[32 * half + jj];
            }
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const uint32_t off = sw128_off(row, half * 64 + ch * 16);
                st_shared_v4(sbase + OFF_ET + off, pack_bf16(e[8 * ch], e[8 * ch + 1]),
                             pack_bf16(e[8 * ch + 2], e[8 * ch + 3]), pack_bf16(e[8 * ch + 4], e[8 * ch + 5]),
                             pack_bf16(e[8 * ch + 6], e[8 * ch + 7]));
                st_shared_v4(sbase + OFF_ETS + off, pack_bf16(es[8 * ch], es[8 * ch + 1]),
                             pack_bf16(es[8 * ch + 2], es[8 * ch + 3]), pack_bf16(es[8 * ch + 4], es[8 * ch + 5]),
                             pack_bf16(es[8 * ch + 6], es[8 * ch + 7]));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (sm.abort) break;

        // ---- (12) (K_end^T E)^T = E^T_s K  and  (A E)^T = E^T A^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tbase + TM_2, sw128_desc(sbase + OFF_ETS + s * 32, 16, 1024),
                         sw128_desc(qk + s * 2048, 16384, 1024), id_2, s);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tbase + TM_3, sw128_desc(sbase + OFF_ET + s * 32, 16, 1024),
                         sw128_desc(sbase + OFF_AQK + s * 32, 16, 1024), id_qk, s);
            mma_commit(bar_2);
        }
        if (!mbar_wait_bounded(bar_2, ph, kWaitLimit)) sm.abort = 1;
        tc_fence_after();

        // ---- (13) S^T <- e^{G_end} S^T + (K_end^T E)^T   (fp32, registers)
        {
            const float gam = sm.expG[kC - 1];
            uint32_t v[32];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                tmem_ld32(tlane + TM_2 + 64 * half + 32 * hh, v);
                tmem_ld_wait();
#pragma unroll
                for (int kk = 0; kk < 32; ++kk)
                    s_reg[32 * hh + kk] = fmaf(gam, s_reg[32 * hh + kk], __uint_as_float(v[kk]));
            }
        }
        // ---- (14) O^T = diag-scaled (Q S)^T + (A E)^T -> staging [blk][token][64 ch] for TMA store
        {
            uint32_t qs[32], ae[32];
            tmem_ld32(tlane + TM_1B + 32 * half, qs);
            tmem_ld32(tlane + TM_3 + 32 * half, ae);
            tmem_ld_wait();
            const int m = row;
            uint8_t *stg = smem + OFF_ETS + (m >> 6) * 8192 + (m & 63) * 2;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int n = 32 * half + jj;
                const float o = fmaf(sm.expG[n], __uint_as_float(qs[jj]), __uint_as_float(ae[jj]));
                *reinterpret_cast<__nv_bfloat16 *>(stg + n * 128) = __float2bfloat16_rn(o);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            const int t0 = c * kC;
            tma_store_4d(&tm_o, sbase + OFF_ETS, 0, h, t0, b);
            tma_store_4d(&tm_o, sbase + OFF_ETS + 8192, 64, h, t0, b);
            tma_store_commit();
            if (c + 2 < nchunks) issue_loads(c + 2);
        }
    }

    if (sm.abort && tid == 0) atomicOr(p.err, kErrTimeout);
    if (tid == 0) tma_store_wait_all();
    if (p.S_T && !sm.abort) {
        float *ST = p.S_T + static_cast<size_t>(bh) * kD * kD;
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

// [B, T, H, 128] bf16 tensor; box = 64 channels x 64 tokens of one (b, h).
bool make_map(CUtensorMap *m, const void *base, int B, int T, int H, bool swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(H) * kD * 2,
                                   static_cast<cuuint64_t>(T) * H * kD * 2};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kC), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_supports(const ChunkArgs &a) {
    return a.dtype == KLA_DTYPE_BF16 && a.d_k == kD && a.d_v == kD && a.chunk == kC && a.gate == KLA_GATE_SCALAR &&
           a.T > 0;
}

cudaError_t launch_chunk_tc(const ChunkArgs &a) {
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, a.q, a.B, a.T, a.H, true) || !make_map(&mk, a.k, a.B, a.T, a.H, true) ||
        !make_map(&mv, a.v, a.B, a.T, a.H, true) || !make_map(&mo, a.o, a.B, a.T, a.H, false))
        return cudaErrorInvalidValue;
    TcParams p{a.alpha, a.eta, a.eps, a.S0, a.S_T, a.B, a.T, a.H, a.err};
    cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    chunk_tc_kernel<<<a.B * a.H, kThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, mo, p);
    return cudaGetLastError();
}

}  // namespace kla
