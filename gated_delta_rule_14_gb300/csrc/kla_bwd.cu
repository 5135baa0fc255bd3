// kla_bwd.cu -- backward pass of the KLA recurrence (reverse-mode derivative), fp32.
//
// The pages give no backward algebra (GeekNews, "Revisando las variantes de atencion lineal de la
// familia DeltaNet", section "KDA por chunks", names training as the use of the chunk mode); this
// is the chain rule through the forward steps in reverse order. With G = dL/dS_t carried from the
// last token down to the first, per token t (state S_{t-1} entering it, S~ = alpha (.) S_{t-1},
// residual e = v - S~^T k, step beta, read o = S_t^T (s q)):
//   read:     dq = s S_t do = s (S~ do + beta k (e . do));      G += s q do^T
//   write:    gk = G^T k;  de = beta gk;  dbeta = gk . e;       dk = beta G e
//   residual: dv = de;  dS~ = G - k de^T;                       dk -= S~ de
//   step:     KLA: deta = dbeta / (n + eps), dk -= 2 beta dbeta / (n + eps) k  (n = ||k||^2;
//             nothing flows when n + eps == 0);  raw: deta = dbeta
//   forget:   dalpha_i = sum_j S_{t-1}[i,j] dS~[i,j] (summed over i for a scalar gate);
//             G = alpha (.) dS~
// and dS0 = G at the end.
//
// One CTA of 4 d_v threads per (sequence, head) chain. A warp owns 8 value columns over all d_k
// rows (lanes: 2 column groups x 16 row groups of kRows = d_k / 16 consecutive rows), so every
// column reduction (S~^T k, G^T k) stays inside the warp; row reductions (dq, dk, per-channel
// dalpha) and the scalars (e . do, dbeta, scalar dalpha) go through shared memory with one
// block barrier per token.
//   phase F: the forward recurrence, saving the state at every kBlk-token boundary and every
//            residual e_t (the only forward quantities the reverse needs besides the inputs);
//   phase R: blocks of kBlk tokens in reverse order: the block's checkpoint and the state
//            half-way through the block are kept in shared memory, and before each reverse token
//            the state entering it is rebuilt from the nearer of the two with the stored
//            residuals (S <- alpha S + beta k e^T: no reductions).
#include <algorithm>

#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr int kBlk = 8;   // tokens per checkpoint block

struct BwdParams {
    const void *q, *k, *v, *dO;
    const float *alpha, *eta;
    float eps;
    const float *S0, *dST;
    float *dq, *dk, *dv, *dalpha, *deta, *dS0;
    float *ckpt;   // [B*H][nblk][DK][DV]
    float *e;      // [B, T, H, DV]
    int B, T, H, DK, DV, nblk;
    int beta_raw;
    float q_scale;
    const unsigned *only;   // NULL, or [B*H]: only chains with a nonzero mark run (the others return at once)
};

__device__ __forceinline__ void prefetch_l2(const void *ptr) {   // the 128-byte line holding ptr
    const uintptr_t line = reinterpret_cast<uintptr_t>(ptr) & ~static_cast<uintptr_t>(127);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
}

// Reduce 4 partial column sums over the 16 row-group lanes (lane bits 1-4) and hand every lane
// the 4 totals of its column group: a two-level reduce-scatter, two plain levels, then 4
// shuffles back.
__device__ __forceinline__ void colsum4(float (&x)[4], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8;
    float y[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float send = b4 ? x[j] : x[j + 2];
        const float keep = b4 ? x[j + 2] : x[j];
        y[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    const float send = b3 ? y[0] : y[1];
    const float keep = b3 ? y[1] : y[0];
    float w = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    w += __shfl_xor_sync(0xffffffffu, w, 4);
    w += __shfl_xor_sync(0xffffffffu, w, 2);
    // lane with bits (4, 3) = (hi, lo) holds column 2 hi + lo of its group
    const int cg = lane & 1;
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = __shfl_sync(0xffffffffu, w, ((j >> 1) << 4) | ((j & 1) << 3) | cg);
}

template <typename TIn, bool kChannel, int kRows>
__global__ void __launch_bounds__(512, 1) bwd_kernel(const BwdParams p) {
    extern __shared__ __align__(16) float bsm[];
    const int DK = p.DK, DV = p.DV, T = p.T;
    const int nwarps = DV / 8;
    // shared memory carve-up (floats)
    // thread-private state copies, interleaved by thread so a warp's float4 accesses are
    // contiguous: element (r, 4 columns) of thread t at float4 index r * blockDim + t
    float4 *sS = reinterpret_cast<float4 *>(bsm);     // state entering the block
    float4 *sMid = sS + kRows * blockDim.x;           // state entering the block's token kBlk / 2
    float *sk = bsm + 8 * kRows * blockDim.x;         // [kBlk][DK]
    float *sq = sk + kBlk * DK;                       // [kBlk][DK]
    float *sa = sq + kBlk * DK;                       // [kBlk][DK] (per-channel gate) or [kBlk]
    float *sv = sa + kBlk * DK;                       // [kBlk][DV]: v (phase F) or e (phase R)
    float *sdo = sv + kBlk * DV;                      // [kBlk][DV]
    float *sbeta = sdo + kBlk * DV;                   // [kBlk]
    float *sden = sbeta + kBlk;                       // [kBlk]: ||k||^2 + eps
    float *sas = sden + kBlk;                         // [kBlk]: scalar gate
    float *red = sas + kBlk;                          // [2][3][16 warps][DK] row partials
    float *reds = red + 2 * 3 * 16 * DK;              // [2][16 warps][4] scalar partials

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = lane & 1, rg = lane >> 1;
    const int h = blockIdx.x, b = blockIdx.y;
    const size_t bh = static_cast<size_t>(b) * p.H + h;
    if (p.only && p.only[bh] == 0u) return;
    const int col = warp * 8 + cg * 4;                // this lane's first value column
    const int r0 = rg * kRows;
    const bool live = r0 < DK;
    const int rr = live ? r0 : 0;
    auto tok = [&](int t) { return (static_cast<size_t>(b) * T + t) * p.H + h; };
    const float s = p.q_scale;
    float *ck = p.ckpt + bh * static_cast<size_t>(p.nblk) * DK * DV;

    // stage tokens [t0, t0 + n) of the block: k, q, gates, beta; v (phase F) or e (phase R), do
    auto stage = [&](int t0, int n, bool reverse) {
        const TIn *gk = static_cast<const TIn *>(p.k), *gq = static_cast<const TIn *>(p.q);
        for (int idx = tid; idx < n * DK; idx += blockDim.x) {
            const int u = idx / DK, c = idx - u * DK;
            const size_t g = tok(t0 + u) * DK + c;
            sk[u * DK + c] = to_f32(gk[g]);
            if (reverse) sq[u * DK + c] = to_f32(gq[g]);
            if (kChannel) sa[u * DK + c] = p.alpha[g];
        }
        for (int idx = tid; idx < n * DV; idx += blockDim.x) {
            const int u = idx / DV, c = idx - u * DV;
            const size_t g = tok(t0 + u) * DV + c;
            if (reverse) {
                sv[u * DV + c] = p.e[g];
                sdo[u * DV + c] = to_f32(static_cast<const TIn *>(p.dO)[g]);
            } else {
                sv[u * DV + c] = to_f32(static_cast<const TIn *>(p.v)[g]);
            }
        }
        if (!kChannel && tid < n) sas[tid] = p.alpha[tok(t0 + tid)];
        __syncthreads();
        for (int u = warp; u < n; u += nwarps) {   // ||k||^2 and beta, one warp per token
            float kk = 0.f;
            for (int c = lane; c < DK; c += 32) kk = fmaf(sk[u * DK + c], sk[u * DK + c], kk);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) kk += __shfl_xor_sync(0xffffffffu, kk, off);
            if (lane == 0) {
                const float eta = p.eta[tok(t0 + u)];
                sden[u] = kk + p.eps;
                sbeta[u] = kla_beta(eta, kk, p.eps, p.beta_raw);
            }
        }
        __syncthreads();
    };
    // Pull the inputs of tokens [t0, t0 + n) (and, in reverse, the block checkpoint) into L2 while
    // the current block runs, so the next block's staging waits on L2 rather than HBM.
    auto prefetch_block = [&](int t0, int n, bool reverse, int blk) {
        const int esz = sizeof(TIn);
        const int lk = (DK * esz + 127) / 128, lv = (DV * esz + 127) / 128, le = (DV * 4 + 127) / 128;
        const int la = kChannel ? (DK * 4 + 127) / 128 : 0;
        const int per = lk * (reverse ? 2 : 1) + (reverse ? le + lv : lv) + la + 1;
        for (int idx = tid; idx < n * per; idx += blockDim.x) {
            const int u = idx / per;
            int l = idx - u * per;
            const size_t tk = tok(t0 + u);
            const char *ptr;
            if (l < lk) ptr = static_cast<const char *>(p.k) + tk * DK * esz + l * 128;
            else if ((l -= lk) < (reverse ? lk : 0)) ptr = static_cast<const char *>(p.q) + tk * DK * esz + l * 128;
            else {
                if (reverse) l -= lk;
                if (!reverse && l < lv) ptr = static_cast<const char *>(p.v) + tk * DV * esz + l * 128;
                else if (reverse && l < le) ptr = reinterpret_cast<const char *>(p.e + tk * DV) + l * 128;
                else if (reverse && (l -= le) < lv) ptr = static_cast<const char *>(p.dO) + tk * DV * esz + l * 128;
                else {
                    l -= lv;
                    if (l < la) ptr = reinterpret_cast<const char *>(p.alpha + tk * DK) + l * 128;
                    else ptr = reinterpret_cast<const char *>(p.eta + tk);
                }
            }
            prefetch_l2(ptr);
        }
        if (reverse && live) {
#pragma unroll
            for (int r = 0; r < kRows; ++r) prefetch_l2(ck + (static_cast<size_t>(blk) * DK + r0 + r) * DV + col);
        }
    };
    auto rows_of = [&](const float *v, float (&out)[kRows]) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) out[r] = v[rr + r];
    };
    auto gate_rows = [&](int u, float (&a)[kRows]) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) a[r] = kChannel ? sa[u * DK + rr + r] : sas[u];
    };

    // ------------------------------------------------------------------ phase F: forward
    float S[kRows][4];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && p.S0) x = *reinterpret_cast<const float4 *>(p.S0 + (bh * DK + r0 + r) * DV + col);
        S[r][0] = x.x; S[r][1] = x.y; S[r][2] = x.z; S[r][3] = x.w;
    }
    for (int blk = 0; blk < p.nblk; ++blk) {
        const int t0 = blk * kBlk, n = min(kBlk, T - t0);
        if (live) {   // checkpoint: the state entering token t0
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                *reinterpret_cast<float4 *>(ck + (static_cast<size_t>(blk) * DK + r0 + r) * DV + col) =
                    make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
        }
        stage(t0, n, false);
        if (blk + 1 < p.nblk) prefetch_block(t0 + kBlk, min(kBlk, T - t0 - kBlk), false, blk + 1);
        for (int u = 0; u < n; ++u) {
            float kr[kRows], a[kRows];
            rows_of(sk + u * DK, kr);
            gate_rows(u, a);
            float pk[4] = {0.f, 0.f, 0.f, 0.f};
            if (live) {
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    const float ak = a[r] * kr[r];
#pragma unroll
                    for (int c = 0; c < 4; ++c) pk[c] = fmaf(ak, S[r][c], pk[c]);
                }
            }
            colsum4(pk, lane);
            const float beta = sbeta[u];
            float e[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) e[c] = sv[u * DV + col + c] - pk[c];
            if (rg == 0)
                *reinterpret_cast<float4 *>(p.e + tok(t0 + u) * DV + col) = make_float4(e[0], e[1], e[2], e[3]);
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const float bk = beta * kr[r];
#pragma unroll
                for (int c = 0; c < 4; ++c) S[r][c] = fmaf(a[r], S[r][c], bk * e[c]);
            }
        }
        __syncthreads();   // the staging area is rewritten by the next block
    }

    // ------------------------------------------------------------------ phase R: reverse
    float G[kRows][4];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && p.dST) x = *reinterpret_cast<const float4 *>(p.dST + (bh * DK + r0 + r) * DV + col);
        G[r][0] = x.x; G[r][1] = x.y; G[r][2] = x.z; G[r][3] = x.w;
    }
    // partial slots of warps that do not exist (d_v < 128) stay zero, so the sums below run over
    // all 16 slots without a bound
    for (int idx = tid; idx < 2 * 3 * 16 * DK + 2 * 16 * 4; idx += blockDim.x) red[idx] = 0.f;
    __syncthreads();
    const int nthr = blockDim.x;
    auto load_state = [&](const float4 *src) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float4 x = src[r * nthr + tid];
            S[r][0] = x.x; S[r][1] = x.y; S[r][2] = x.z; S[r][3] = x.w;
        }
    };
    auto store_state = [&](float4 *dst) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) dst[r * nthr + tid] = make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
    };
    // S <- alpha_w (.) S + beta_w k_w e_w^T with the stored residual of token w of the block
    auto replay = [&](int w) {
        float kr[kRows], a[kRows];
        rows_of(sk + w * DK, kr);
        gate_rows(w, a);
        const float beta = sbeta[w];
        const float4 ew = *reinterpret_cast<const float4 *>(sv + w * DV + col);
        const float e[4] = {ew.x, ew.y, ew.z, ew.w};
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float bk = beta * kr[r];
#pragma unroll
            for (int c = 0; c < 4; ++c) S[r][c] = fmaf(a[r], S[r][c], bk * e[c]);
        }
    };
    constexpr int kHalf = kBlk / 2;
    int par = 0;
    for (int blk = p.nblk - 1; blk >= 0; --blk) {
        const int t0 = blk * kBlk, n = min(kBlk, T - t0);
        // this lane's part of the block checkpoint (its own rows and columns: no barrier needed)
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (live) x = *reinterpret_cast<const float4 *>(ck + (static_cast<size_t>(blk) * DK + r0 + r) * DV + col);
            sS[r * nthr + tid] = x;
        }
        stage(t0, n, true);
        if (blk > 0) prefetch_block(t0 - kBlk, kBlk, true, blk - 1);
        if (n > kHalf) {   // the state entering token kHalf of the block
            load_state(sS);
            for (int w = 0; w < kHalf; ++w) replay(w);
            store_state(sMid);
        }
        for (int u = n - 1; u >= 0; --u) {
            // the state entering token t0 + u: the nearest saved state, then the stored updates
            const int from = u >= kHalf ? kHalf : 0;
            load_state(u >= kHalf ? sMid : sS);
            for (int w = from; w < u; ++w) replay(w);
            // the reverse step of token t = t0 + u
            float kr[kRows], qr[kRows], a[kRows];
            rows_of(sk + u * DK, kr);
            rows_of(sq + u * DK, qr);
            gate_rows(u, a);
            const float beta = sbeta[u];
            const float4 e4 = *reinterpret_cast<const float4 *>(sv + u * DV + col);
            const float4 d4 = *reinterpret_cast<const float4 *>(sdo + u * DV + col);
            const float e[4] = {e4.x, e4.y, e4.z, e4.w}, dov[4] = {d4.x, d4.y, d4.z, d4.w};
            float rowA[kRows], rowB[kRows], rowC[kRows];
            float gk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                float sdo_ = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float st = a[r] * S[r][c];              // S~
                    sdo_ = fmaf(st, dov[c], sdo_);
                    G[r][c] = fmaf(s * qr[r], dov[c], G[r][c]);   // read
                    gk[c] = fmaf(G[r][c], kr[r], gk[c]);
                }
                rowA[r] = sdo_;
            }
            if (!live) {
#pragma unroll
                for (int c = 0; c < 4; ++c) gk[c] = 0.f;
            }
            colsum4(gk, lane);
            float de[4], sc_edo = 0.f, sc_db = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                de[c] = beta * gk[c];
                sc_edo = fmaf(e[c], dov[c], sc_edo);
                sc_db = fmaf(gk[c], e[c], sc_db);
            }
            if (rg == 0)
                *reinterpret_cast<float4 *>(p.dv + tok(t0 + u) * DV + col) = make_float4(de[0], de[1], de[2], de[3]);
            float sc_da = 0.f;
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                float ge = 0.f, sde = 0.f, da = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float st = a[r] * S[r][c];
                    ge = fmaf(G[r][c], e[c], ge);
                    sde = fmaf(st, de[c], sde);
                    const float dst = fmaf(-kr[r], de[c], G[r][c]);   // dS~
                    da = fmaf(S[r][c], dst, da);
                    G[r][c] = a[r] * dst;                               // forget
                }
                rowB[r] = fmaf(beta, ge, -sde);
                rowC[r] = da;
                sc_da += da;
            }
            // row partials: combine the two column groups, then one row set per warp
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                rowA[r] += __shfl_xor_sync(0xffffffffu, rowA[r], 1);
                rowB[r] += __shfl_xor_sync(0xffffffffu, rowB[r], 1);
                rowC[r] += __shfl_xor_sync(0xffffffffu, rowC[r], 1);
            }
            float *rd = red + (par * 3 * 16 + warp) * DK;   // quantity q at rd + q * 16 * DK
            if (cg == 0 && live) {
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    rd[r0 + r] = rowA[r];
                    rd[16 * DK + r0 + r] = rowB[r];
                    rd[32 * DK + r0 + r] = rowC[r];
                }
            }
            // scalars: e . do and dbeta over the columns (row group 0 holds them), the scalar
            // dalpha over everything
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sc_da += __shfl_xor_sync(0xffffffffu, sc_da, off);
            sc_edo += __shfl_xor_sync(0xffffffffu, sc_edo, 1);
            sc_db += __shfl_xor_sync(0xffffffffu, sc_db, 1);
            if (lane == 0)
                reinterpret_cast<float4 *>(reds)[par * 16 + warp] = make_float4(sc_edo, sc_db, sc_da, 0.f);
            __syncthreads();
            {
                const size_t tk = tok(t0 + u);
                const float den = sden[u];
                const bool flows = p.beta_raw || den != 0.f;
                for (int idx = tid; idx < 3 * DK; idx += nthr) {
                    const int qn = idx / DK, i = idx - qn * DK;   // quantity: 0 dq, 1 dk, 2 dalpha
                    if (qn == 2 && !kChannel) {
                        if (i == 0) {
                            float dat = 0.f;
#pragma unroll
                            for (int w = 0; w < 16; ++w) dat += reinterpret_cast<const float4 *>(reds)[par * 16 + w].z;
                            p.dalpha[tk] = dat;
                        }
                        continue;
                    }
                    const float *src = red + ((par * 3 + qn) * 16) * DK + i;
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < 16; ++w) acc += src[w * DK];
                    if (qn == 2) {
                        p.dalpha[tk * DK + i] = acc;
                        continue;
                    }
                    float edo = 0.f, db = 0.f;
#pragma unroll
                    for (int w = 0; w < 16; ++w) {
                        const float4 x = reinterpret_cast<const float4 *>(reds)[par * 16 + w];
                        edo += x.x;
                        db += x.y;
                    }
                    const float ki = sk[u * DK + i];
                    if (qn == 0) {
                        p.dq[tk * DK + i] = s * fmaf(beta * ki, edo, acc);
                    } else {
                        float dki = acc;
                        if (!p.beta_raw && flows) dki = fmaf(-2.f * beta * db / den, ki, dki);
                        p.dk[tk * DK + i] = dki;
                        if (i == 0) p.deta[tk] = p.beta_raw ? db : (flows ? db / den : 0.f);
                    }
                }
            }
            par ^= 1;   // the other buffer is rewritten only after the next barrier
        }
        __syncthreads();   // the staging area is rewritten by the next block
    }
    if (p.dS0 && live) {
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            *reinterpret_cast<float4 *>(p.dS0 + (bh * DK + r0 + r) * DV + col) =
                make_float4(G[r][0], G[r][1], G[r][2], G[r][3]);
    }
}

size_t bwd_smem_bytes(int DK, int DV, int rows) {
    const size_t threads = 4ull * DV;
    const size_t floats = 8ull * rows * threads + 3ull * kBlk * DK + 2ull * kBlk * DV + 3 * kBlk +
                          2ull * 3 * 16 * DK + 2 * 16 * 4;
    return floats * sizeof(float);
}

template <typename TIn, bool kChannel>
cudaError_t launch_t(const BwdArgs &a, const unsigned *only) {
    const int nblk = (a.T + kBlk - 1) / kBlk;
    float *ck = static_cast<float *>(a.workspace);
    float *ew = ck + static_cast<size_t>(a.B) * a.H * nblk * a.d_k * a.d_v;
    BwdParams p{a.q, a.k, a.v, a.dO, a.alpha, a.eta, a.eps, a.S0, a.dS_T, a.dq, a.dk, a.dv, a.dalpha, a.deta,
                a.dS0, ck, ew, a.B, a.T, a.H, a.d_k, a.d_v, nblk, a.beta_raw, a.q_scale, only};
    const int rows = std::max(1, a.d_k / 16);
    const size_t smem = bwd_smem_bytes(a.d_k, a.d_v, rows);
    auto kern = rows == 1 ? bwd_kernel<TIn, kChannel, 1>
              : rows == 2 ? bwd_kernel<TIn, kChannel, 2>
              : rows == 4 ? bwd_kernel<TIn, kChannel, 4>
                          : bwd_kernel<TIn, kChannel, 8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(a.H, a.B);
    kern<<<grid, 4 * a.d_v, smem, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

// The chunkwise tensor-core backward (kla_bwd_chunk.cu, kla_bwd_chunk_ch.cu): bf16, d_k = d_v = 128.
bool bwd_chunk_supports(const BwdArgs &a);
size_t bwd_chunk_workspace_bytes(int B, int T, int H, kla_gate gate);
cudaError_t launch_bwd_chunk(const BwdArgs &a);

size_t bwd_seq_workspace_bytes(int B, int T, int H, int d_k, int d_v) {
    if (B < 1 || H < 1 || T < 1) return 0;
    const size_t nblk = (static_cast<size_t>(T) + kBlk - 1) / kBlk;
    return (static_cast<size_t>(B) * H * nblk * d_k * d_v + static_cast<size_t>(B) * T * H * d_v) * sizeof(float);
}

size_t bwd_workspace_bytes(int B, int T, int H, int d_k, int d_v) {   // either path, either gate
    const size_t seq = bwd_seq_workspace_bytes(B, T, H, d_k, d_v);
    if (!(d_k == 128 && d_v == 128 && T > kShortSeqMaxT)) return seq;
    return std::max({seq, bwd_chunk_workspace_bytes(B, T, H, KLA_GATE_SCALAR),
                     bwd_chunk_workspace_bytes(B, T, H, KLA_GATE_CHANNEL)});
}

cudaError_t launch_bwd_seq(const BwdArgs &a, const unsigned *only) {
    const bool ch = a.gate == KLA_GATE_CHANNEL;
    if (a.dtype == KLA_DTYPE_BF16)
        return ch ? launch_t<__nv_bfloat16, true>(a, only) : launch_t<__nv_bfloat16, false>(a, only);
    return ch ? launch_t<float, true>(a, only) : launch_t<float, false>(a, only);
}

cudaError_t launch_bwd(const BwdArgs &a) {
    if (bwd_chunk_supports(a)) return launch_bwd_chunk(a);
    return launch_bwd_seq(a, nullptr);
}

}  // namespace kla
