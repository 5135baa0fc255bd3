// kla_bwd_chunk.cu -- chunkwise backward pass on the tensor cores: bf16 q/k/v/dO, scalar gate,
// d_k = d_v = 128, chunk C = 64, fp32 gradients.
//
// The pages give no backward algebra (GeekNews, "Revisando las variantes de atencion lineal de la
// familia DeltaNet", section "KDA por chunks", names training as the use of the chunk mode). This
// differentiates the chunk form of the forward (same page and section; KLA page, section
// "Implementazione": beta enters only through the chunk solver). Per chunk, with S the state
// entering it, G the in-chunk inclusive log-decay prefix, gamma = e^G, Gamma = e^{G_end},
// e_end = e^{G_end - G}, ratio_ij = e^{G_i - G_j}, beta = eta / (||k||^2 + eps) (raw mode: eta):
//   forward:  R = strict_lower(beta_i ratio_ij k_i.k_j), T = (I + R)^{-1},
//             W = T diag(beta gamma) K,  U = T diag(beta) V,  E = U - W S,
//             O = s (diag(gamma) Q S + A E),  A = lower(ratio_ij q_i.k_j),
//             S' = Gamma S + (diag(e_end) K)^T E.
//   reverse, with dS' = dL/dS' arriving from the next chunk and dO = dL/dO:
//             dE  = diag(e_end) K dS' + s A^T dO
//             dS  = Gamma dS' + s (diag(gamma) Q)^T dO - W^T dE           (to the previous chunk)
//             dW  = -dE S^T,  dXK = T^T dW,  dXV = T^T dE
//             dT  = dW K^T diag(beta gamma) + dE V^T diag(beta),  dR = -strict_lower(T^T dT T^T)
//             dA  = s lower(dO E^T);  dAr = dA . ratio,  dRr = dR . ratio
//             dq  = s diag(gamma) dO S^T + dAr K
//             dk  = diag(e_end) E dS'^T + diag(beta gamma) dXK + dAr^T Q + diag(beta) dRr K
//                   + (diag(beta) dRr)^T K  - 2 beta dbeta / (||k||^2 + eps) k     (KLA only)
//             dv  = diag(beta) dXV
//             dbeta_i = gamma_i k_i.dXK_i + v_i.dXV_i + sum_j dRr_ij k_i.k_j;   deta = dbeta / den
//             dG_i    = gamma_i q_i.dQg_i + beta_i gamma_i k_i.dXK_i + rowsum_i(M) - colsum_i(M)
//                       + rowsum_i(N) - colsum_i(N) - e_end_i k_i.dKt_i
//                       (+ sum_j e_end_j k_j.dKt_j + Gamma <S, dS'> for the chunk's last row)
//             with dQg = s dO S^T, dKt = E dS'^T, M = dAr . (q_i.k_j), N = beta_i dRr . (k_i.k_j);
//             d log alpha_t = sum over the chunk's rows i >= t of dG_i,  dalpha = that / alpha.
//
// Four kernels (one pass over the workspace each way):
//   prep_tc_kernel   (chunk-parallel)  gates, [K;Q]K^T, R and A, T by blocked substitution (fp32),
//                                      W and U; stores G, beta, den, W, U, A and T per chunk
//                                      (tcgen05, kla_bwd_prep_tc.cu);
//   carry_tc_kernel<false>             the state carry S_c -> S_{c+1} per chain (fp32 registers,
//                                      tcgen05 products), storing S_c and E_c per chunk;
//   carry_tc_kernel<true>              the reverse carry dS_{c+1} -> dS_c per chain, storing dS_{c+1}
//                                      and dE_c per chunk, and dS0 (both in kla_bwd_carry_tc.cu);
//   bwd_grad_kernel  (chunk-parallel)  every gradient of the chunk's tokens from S_c, dS_{c+1},
//                                      E_c, dE_c, T and the inputs.
// In the gradient kernel every product is a warp-level bf16 mma.sync (m16n8k16, fp32 accumulate)
// on 64- or 128-wide tiles staged in shared memory with rows padded by 16 bytes, so that every
// ldmatrix phase hits 8 distinct bank quads. Operands are bf16 (inputs as stored;
// derived tiles rounded once); the carried states, the solve and every sum of a gradient are fp32.
#include <algorithm>
#include <mutex>

#include "kla_bwd_chunk.cuh"

namespace kla {
namespace {

using namespace bwdc;

// Segments for the two carries of a long chain (the forward prefill's sequence-parallel scan,
// applied to them): both carries are affine in their state, X_end = M X_start + Z over a
// segment. Cost model in chunk-steps, one CTA per SM: pass 1 runs the value runs of segments
// 0..n-2 and the transitions of 1..n-2, pass 3 reruns 1..n-1; split only when it saves a fifth.
struct CarryPlan {
    int nseg, seg_len;   // seg_len in chunks
};
CarryPlan carry_plan(int chains, int nc) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0)
        return {1, nc};
    auto waves = [&](long ctas) { return (ctas + sms - 1) / sms; };
    double best = 0.8 * static_cast<double>(waves(chains)) * nc;
    int best_n = 1;
    for (int n = 2; n <= 64; ++n) {
        const int L = (nc + n - 1) / n;
        if (L < 8) break;
        const int nn = (nc + L - 1) / L;
        if (nn < 2) continue;
        const double cost = static_cast<double>(waves(static_cast<long>(chains) * (2 * nn - 3)) +
                                                waves(static_cast<long>(chains) * (nn - 1))) * L;
        if (cost < best) {
            best = cost;
            best_n = n;
        }
    }
    if (best_n <= 1) return {1, nc};
    const int L = (nc + best_n - 1) / best_n;
    return {(nc + L - 1) / L, L};
}

// ============================================================== kernel 1: per-chunk operands
// Gates and their prefix, ||k||^2 from the diagonal of K K^T, [K;Q] K^T, R and A, T by blocked
// substitution (fp32), W and U, storing G, beta, den, W, U, A and T per chunk: on the tensor
// cores, launch_prep_tc in kla_bwd_prep_tc.cu.

// ============================================================== kernel 2: the carry across chunks
// The forward carry (X = S entering chunk c, c ascending: E = U - W X, X <- Gamma X +
// K^T diag(e_end) E, storing X and E per chunk) and the reverse carry (X = dL/d(state leaving
// chunk c), c descending: dE = diag(e_end) K X + s A^T dO, X <- Gamma X + (s diag(gamma) Q)^T dO
// - W^T dE, storing X and dE per chunk) run on the tensor cores: launch_carry_tc in
// kla_bwd_carry_tc.cu.

// ============================================================== kernel 3: gradients of a chunk
// One CTA of 16 warps per chunk, in two sides that each own one 64 x 128 accumulator in
// registers (32 x 32 per warp):
//   K side (warps 0-7): dk <- e_end dKt + beta gamma dXK + dAr^T Q + (beta dRr)^T K + beta dRr K;
//                       the 64 x 64 products QK^T, dA, KK^T, Y = T^T dT and dR (16 x 32 per warp);
//   Q side (warps 8-15): dq <- s gamma dO S^T + dAr K;  dW = -dE S^T, dv = beta T^T dE, dT, and
//                       beta dRr K, handed to the K side through shared memory.
// Phases (block barriers between them): 1 dKt, QK^T, dA | <S,dS'>, dQg, dW;  2 dXK, dAr^T Q, KK^T |
// dXV, dT;  3 Y, dR | dAr K;  4 (beta dRr)^T K | beta dRr K;  then the per-token sums.
struct GradParams {
    const bf16 *q, *k, *v, *dO;
    const float *alpha;
    float q_scale;
    int beta_raw;
    float *dq, *dk, *dv, *dalpha, *deta;
    int B, T, H, nc;
    Ws ws;
};
constexpr int kGradThreads = 512;
enum { RQ_KT = 0, RQ_Q, RQ_B1, RQ_B2, RQ_B3, RQ_MA, kRowQty };   // per-row partial sums
enum { CQ_MA = 0, CQ_MR, kColQty };                             // per-column partial sums
constexpr int GR_Q = 0, GR_K = GR_Q + kTileTok, GR_V = GR_K + kTileTok, GR_DO = GR_V + kTileTok;
constexpr int GR_E = GR_DO + kTileTok, GR_DE = GR_E + kTileTok;
constexpr int GR_S = GR_DE + kTileTok, GR_DS = GR_S + kTileSt;     // S_c, dS_{c+1}
constexpr int GR_DW = GR_S;                                         // dW over S once S is read
constexpr int GR_T = GR_DS + kTileSt, GR_DAR = GR_T + kTileSq, GR_DT = GR_DAR + kTileSq;
constexpr int GR_Y = GR_DS, GR_DRR = GR_Y + kTileSq, GR_BDRR = GR_DRR + kTileSq;   // over dS' in phase 3
constexpr int GR_CG = GR_DT + kTileSq;
constexpr int kPX1 = kD + 8;                                        // fp32 hand-over tile over V and dO (phase 3)
constexpr int GR_XCH = GR_V;
static_assert(GR_XCH + kC * kPX1 * 4 <= GR_DO + kTileTok, "hand-over tile");
constexpr int GR_RROW = GR_CG + static_cast<int>(kCgFloats) * 4;   // fp32 [kRowQty][4][64]
constexpr int GR_RCOL = GR_RROW + kRowQty * 4 * kC * 4;            // fp32 [kColQty][4][64]
constexpr int GR_SC = GR_RCOL + kColQty * 4 * kC * 4;              // fp32 [8] partials of <S, dS'>
constexpr int GR_KC = GR_SC + 8 * 4;                               // fp32 [64] coefficient of k in dk
constexpr int GR_XS = GR_KC + kC * 4;                              // fp32 [4] scratch of the token pass
constexpr int GR_BYTES = GR_XS + 16;
static_assert(GR_BYTES <= 232448, "gradient kernel shared memory");
constexpr uint32_t kBarToken = 1, kBarK = 2, kBarQ = 3;           // named barriers (0 = __syncthreads)

__global__ void __launch_bounds__(kGradThreads, 1) bwd_grad_kernel(GradParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    auto tile = [&](int off) { return reinterpret_cast<bf16 *>(smem + off); };
    bf16 *sQ = tile(GR_Q), *sK = tile(GR_K), *sV = tile(GR_V), *sDO = tile(GR_DO), *sE = tile(GR_E),
         *sDE = tile(GR_DE), *sS = tile(GR_S), *sDS = tile(GR_DS), *sT = tile(GR_T), *sDW = tile(GR_DW),
         *sDAR = tile(GR_DAR), *sDT = tile(GR_DT), *sY = tile(GR_Y), *sDRR = tile(GR_DRR), *sBDRR = tile(GR_BDRR);
    const float *cg = reinterpret_cast<const float *>(smem + GR_CG);
    float(*rrow)[4][kC] = reinterpret_cast<float(*)[4][kC]>(smem + GR_RROW);
    float(*rcol)[4][kC] = reinterpret_cast<float(*)[4][kC]>(smem + GR_RCOL);
    float *rsc = reinterpret_cast<float *>(smem + GR_SC), *kcoef = reinterpret_cast<float *>(smem + GR_KC),
          *xs = reinterpret_cast<float *>(smem + GR_XS);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, q4 = lane & 3;
    const int c = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
    const int t0 = c * kC, L = min(kC, p.T - t0);
    const size_t n = static_cast<size_t>(bh) * p.nc + c;
    const size_t rs = static_cast<size_t>(p.H) * kD;
    const size_t tok0 = (static_cast<size_t>(b) * p.T + t0) * p.H + h;   // (b, t0, h)

    load_tok(sQ, p.q + tok0 * kD, rs, L, tid, kGradThreads);
    load_tok(sK, p.k + tok0 * kD, rs, L, tid, kGradThreads);
    load_tok(sV, p.v + tok0 * kD, rs, L, tid, kGradThreads);
    load_tok(sDO, p.dO + tok0 * kD, rs, L, tid, kGradThreads);
    load_dense<kD>(sE, p.ws.E + n * kC * kD, kC, tid, kGradThreads);
    load_dense<kD>(sDE, p.ws.dE + n * kC * kD, kC, tid, kGradThreads);
    load_dense<kD>(sS, p.ws.S + n * kD * kD, kD, tid, kGradThreads);
    load_dense<kD>(sDS, p.ws.dS + n * kD * kD, kD, tid, kGradThreads);
    load_dense<kC>(sT, p.ws.Tm + n * kC * kC, kC, tid, kGradThreads);
    if (tid < static_cast<int>(kCgFloats) / 4)
        cp16(smem + GR_CG + 16 * tid, p.ws.cg + n * kCgFloats + 4 * tid, true);
    cp_commit();
    cp_wait<0>();
    __syncthreads();

    const bool kside = warp < 8;
    const int sw = warp & 7;
    const int r1 = 32 * (sw & 1), c1 = 32 * (sw >> 1), cb1 = sw >> 1;   // 64 x 128 products: 32 x 32 per warp
    const int r2 = 16 * (sw & 3), c2 = 32 * (sw >> 2), cb2 = sw >> 2;   // 64 x 64 products: 16 x 32 per warp
    const float s = p.q_scale, Gend = cg[kC - 1];
    auto row1 = [&](int mi, int hh) { return r1 + 16 * mi + g + 8 * hh; };
    auto row2 = [&](int hh) { return r2 + g + 8 * hh; };
    // sum over this thread's columns of X[row][col] * a for a 64 x 128 accumulator and a bf16 tile X
    auto rowdot1 = [&](const bf16 *X, const float (&a)[2][4][4], int mi, int hh) {
        float sum = 0.f;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const float2 x = ld_pair(X, kP, row1(mi, hh), c1 + 8 * ni + 2 * q4);
            sum = fmaf(x.x, a[mi][ni][2 * hh], fmaf(x.y, a[mi][ni][2 * hh + 1], sum));
        }
        return sum;
    };
    // row partials over the 4 lanes of a row, into slot `cb` of quantity `qi`
    auto put_row = [&](int qi, int cb, int row, float x) {
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        if (q4 == 0) rrow[qi][cb][row] = x;
    };
    // column partials of a 64 x 64 product over the 16 rows of the warp, into row block sw & 3
    auto put_col = [&](int qi, const float (&x)[4][2]) {
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float y = x[ni][e];
                y += __shfl_xor_sync(0xffffffffu, y, 4);
                y += __shfl_xor_sync(0xffffffffu, y, 8);
                y += __shfl_xor_sync(0xffffffffu, y, 16);
                if (g == 0) rcol[qi][sw & 3][c2 + 8 * ni + 2 * q4 + e] = y;
            }
    };
    auto ratio = [&](int i, int j) { return __expf(cg[i] - cg[j]); };

    float acc[2][4][4];   // the side's 64 x 128 accumulator (dk or dq)
    float tmp[2][4][4];
    float kk[1][4][4];    // K side: K K^T, kept from phase 2 to phase 3
    if (kside) {
        // ---- phase 1 (K side): dKt = E dS'^T -> dk = e_end dKt;  QK^T;  dA = s lower(dO E^T)
        zero(acc[0]);
        zero(acc[1]);
        gemm_m<2, 4, 8, false, false>(acc, sptr(sE), kP, r1, 0, sptr(sDS), kP, c1, 0, lane);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = row1(mi, hh);
                put_row(RQ_KT, cb1, r, rowdot1(sK, acc, mi, hh));
                const float ee = __expf(Gend - cg[r]);
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) {
                    acc[mi][ni][2 * hh] *= ee;
                    acc[mi][ni][2 * hh + 1] *= ee;
                }
            }
        float qk[1][4][4], da[1][4][4];
        zero(qk[0]);
        zero(da[0]);
        gemm_m<1, 4, 8, false, false>(qk, sptr(sQ), kP, r2, 0, sptr(sK), kP, c2, 0, lane);
        gemm_m<1, 4, 8, false, false>(da, sptr(sDO), kP, r2, 0, sptr(sE), kP, c2, 0, lane);
        float colm[4][2] = {};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int i = row2(hh);
            float rowm = 0.f;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                float v2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int j = c2 + 8 * ni + 2 * q4 + e;
                    const float x = j <= i ? s * da[0][ni][2 * hh + e] * ratio(i, j) : 0.f;
                    v2[e] = x;
                    const float m = x * qk[0][ni][2 * hh + e];
                    rowm += m;
                    colm[ni][e] += m;
                }
                st_pair(sDAR, kPs, i, c2 + 8 * ni + 2 * q4, v2[0], v2[1]);
            }
            put_row(RQ_MA, cb2, i, rowm);
        }
        put_col(CQ_MA, colm);
    } else {
        // ---- phase 1 (Q side): <S, dS'>;  dQg = s dO S^T -> dq = gamma dQg;  dW = -dE S^T
        {
            float sum = 0.f;
            for (int i = tid - 256; i < kD * 16; i += 256) {
                const int r = i >> 4, cc = (i & 15) * 8;
                const uint4 x = *reinterpret_cast<const uint4 *>(sS + r * kP + cc);
                const uint4 y = *reinterpret_cast<const uint4 *>(sDS + r * kP + cc);
                const uint32_t *xw = reinterpret_cast<const uint32_t *>(&x), *yw = reinterpret_cast<const uint32_t *>(&y);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 u = unpack2(xw[e]), w = unpack2(yw[e]);
                    sum = fmaf(u.x, w.x, fmaf(u.y, w.y, sum));
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) rsc[sw] = sum;
        }
        zero(acc[0]);
        zero(acc[1]);
        gemm_m<2, 4, 8, false, false>(acc, sptr(sDO), kP, r1, 0, sptr(sS), kP, c1, 0, lane);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = row1(mi, hh);
                put_row(RQ_Q, cb1, r, s * rowdot1(sQ, acc, mi, hh));
                const float f = s * __expf(cg[r]);
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) {
                    acc[mi][ni][2 * hh] *= f;
                    acc[mi][ni][2 * hh + 1] *= f;
                }
            }
        zero(tmp[0]);
        zero(tmp[1]);
        gemm_m<2, 4, 8, false, false>(tmp, sptr(sDE), kP, r1, 0, sptr(sS), kP, c1, 0, lane);
        bar_named(kBarQ, 256);   // every read of S is done (only this side reads it): dW goes over it
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni)
                    st_pair(sDW, kP, row1(mi, hh), c1 + 8 * ni + 2 * q4, -tmp[mi][ni][2 * hh], -tmp[mi][ni][2 * hh + 1]);
    }
    __syncthreads();   // dW and dAr are visible; dS' is no longer read

    if (kside) {
        // ---- phase 2 (K side): dXK = T^T dW -> dk += beta gamma dXK;  dk += dAr^T Q;  KK^T
        zero(tmp[0]);
        zero(tmp[1]);
        gemm_m<2, 4, 4, true, true>(tmp, sptr(sT), kPs, r1, 0, sptr(sDW), kP, c1, 0, lane);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = row1(mi, hh);
                put_row(RQ_B1, cb1, r, rowdot1(sK, tmp, mi, hh));
                const float f = cg[kC + r] * __expf(cg[r]);
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) {
                    acc[mi][ni][2 * hh] = fmaf(f, tmp[mi][ni][2 * hh], acc[mi][ni][2 * hh]);
                    acc[mi][ni][2 * hh + 1] = fmaf(f, tmp[mi][ni][2 * hh + 1], acc[mi][ni][2 * hh + 1]);
                }
            }
        gemm_m<2, 4, 4, true, true>(acc, sptr(sDAR), kPs, r1, 0, sptr(sQ), kP, c1, 0, lane);
        zero(kk[0]);
        gemm_m<1, 4, 8, false, false>(kk, sptr(sK), kP, r2, 0, sptr(sK), kP, c2, 0, lane);
    } else {
        // ---- phase 2 (Q side): dXV = T^T dE -> dv;  dT;  dq += dAr K -> dq out
        zero(tmp[0]);
        zero(tmp[1]);
        gemm_m<2, 4, 4, true, true>(tmp, sptr(sT), kPs, r1, 0, sptr(sDE), kP, c1, 0, lane);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = row1(mi, hh);
                put_row(RQ_B2, cb1, r, rowdot1(sV, tmp, mi, hh));
                if (r < L) {
                    const float bt = cg[kC + r];
                    float *dst = p.dv + (tok0 + static_cast<size_t>(r) * p.H) * kD;
#pragma unroll
                    for (int ni = 0; ni < 4; ++ni)
                        *reinterpret_cast<float2 *>(dst + c1 + 8 * ni + 2 * q4) =
                            make_float2(bt * tmp[mi][ni][2 * hh], bt * tmp[mi][ni][2 * hh + 1]);
                }
            }
        {   // dT = dW K^T diag(beta gamma) + dE V^T diag(beta)
            float a1[1][4][4], a2[1][4][4];
            zero(a1[0]);
            zero(a2[0]);
            gemm_m<1, 4, 8, false, false>(a1, sptr(sDW), kP, r2, 0, sptr(sK), kP, c2, 0, lane);
            gemm_m<1, 4, 8, false, false>(a2, sptr(sDE), kP, r2, 0, sptr(sV), kP, c2, 0, lane);
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int j = c2 + 8 * ni + 2 * q4;
                const float bj0 = cg[kC + j], bj1 = cg[kC + j + 1];
                const float fj0 = bj0 * __expf(cg[j]), fj1 = bj1 * __expf(cg[j + 1]);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    st_pair(sDT, kPs, row2(hh), j, fmaf(fj0, a1[0][ni][2 * hh], bj0 * a2[0][ni][2 * hh]),
                            fmaf(fj1, a1[0][ni][2 * hh + 1], bj1 * a2[0][ni][2 * hh + 1]));
            }
        }
    }
    __syncthreads();   // dT is visible

    float *xch = reinterpret_cast<float *>(smem + GR_XCH);   // fp32 [64][kPX1]: Q side -> K side
    if (kside) {
        // ---- phase 3 (K side): Y = T^T dT;  dR = -strict_lower(Y T^T), dRr = dR . ratio
        {
            float y[1][4][4];
            zero(y[0]);
            gemm_m<1, 4, 4, true, true>(y, sptr(sT), kPs, r2, 0, sptr(sDT), kPs, c2, 0, lane);
#pragma unroll
            for (int ni = 0; ni < 4; ++ni)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    st_pair(sY, kPs, row2(hh), c2 + 8 * ni + 2 * q4, y[0][ni][2 * hh], y[0][ni][2 * hh + 1]);
        }
        bar_named(kBarK, 256);
        {
            float dr[1][4][4];
            zero(dr[0]);
            gemm_m<1, 4, 4, false, false>(dr, sptr(sY), kPs, r2, 0, sptr(sT), kPs, c2, 0, lane);
            float coln[4][2] = {};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = row2(hh);
                const float bi = cg[kC + i];
                float rown = 0.f;
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) {
                    float v2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = c2 + 8 * ni + 2 * q4 + e;
                        const float x = j < i ? -dr[0][ni][2 * hh + e] * ratio(i, j) : 0.f;
                        v2[e] = x;
                        const float m = x * kk[0][ni][2 * hh + e];
                        rown += m;
                        coln[ni][e] += bi * m;
                    }
                    st_pair(sDRR, kPs, i, c2 + 8 * ni + 2 * q4, v2[0], v2[1]);
                    st_pair(sBDRR, kPs, i, c2 + 8 * ni + 2 * q4, bi * v2[0], bi * v2[1]);
                }
                put_row(RQ_B3, cb2, i, rown);
            }
            put_col(CQ_MR, coln);
        }
    } else {
        // ---- phase 3 (Q side): dq += dAr K -> dq out
        gemm_m<2, 4, 4, false, true>(acc, sptr(sDAR), kPs, r1, 0, sptr(sK), kP, c1, 0, lane);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = row1(mi, hh);
                if (r >= L) continue;
                float *dst = p.dq + (tok0 + static_cast<size_t>(r) * p.H) * kD;
#pragma unroll
                for (int ni = 0; ni < 4; ++ni)
                    *reinterpret_cast<float2 *>(dst + c1 + 8 * ni + 2 * q4) =
                        make_float2(acc[mi][ni][2 * hh], acc[mi][ni][2 * hh + 1]);
            }
    }
    __syncthreads();   // dRr and beta dRr are visible
    if (kside) {
        gemm_m<2, 4, 4, true, true>(acc, sptr(sBDRR), kPs, r1, 0, sptr(sK), kP, c1, 0, lane);   // dk += (beta dRr)^T K
    } else {
        // beta dRr K for the K side, handed over in fp32 at the same fragment positions
        zero(tmp[0]);
        zero(tmp[1]);
        gemm_m<2, 4, 4, false, true>(tmp, sptr(sDRR), kPs, r1, 0, sptr(sK), kP, c1, 0, lane);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = row1(mi, hh);
                const float bt = cg[kC + r];
#pragma unroll
                for (int ni = 0; ni < 4; ++ni)
                    *reinterpret_cast<float2 *>(xch + r * kPX1 + c1 + 8 * ni + 2 * q4) =
                        make_float2(bt * tmp[mi][ni][2 * hh], bt * tmp[mi][ni][2 * hh + 1]);
            }
    }
    __syncthreads();   // the hand-over and every partial sum are in shared memory
    if (kside) {
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) {
                    const float2 x = *reinterpret_cast<const float2 *>(xch + row1(mi, hh) * kPX1 + c1 + 8 * ni + 2 * q4);
                    acc[mi][ni][2 * hh] += x.x;
                    acc[mi][ni][2 * hh + 1] += x.y;
                }
    }

    // per token (warps 8-9, token = tid - 256): dbeta, deta, the k coefficient, dG and its reverse prefix
    if (tid >= 256 && tid < 256 + kC) {
        const int t = tid - 256;
        auto rsum4 = [&](int qi) { return rrow[qi][0][t] + rrow[qi][1][t] + rrow[qi][2][t] + rrow[qi][3][t]; };
        auto rsum2 = [&](int qi) { return rrow[qi][0][t] + rrow[qi][1][t]; };
        const float kt_raw = rsum4(RQ_KT), qd = rsum4(RQ_Q), b1 = rsum4(RQ_B1), b2 = rsum4(RQ_B2);
        const float b3 = rsum2(RQ_B3), ma = rsum2(RQ_MA);
        const float cma = rcol[CQ_MA][0][t] + rcol[CQ_MA][1][t] + rcol[CQ_MA][2][t] + rcol[CQ_MA][3][t];
        const float cmr = rcol[CQ_MR][0][t] + rcol[CQ_MR][1][t] + rcol[CQ_MR][2][t] + rcol[CQ_MR][3][t];
        const float gt = __expf(cg[t]), et = __expf(Gend - cg[t]), bt = cg[kC + t], den = cg[2 * kC + t];
        const float dbeta = fmaf(gt, b1, b2 + b3);
        float deta = dbeta, kc = 0.f;
        if (!p.beta_raw) {
            const bool flows = den != 0.f;
            deta = flows ? dbeta / den : 0.f;
            kc = flows ? -2.f * bt * dbeta / den : 0.f;
        }
        kcoef[t] = kc;
        const float kt = et * kt_raw;
        float dG = gt * qd + bt * gt * b1 + ma - cma + bt * b3 - cmr - kt;
        // the chunk's last row also carries the end decay's terms: sum_j e_end_j k_j.dKt_j + Gamma <S, dS'>
        float ktot = kt;
#pragma unroll
        for (int o = 16; o; o >>= 1) ktot += __shfl_xor_sync(0xffffffffu, ktot, o);
        if (lane == 0) xs[warp - 8] = ktot;
        bar_named(kBarToken, 64);
        if (t == kC - 1) {
            float sds = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) sds += rsc[w];
            dG += xs[0] + xs[1] + __expf(Gend) * sds;
        }
        // reverse inclusive prefix over the 64 tokens: suffix sums within each warp, then the
        // first warp adds the second warp's total
        float x = dG;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, x, o);
            if (lane + o < 32) x += y;
        }
        if (t == 32) xs[2] = x;
        bar_named(kBarToken, 64);
        if (t < 32) x += xs[2];
        if (t < L) {
            const size_t o = tok0 + static_cast<size_t>(t) * p.H;
            p.deta[o] = deta;
            p.dalpha[o] = x / p.alpha[o];
        }
    }
    __syncthreads();   // kcoef is visible

    if (kside) {   // dk += kcoef k; write dk
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = row1(mi, hh);
                if (r >= L) continue;
                const float kc = kcoef[r];
                float *dst = p.dk + (tok0 + static_cast<size_t>(r) * p.H) * kD;
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) {
                    const int col = c1 + 8 * ni + 2 * q4;
                    const float2 kx = ld_pair(sK, kP, r, col);
                    *reinterpret_cast<float2 *>(dst + col) =
                        make_float2(fmaf(kc, kx.x, acc[mi][ni][2 * hh]), fmaf(kc, kx.y, acc[mi][ni][2 * hh + 1]));
                }
            }
    }
}

}  // namespace

namespace {
// Per-channel gate: one mark per chain (256-byte aligned) in front of the rest of the workspace.
size_t mark_bytes(int B, int H) { return (static_cast<size_t>(B) * H * sizeof(unsigned) + 255) & ~size_t(255); }
size_t record_bytes(int B, int T, int H, bool ch) {
    const size_t nc = (static_cast<size_t>(T) + kC - 1) / kC, chains = static_cast<size_t>(B) * H;
    const CarryPlan pl = carry_plan(B * H, static_cast<int>(nc));
    const size_t seg = pl.nseg > 1 ? 3 * chains * pl.nseg * kD * kD * sizeof(float) : 0;
    return chains * nc * ws_bytes_per_chunk(ch) + seg;
}
}  // namespace

// Scalar gate: the per-chunk records (and segment states). Per-channel gate: the marks, then room
// for either the records or the token-sequential path's checkpoints, which rerun the marked chains
// after the chunkwise kernels are done with the records.
size_t bwd_chunk_workspace_bytes(int B, int T, int H, kla_gate gate) {
    if (B < 1 || T < 1 || H < 1) return 0;
    if (gate != KLA_GATE_CHANNEL) return record_bytes(B, T, H, false);
    return mark_bytes(B, H) + std::max(record_bytes(B, T, H, true), bwd_seq_workspace_bytes(B, T, H, kD, kD));
}

// Sequences of at most kShortSeqMaxT tokens take the token-by-token fp32 backward: there a
// gradient can hinge on a handful of dot products taken after a bf16 rounding, with nothing to
// average the rounding over, and the sequential walk is short.
bool bwd_chunk_supports(const BwdArgs &a) {
    auto al16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    const bool ch = a.gate == KLA_GATE_CHANNEL;
    return a.dtype == KLA_DTYPE_BF16 && (a.gate == KLA_GATE_SCALAR || ch) && a.d_k == kD && a.d_v == kD &&
           a.T > kShortSeqMaxT && static_cast<long long>(a.B) * a.H <= 65535 && al16(a.q) && al16(a.k) &&
           al16(a.v) && al16(a.dO) && (!ch || al16(a.alpha)) && al16(a.workspace) &&
           a.workspace_bytes >= bwd_chunk_workspace_bytes(a.B, a.T, a.H, a.gate);
}

// Two launches that fit on the SMs together run side by side: the second on a stream of the
// library's, between a fork and a join recorded on the caller's stream. That is pass 1a and pass
// 1b of a segmented carry (the plan counts them as one wave), and the forward and reverse carries
// themselves when neither is segmented and their CTAs fit in one wave (the reverse recursion reads
// neither S nor E, only the prep's records). With two waves everything stays in order on the
// caller's stream. One stream and two events per device; the mutex keeps a call's fork and join
// records from interleaving with another thread's.
namespace {
struct CarryAux {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxCarryDevices = 64;
CarryAux g_carry_aux[kMaxCarryDevices];
std::mutex g_carry_aux_mutex[kMaxCarryDevices];
cudaError_t carry_aux(int dev, CarryAux **out) {   // the caller holds g_carry_aux_mutex[dev]
    if (dev < 0 || dev >= kMaxCarryDevices) return cudaErrorInvalidDevice;
    CarryAux &ax = g_carry_aux[dev];
    cudaError_t e;
    if (!ax.s) {
        if ((e = cudaStreamCreateWithFlags(&ax.s, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&ax.fork, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&ax.join, cudaEventDisableTiming)) != cudaSuccess)
            return e;
    }
    *out = &ax;
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_bwd_chunk(const BwdArgs &a) {
    const int nc = (a.T + kC - 1) / kC, chains = a.B * a.H;
    const bool ch = a.gate == KLA_GATE_CHANNEL;
    // per-channel gate: marks of the chains out of the factorised range, then the records
    unsigned *marks = ch ? static_cast<unsigned *>(a.workspace) : nullptr;
    void *rec = ch ? static_cast<char *>(a.workspace) + mark_bytes(a.B, a.H) : a.workspace;
    const Ws ws = carve(rec, static_cast<size_t>(chains) * nc, ch);
    const bf16 *q = static_cast<const bf16 *>(a.q), *k = static_cast<const bf16 *>(a.k),
               *v = static_cast<const bf16 *>(a.v), *dO = static_cast<const bf16 *>(a.dO);
    cudaError_t e;
    unsigned *err = nullptr;
    if ((e = device_error_word(&err)) != cudaSuccess) return e;
    const ChBwd cp{q, k, v, dO, a.alpha, a.eta, a.eps, a.q_scale, a.beta_raw, a.B, a.T, a.H, nc, ws, marks,
                   a.dq, a.dk, a.dv, a.dalpha, a.deta, err};
    if (ch) {
        if ((e = launch_gate_range(a.alpha, a.B, a.T, a.H, marks, a.stream)) != cudaSuccess ||
            (e = launch_bwd_prep_ch(cp, a.stream)) != cudaSuccess)
            return e;
    } else {
        if ((e = cudaFuncSetAttribute(bwd_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GR_BYTES)) ||
            (e = launch_prep_tc(q, k, v, a.alpha, a.eta, a.eps, a.beta_raw, a.B, a.T, a.H, nc, ws, err, a.stream)))
            return e;
    }
    const CarryPlan pl = carry_plan(chains, nc);
    const size_t part = static_cast<size_t>(chains) * pl.nseg * kD * kD;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const bool side_by_side = pl.nseg <= 1 && 2L * chains <= sms && ws.dE != ws.UdE;
    if (side_by_side) {   // both carries in one wave
        ScanParams sf{q, k, dO, a.S0, nullptr, a.q_scale, a.B, a.T, a.H, nc, ws,
                      pl.seg_len, 0, 1, pl.nseg, kX0Chain, 1, 1, nullptr, nullptr, marks, err};
        ScanParams sr = sf;
        sr.X0 = a.dS_T;
        sr.X_end = a.dS0;
        std::lock_guard<std::mutex> lock(g_carry_aux_mutex[dev]);
        CarryAux *ax = nullptr;
        if ((e = carry_aux(dev, &ax)) != cudaSuccess || (e = cudaEventRecord(ax->fork, a.stream)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(ax->s, ax->fork, 0)) != cudaSuccess)
            return e;
        if ((e = launch_carry_tc(sr, true, ch, chains, a.stream)) != cudaSuccess ||
            (e = launch_carry_tc(sf, false, ch, chains, ax->s)) != cudaSuccess)
            return e;
        if ((e = cudaEventRecord(ax->join, ax->s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(a.stream, ax->join, 0)) != cudaSuccess)
            return e;
    }
    for (int rev = 0; rev < 2 && !side_by_side; ++rev) {
        auto kern = [&](const ScanParams &sp, int grid, cudaStream_t st) {
            return launch_carry_tc(sp, rev != 0, ch, grid, st);
        };
        ScanParams sp{q, k, dO, rev ? a.dS_T : a.S0, rev ? a.dS0 : nullptr, a.q_scale, a.B, a.T, a.H, nc, ws,
                      pl.seg_len, 0, 1, pl.nseg, kX0Chain, 1, 1, nullptr, nullptr, marks, err};
        if (pl.nseg <= 1) {
            if ((e = kern(sp, chains, a.stream)) != cudaSuccess) return e;
            continue;
        }
        float *Z = ws.seg, *M = Z + part, *Sst = M + part;
        // pass 1a: segments 0..n-2 (in processing order) from the chain's start (segment 0, the
        // true run: records kept) or from zero; their end states Z
        ScanParams p1 = sp;
        p1.seg_count = pl.nseg - 1;
        p1.records = 2;
        p1.Xseg = Z;
        p1.X_end = nullptr;
        // pass 1b: transitions M of segments 1..n-2 (from the identity, linear part only); it
        // writes only M and reads only the prep's records, so it may run beside pass 1a
        ScanParams p2 = sp;
        p2.seg_begin = 1;
        p2.seg_count = pl.nseg - 2;
        p2.x0_mode = kX0Identity;
        p2.drive = 0;
        p2.records = 0;
        p2.Xseg = M;
        p2.X_end = nullptr;
        const bool one_wave = static_cast<long>(chains) * (p1.seg_count + p2.seg_count) <= sms;
        if (pl.nseg <= 2 || !one_wave) {
            if ((e = kern(p1, chains * p1.seg_count, a.stream)) != cudaSuccess) return e;
            if (pl.nseg > 2 && (e = kern(p2, chains * p2.seg_count, a.stream)) != cudaSuccess) return e;
        } else {
            std::lock_guard<std::mutex> lock(g_carry_aux_mutex[dev]);
            CarryAux *ax = nullptr;
            if ((e = carry_aux(dev, &ax)) != cudaSuccess || (e = cudaEventRecord(ax->fork, a.stream)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(ax->s, ax->fork, 0)) != cudaSuccess)
                return e;
            if ((e = kern(p1, chains * p1.seg_count, a.stream)) != cudaSuccess ||
                (e = kern(p2, chains * p2.seg_count, ax->s)) != cudaSuccess)
                return e;
            if ((e = cudaEventRecord(ax->join, ax->s)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(a.stream, ax->join, 0)) != cudaSuccess)
                return e;
        }
        // pass 2: true start states of segments 1..n-1; pass 3: rerun them with records
        if ((e = launch_seg_combine(Z, M, Sst, chains, pl.nseg, a.stream)) != cudaSuccess) return e;
        ScanParams p3 = sp;
        p3.seg_begin = 1;
        p3.seg_count = pl.nseg - 1;
        p3.x0_mode = kX0Given;
        p3.Xst = Sst;
        if ((e = kern(p3, chains * p3.seg_count, a.stream)) != cudaSuccess) return e;
    }
    if (ch) {
        // the chunkwise gradients, then the marked chains again on the exact token-sequential path,
        // its checkpoints over the records (every kernel that reads them has run by then)
        if ((e = launch_bwd_grad_ch(cp, a.stream)) != cudaSuccess) return e;
        BwdArgs r = a;
        r.workspace = rec;
        r.workspace_bytes = a.workspace_bytes - mark_bytes(a.B, a.H);
        return launch_bwd_seq(r, marks);
    }
    GradParams gp{q, k, v, dO, a.alpha, a.q_scale, a.beta_raw, a.dq, a.dk, a.dv, a.dalpha, a.deta, a.B, a.T, a.H, nc, ws};
    bwd_grad_kernel<<<dim3(nc, chains), kGradThreads, GR_BYTES, a.stream>>>(gp);
    return cudaGetLastError();
}

}  // namespace kla
