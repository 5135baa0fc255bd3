// kla_bwd_chunk_ch.cu -- chunkwise backward pass with the per-key-channel (KDA) gate: bf16
// q/k/v/dO, d_k = d_v = 128, chunk C = 64, fp32 gradients. The two chunk-state carries are the
// scalar path's (kla_bwd_chunk.cu, chunk_scan_kernel<., true>); this file holds the per-chunk
// prep and gradient kernels.
//
// The pages give no backward algebra (GeekNews, "Revisando las variantes de atencion lineal de la
// familia DeltaNet", section "KDA por chunks", names training as the use of the chunk mode). This
// differentiates the chunk form of the forward with a decay per key channel (same page, sections
// "Kimi Delta Attention" and "KDA por chunks"). Per chunk, with S the state entering it and G the
// in-chunk inclusive log-decay prefix per (token, channel), every in-chunk decay is factorised
// around the chunk's token r = 31, as in the forward's tensor-core kernel:
//   K_r = K e^{G - G_r},  Q_r = Q e^{G - G_r},  K_m = K e^{G_r - G}      (e^{G_i - G_j} = K_r K_m^T's factor)
//   K_g = K e^{G},  Q_g = Q e^{G},  K_e = K e^{G_end - G},  Gamma = diag(e^{G_end})
//   forward:  P = K_r K_m^T, R = strict_lower(diag(beta) P), T = (I + R)^{-1},
//             W = T diag(beta) K_g, U = T diag(beta) V, E = U - W S,
//             O = s (Q_g S + A E), A = lower(Q_r K_m^T),  S' = Gamma S + K_e^T E.
//   reverse, with dS' = dL/dS' arriving from the next chunk:
//             dE  = K_e dS' + s A^T dO,  dS = Gamma dS' + s Q_g^T dO - W^T dE      (the carry)
//             dQg = s dO S^T, dKe = E dS'^T, dGam_c = <S_c., dS'_c.>,  dW = -dE S^T
//             dXK = T^T dW, dXV = T^T dE,  dT = (dW K_g^T + dE V^T) diag(beta)
//             dR  = -strict_lower(T^T dT T^T),  dA = s lower(dO E^T),  dP = diag(beta) dR
//             dKr = dP K_m,  dQr = dA K_m,  dKm = dP^T K_r + dA^T Q_r
//             dq  = dQg e^{G} + dQr e^{G - G_r}
//             dk  = beta dXK e^{G} + dKe e^{G_end - G} + dKr e^{G - G_r} + dKm e^{G_r - G} - 2 beta dbeta / den k
//             dv  = beta dXV,  dbeta_i = K_g,i . dXK_i + V_i . dXV_i + sum_j dR_ij P_ij,  deta = dbeta / den
//             dG  = dQg Q_g + beta dXK K_g - dKe K_e + dKr K_r + dQr Q_r - dKm K_m   (elementwise),
//                   the last row adding sum_i dKe K_e + Gamma dGam (the end decay),
//             d log alpha_t = sum over the chunk's rows i >= t of dG_i (per channel), dalpha = that / alpha.
// In exact arithmetic the terms of dG that come from A and R cancel in pairs inside the reverse
// prefix (a pair (i, j) contributes to tokens j < t <= i only). The kernel multiplies each such term
// by the same bf16 tile the matching product read (K_r, K_m, Q_r as rounded), so the pairs still
// cancel up to fp32 summation order: with fp32 factors instead, bf16 rounding of the two sides left
// d alpha ~1.3e-2 off under strong decay, against ~4e-3 this way (fp64 model of the kernel).
//
// Range: the factors e^{G_i - G_r} (i < r) and e^{G_r - G_j} (j > r) grow as the gates shrink. The
// forward's range check (a half-chunk product of gates below ~e^-78 marks the chain) applies
// unchanged; marked chains skip these kernels and take the token-sequential fp32 backward.
#include "kla_bwd_chunk.cuh"

namespace kla {
namespace bwdc {
namespace {

// Log-gate prefix over the 32 tokens [32 hf, 32 hf + 32) of the chunk for key channel c; tokens at
// or past L count as alpha = 1. lg receives the 32 clamped log-gates; returns their sum.
__device__ __forceinline__ float gate_logs(const float *alpha, size_t tok0, int H, int L, int c, int hf,
                                           float (&lg)[32]) {
    float sum = 0.f;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
        const int t = 32 * hf + u;
        const float a = t < L ? alpha[(tok0 + static_cast<size_t>(t) * H) * kD + c] : 1.f;
        lg[u] = fmaxf(logf(a), kMinLogGate);
        sum += lg[u];
    }
    return sum;
}

// ============================================================== prep: per-chunk operands
constexpr int kPrepThreads = 256;
constexpr int PC_K = 0;                               // K, then K_r in place
constexpr int PC_Q = PC_K + kTileTok;                 // Q, then Q_r in place; W staging at the end
constexpr int PC_V = PC_Q + kTileTok;                 // V
constexpr int PC_KM = PC_V + kTileTok;                // K_m; U staging at the end
constexpr int PC_R = PC_KM + kTileTok;                // fp32 [64][kPR]: R, then T in place
constexpr int PC_TB = PC_R + kC * kPR * 4;            // bf16 T diag(beta)
constexpr int PC_A = PC_TB + kTileSq;                 // bf16 A, then T, staging
constexpr int PC_X = PC_A + kTileSq;                  // fp32 [32][kPX] merge scratch
constexpr int PC_VEC = PC_X + 32 * kPX * 4;           // eta, beta [64]; half sums [2][128]; e^{G_r} [128]
constexpr int PC_BYTES = PC_VEC + (2 * kC + 3 * kD) * 4;
static_assert(2 * (PC_BYTES + 1024) <= 233472, "two prep CTAs per SM");

__global__ void __launch_bounds__(kPrepThreads, 2) bwd_prep_ch_kernel(ChBwd p) {
    extern __shared__ __align__(16) unsigned char smem[];
    bf16 *sK = reinterpret_cast<bf16 *>(smem + PC_K), *sQ = reinterpret_cast<bf16 *>(smem + PC_Q),
         *sV = reinterpret_cast<bf16 *>(smem + PC_V), *sKM = reinterpret_cast<bf16 *>(smem + PC_KM);
    float(*sR)[kPR] = reinterpret_cast<float(*)[kPR]>(smem + PC_R);
    bf16 *sTB = reinterpret_cast<bf16 *>(smem + PC_TB), *sA = reinterpret_cast<bf16 *>(smem + PC_A);
    float *sX = reinterpret_cast<float *>(smem + PC_X);
    float *seta = reinterpret_cast<float *>(smem + PC_VEC), *sb = seta + kC, *shalf = sb + kC, *segr = shalf + 2 * kD;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
    if (p.skip && p.skip[bh]) return;
    const size_t rs = static_cast<size_t>(p.H) * kD;
    const int t0 = c * kC, L = min(kC, p.T - t0);
    const size_t n = static_cast<size_t>(bh) * p.nc + c;
    const size_t tok0 = (static_cast<size_t>(b) * p.T + t0) * p.H + h;

    load_tok(sK, p.k + tok0 * kD, rs, L, tid, kPrepThreads);
    load_tok(sQ, p.q + tok0 * kD, rs, L, tid, kPrepThreads);
    load_tok(sV, p.v + tok0 * kD, rs, L, tid, kPrepThreads);
    cp_commit();
    // log-gates while the tiles land: thread (channel ch, half hf)
    const int ch = tid & (kD - 1), hf = tid >> 7;
    float lg[32];
    shalf[hf * kD + ch] = gate_logs(p.alpha, tok0, p.H, L, ch, hf, lg);
    if (tid < kC) seta[tid] = tid < L ? p.eta[tok0 + static_cast<size_t>(tid) * p.H] : 0.f;
    cp_wait<0>();
    __syncthreads();

    // ||k||^2, beta and the cg record: warp w takes tokens 8 w .. 8 w + 7, a lane 4 channels
    float *cg = p.ws.cg + n * kCgFloats;
    for (int u = 0; u < 8; ++u) {
        const int i = 8 * warp + u;
        const uint2 x = *reinterpret_cast<const uint2 *>(sK + i * kP + 4 * lane);
        const float2 a = unpack2(x.x), bb = unpack2(x.y);
        float n2 = fmaf(a.x, a.x, fmaf(a.y, a.y, fmaf(bb.x, bb.x, bb.y * bb.y)));
#pragma unroll
        for (int o = 16; o; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
        if (lane == 0) {
            const float beta = i < L ? kla_beta(seta[i], n2, p.eps, p.beta_raw) : 0.f;
            sb[i] = beta;
            cg[i] = 0.f;
            cg[kC + i] = beta;
            cg[2 * kC + i] = n2 + p.eps;
        }
    }
    __syncthreads();   // every read of the raw K is done; the half sums are visible

    // factor tiles, in place: K_r, Q_r (over K, Q) and K_m; the records K_e, s Q_g and e^{G_end}
    {
        const float Gr = shalf[ch], Gend = Gr + shalf[kD + ch];
        float G = hf ? Gr : 0.f;
        bf16 *ke = p.ws.Ke + n * kC * kD, *qg = p.ws.Qg + n * kC * kD;
        if (hf == 0) segr[ch] = __expf(Gr);
        else p.ws.gend[n * kD + ch] = __expf(Gend);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int i = 32 * hf + u;
            G += lg[u];
            const float fr = __expf(G - Gr), fm = __expf(Gr - G), eg = __expf(G), ee = __expf(Gend - G);
            const float kv = __bfloat162float(sK[i * kP + ch]), qv = __bfloat162float(sQ[i * kP + ch]);
            sK[i * kP + ch] = __float2bfloat16_rn(kv * fr);
            sQ[i * kP + ch] = __float2bfloat16_rn(qv * fr);
            sKM[i * kP + ch] = __float2bfloat16_rn(kv * fm);
            ke[i * kD + ch] = __float2bfloat16_rn(kv * ee);
            qg[i * kD + ch] = __float2bfloat16_rn(p.q_scale * qv * eg);
        }
    }
    __syncthreads();

    // [K_r; Q_r] K_m^T: warp w owns rows 16 (w & 3) of P (w < 4: R = beta P, strictly lower) or of
    // Q_r K_m^T (w >= 4: A, lower)
    {
        float acc[8][4];
        zero(acc);
        const int r0 = 16 * (warp & 3);
        gemm<8, 8, false, false>(acc, sptr(warp < 4 ? sK : sQ), kP, r0, 0, sptr(sKM), kP, 0, 0, lane);
        const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = r0 + g + 8 * hh, j = 8 * nt + 2 * q4;
                if (warp < 4) {
                    const float bi = sb[i];
                    sR[i][j] = j < i ? bi * acc[nt][2 * hh] : 0.f;
                    sR[i][j + 1] = j + 1 < i ? bi * acc[nt][2 * hh + 1] : 0.f;
                } else {
                    st_pair(sA, kPs, i, j, j <= i ? acc[nt][2 * hh] : 0.f, j + 1 <= i ? acc[nt][2 * hh + 1] : 0.f);
                }
            }
    }
    __syncthreads();
    store_dense<kC>(p.ws.A + n * kC * kC, sA, kC, tid, kPrepThreads);

    unit_lower_inverse64(sR, sX, warp, lane);
    // T diag(beta) and T as bf16 (the upper triangle is zero)
    for (int e = tid; e < kC * kC / 2; e += kPrepThreads) {
        const int i = e / (kC / 2), j = 2 * (e % (kC / 2));
        const float t0v = j <= i ? sR[i][j] : 0.f, t1v = j + 1 <= i ? sR[i][j + 1] : 0.f;
        st_pair(sTB, kPs, i, j, t0v * sb[j], t1v * sb[j + 1]);
        st_pair(sA, kPs, i, j, t0v, t1v);
    }
    __syncthreads();
    store_dense<kC>(p.ws.Tm + n * kC * kC, sA, kC, tid, kPrepThreads);
    // W = (T diag(beta) K_r) diag(e^{G_r}) (warps 0-3) and U = T diag(beta) V (warps 4-7)
    float acc[16][4];
    zero(acc);
    const int r0 = 16 * (warp & 3);
    gemm<16, 4, false, true>(acc, sptr(sTB), kPs, r0, 0, sptr(warp < 4 ? sK : sV), kP, 0, 0, lane);
    __syncthreads();   // every read of K_r, V is done: stage W in Q_r's tile and U in K_m's
    {
        bf16 *st = warp < 4 ? sQ : sKM;
        const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int col = 8 * nt + 2 * q4;
            const float f0 = warp < 4 ? segr[col] : 1.f, f1 = warp < 4 ? segr[col + 1] : 1.f;
            st_pair(st, kP, r0 + g, col, f0 * acc[nt][0], f1 * acc[nt][1]);
            st_pair(st, kP, r0 + g + 8, col, f0 * acc[nt][2], f1 * acc[nt][3]);
        }
    }
    __syncthreads();
    store_dense<kD>(p.ws.W + n * kC * kD, sQ, kC, tid, kPrepThreads);
    store_dense<kD>(p.ws.UdE + n * kC * kD, sKM, kC, tid, kPrepThreads);
}

// gemm_m with the k-steps unrolled by two only: with 255 registers a thread, full unrolling lets the
// compiler load every step's fragments ahead of the MMAs and spill the accumulators.
template <int MT, int NT, int KS, bool kAT, bool kBT>
__device__ __forceinline__ void gemm_k2(float (&acc)[MT][NT][4], uint32_t ta, int pa, int r0, int ka, uint32_t tb,
                                        int pb, int n0, int kb, int lane) {
#pragma unroll 2
    for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[MT][4];
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) {
            if (kAT) frag_a_kr(ta, pa, r0 + 16 * mi, ka + 16 * ks, lane, a[mi]);
            else frag_a_rk(ta, pa, r0 + 16 * mi, ka + 16 * ks, lane, a[mi]);
        }
#pragma unroll
        for (int j = 0; j < NT / 2; ++j) {
            uint32_t b[4];
            if (kBT) frag_b_kr(tb, pb, n0 + 16 * j, kb + 16 * ks, lane, b);
            else frag_b_rk(tb, pb, n0 + 16 * j, kb + 16 * ks, lane, b);
#pragma unroll
            for (int mi = 0; mi < MT; ++mi) {
                mma(acc[mi][2 * j], a[mi], b[0], b[1]);
                mma(acc[mi][2 * j + 1], a[mi], b[2], b[3]);
            }
        }
    }
}

// ============================================================== gradients of a chunk
// One CTA of 8 warps per chunk. Warp w owns the 32 x 32 block (rows 32 (w & 1), columns
// 32 (w >> 1)) of every 64 x 128 quantity and keeps dk, dq and dG for it in registers, so every
// elementwise step is local; 64 x 64 products give a warp 16 x 32 (rows 16 (w & 3), columns
// 32 (w >> 2)). Phases (block barriers between them):
//   1  <S, dS'> per channel; dKe = E dS'^T; dQg = s dO S^T; dW = -dE S^T; dA = s lower(dO E^T)
//   1b dW and dA stored; the bf16 factor tiles K_g, K_r, K_m, Q_r built over S, dS' and E
//   2  dXK = T^T dW; dXV = T^T dE -> dv; dT
//   3  Y = T^T dT; P = K_r K_m^T, dR and dP = beta dR; dQr = dA K_m -> dq
//   4  dKr = dP K_m; dKm = dP^T K_r + dA^T Q_r; then per token dbeta, deta, the k coefficient,
//      dk, and the reverse prefix of dG per channel -> dalpha.
constexpr int kGradThreads = 256;
constexpr int kPG = kD + 8;                                   // pitch (floats) of the fp32 64 x 128 tiles
constexpr int GC_S = 0;                                       // S; then dW | K_g; then dG (fp32)
constexpr int GC_DS = GC_S + kTileSt;                         // dS'; then K_r | K_m
constexpr int GC_E = GC_DS + kTileSt;                         // E; then Q_r
constexpr int GC_DO = GC_E + kTileTok;                        // dO; then dA
constexpr int GC_Q = GC_DO + kTileTok;                        // Q; then dT
constexpr int GC_K = GC_Q + kTileTok;                         // K
constexpr int GC_V = GC_K + kTileTok;                         // V; then Y
constexpr int GC_DE = GC_V + kTileTok;                        // dE; then dP
constexpr int GC_T = GC_DE + kTileTok;                        // T
constexpr int GC_G = GC_T + kTileSq;                          // fp32 [64][kPG] G
constexpr int GC_CG = GC_G + kC * kPG * 4;                    // cg record: (G), beta, den
constexpr int GC_GR = GC_CG + static_cast<int>(kCgFloats) * 4;   // fp32 [128] G_r
constexpr int GC_GE = GC_GR + kD * 4;                         // fp32 [128] G_end
constexpr int GC_DGAM = GC_GE + kD * 4;                       // fp32 [128] <S, dS'> per channel
constexpr int GC_COLK = GC_DGAM + kD * 4;                     // fp32 [2][128] column sums of dKe K_e
constexpr int GC_RROW = GC_COLK + 2 * kD * 4;                 // fp32 [3][4][64] row partials
constexpr int GC_KC = GC_RROW + 3 * 4 * kC * 4;               // fp32 [64] k coefficient
constexpr int GC_HALF = GC_KC + kC * 4;                       // fp32 [2][128] half sums of the gates / of dG
constexpr int GC_BYTES = GC_HALF + 2 * kD * 4;
static_assert(kC * kPG * 4 == kTileSt, "dG tile over S");
static_assert(GC_BYTES <= 232448, "gradient kernel shared memory");
enum { RB_XK = 0, RB_XV, RB_R };   // row partials: K_g . dXK, V . dXV, dR . P

__global__ void __launch_bounds__(kGradThreads, 1) bwd_grad_ch_kernel(ChBwd p) {
    extern __shared__ __align__(16) unsigned char smem[];
    auto tile = [&](int off) { return reinterpret_cast<bf16 *>(smem + off); };
    bf16 *sS = tile(GC_S), *sDS = tile(GC_DS), *sE = tile(GC_E), *sDO = tile(GC_DO), *sQ = tile(GC_Q),
         *sK = tile(GC_K), *sV = tile(GC_V), *sDE = tile(GC_DE), *sT = tile(GC_T);
    bf16 *sDW = sS, *sKG = tile(GC_S + kTileTok), *sKR = sDS, *sKM = tile(GC_DS + kTileTok), *sQR = sE,
         *sDA = sDO, *sDT = sQ, *sY = sV, *sDP = sDE;
    float *sG = reinterpret_cast<float *>(smem + GC_G), *sDG = reinterpret_cast<float *>(smem + GC_S);
    const float *cg = reinterpret_cast<const float *>(smem + GC_CG);
    float *sGr = reinterpret_cast<float *>(smem + GC_GR), *sGe = reinterpret_cast<float *>(smem + GC_GE),
          *sDGam = reinterpret_cast<float *>(smem + GC_DGAM), *sColK = reinterpret_cast<float *>(smem + GC_COLK),
          *kcoef = reinterpret_cast<float *>(smem + GC_KC), *shalf = reinterpret_cast<float *>(smem + GC_HALF);
    float(*rrow)[4][kC] = reinterpret_cast<float(*)[4][kC]>(smem + GC_RROW);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, q4 = lane & 3;
    const int c = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
    if (p.skip && p.skip[bh]) return;
    const int t0 = c * kC, L = min(kC, p.T - t0);
    const size_t n = static_cast<size_t>(bh) * p.nc + c;
    const size_t rs = static_cast<size_t>(p.H) * kD;
    const size_t tok0 = (static_cast<size_t>(b) * p.T + t0) * p.H + h;
    const float s = p.q_scale;

    load_tok(sQ, p.q + tok0 * kD, rs, L, tid, kGradThreads);
    load_tok(sK, p.k + tok0 * kD, rs, L, tid, kGradThreads);
    load_tok(sV, p.v + tok0 * kD, rs, L, tid, kGradThreads);
    load_tok(sDO, p.dO + tok0 * kD, rs, L, tid, kGradThreads);
    load_dense<kD>(sE, p.ws.E + n * kC * kD, kC, tid, kGradThreads);
    load_dense<kD>(sDE, p.ws.UdE + n * kC * kD, kC, tid, kGradThreads);
    load_dense<kD>(sS, p.ws.S + n * kD * kD, kD, tid, kGradThreads);
    load_dense<kD>(sDS, p.ws.dS + n * kD * kD, kD, tid, kGradThreads);
    load_dense<kC>(sT, p.ws.Tm + n * kC * kC, kC, tid, kGradThreads);
    if (tid < static_cast<int>(kCgFloats) / 4)
        cp16(smem + GC_CG + 16 * tid, p.ws.cg + n * kCgFloats + 4 * tid, true);
    cp_commit();
    // G per (token, channel) while the tiles land, in the prep kernel's order of summation
    {
        const int ch = tid & (kD - 1), hf = tid >> 7;
        float lg[32];
        shalf[hf * kD + ch] = gate_logs(p.alpha, tok0, p.H, L, ch, hf, lg);
        __syncthreads();
        const float Gr = shalf[ch];
        float G = hf ? Gr : 0.f;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            G += lg[u];
            sG[(32 * hf + u) * kPG + ch] = G;
        }
        if (hf == 0) sGr[ch] = Gr;
        else sGe[ch] = G;
    }
    cp_wait<0>();
    __syncthreads();

    const int r1 = 32 * (warp & 1), c1 = 32 * (warp >> 1), cb1 = warp >> 1;   // 64 x 128: 32 x 32 per warp
    const int r2 = 16 * (warp & 3), c2 = 32 * (warp >> 2), cb2 = warp >> 2;   // 64 x 64: 16 x 32 per warp
    auto row1 = [&](int mi, int hh) { return r1 + 16 * mi + g + 8 * hh; };
    auto col1 = [&](int ni) { return c1 + 8 * ni + 2 * q4; };
    auto row2 = [&](int hh) { return r2 + g + 8 * hh; };
    auto gpair = [&](int r, int col) { return *reinterpret_cast<const float2 *>(sG + r * kPG + col); };
    auto put_row = [&](int qi, int cb, int row, float x) {   // sum over the 4 lanes of a row
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        if (q4 == 0) rrow[qi][cb][row] = x;
    };

    float dk[2][4][4], dg[2][4][4], tmp[2][4][4];
    float da[1][4][4];
    // ---- phase 1
    {   // <S, dS'> per key channel (row of S): two threads per row
        const int r = tid >> 1, h0 = (tid & 1) * 64;
        float sum = 0.f;
#pragma unroll
        for (int cc = 0; cc < 64; cc += 8) {
            const uint4 x = *reinterpret_cast<const uint4 *>(sS + r * kP + h0 + cc);
            const uint4 y = *reinterpret_cast<const uint4 *>(sDS + r * kP + h0 + cc);
            const uint32_t *xw = reinterpret_cast<const uint32_t *>(&x), *yw = reinterpret_cast<const uint32_t *>(&y);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 u = unpack2(xw[e]), w = unpack2(yw[e]);
                sum = fmaf(u.x, w.x, fmaf(u.y, w.y, sum));
            }
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        if ((tid & 1) == 0) sDGam[r] = sum;
    }
    // dKe = E dS'^T: dk = dKe e^{G_end - G}, dG = -dKe K_e, column sums of dKe K_e for the last row
    zero(dk[0]);
    zero(dk[1]);
    gemm_k2<2, 4, 8, false, false>(dk, sptr(sE), kP, r1, 0, sptr(sDS), kP, c1, 0, lane);
    {
        float colk[4][2] = {};
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int col = col1(ni);
            const float ge0 = sGe[col], ge1 = sGe[col + 1];
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = row1(mi, hh);
                    const float2 G2 = gpair(r, col), k2 = ld_pair(sK, kP, r, col);
                    const float e0 = __expf(ge0 - G2.x), e1 = __expf(ge1 - G2.y);
                    const float x0 = dk[mi][ni][2 * hh] * e0, x1 = dk[mi][ni][2 * hh + 1] * e1;   // dk terms
                    const float m0 = x0 * k2.x, m1 = x1 * k2.y;                                  // dKe . K_e
                    dg[mi][ni][2 * hh] = -m0;
                    dg[mi][ni][2 * hh + 1] = -m1;
                    colk[ni][0] += m0;
                    colk[ni][1] += m1;
                    dk[mi][ni][2 * hh] = x0;
                    dk[mi][ni][2 * hh + 1] = x1;
                }
        }
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float y = colk[ni][e];
                y += __shfl_xor_sync(0xffffffffu, y, 4);
                y += __shfl_xor_sync(0xffffffffu, y, 8);
                y += __shfl_xor_sync(0xffffffffu, y, 16);
                if (g == 0) sColK[(warp & 1) * kD + col1(ni) + e] = y;
            }
    }
    // dQg = s dO S^T: dq = dQg e^{G} (written out now; the same thread adds the dQr term in phase 3),
    // dG += dQg Q_g
    zero(tmp[0]);
    zero(tmp[1]);
    gemm_k2<2, 4, 8, false, false>(tmp, sptr(sDO), kP, r1, 0, sptr(sS), kP, c1, 0, lane);
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = row1(mi, hh);
            float *dst = p.dq + (tok0 + static_cast<size_t>(r) * p.H) * kD;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int col = col1(ni);
                const float2 G2 = gpair(r, col), q2 = ld_pair(sQ, kP, r, col);
                const float e0 = s * __expf(G2.x), e1 = s * __expf(G2.y);
                const float x0 = tmp[mi][ni][2 * hh] * e0, x1 = tmp[mi][ni][2 * hh + 1] * e1;
                dg[mi][ni][2 * hh] = fmaf(x0, q2.x, dg[mi][ni][2 * hh]);
                dg[mi][ni][2 * hh + 1] = fmaf(x1, q2.y, dg[mi][ni][2 * hh + 1]);
                if (r < L) *reinterpret_cast<float2 *>(dst + col) = make_float2(x0, x1);
            }
        }
    // dW = -dE S^T (stored after the barrier, over S)
    zero(tmp[0]);
    zero(tmp[1]);
    gemm_k2<2, 4, 8, false, false>(tmp, sptr(sDE), kP, r1, 0, sptr(sS), kP, c1, 0, lane);
    // dA = s lower(dO E^T) (stored after the barrier, over dO)
    zero(da[0]);
    gemm_k2<1, 4, 8, false, false>(da, sptr(sDO), kP, r2, 0, sptr(sE), kP, c2, 0, lane);
    __syncthreads();   // every read of S, dS', E and dO is done

    // ---- phase 1b: dW, dA; the factor tiles
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int ni = 0; ni < 4; ++ni)
                st_pair(sDW, kP, row1(mi, hh), col1(ni), -tmp[mi][ni][2 * hh], -tmp[mi][ni][2 * hh + 1]);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int i = row2(hh);
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int j = c2 + 8 * ni + 2 * q4;
            st_pair(sDA, kPs, i, j, j <= i ? s * da[0][ni][2 * hh] : 0.f, j + 1 <= i ? s * da[0][ni][2 * hh + 1] : 0.f);
        }
    }
    for (int e = tid; e < kC * kD / 8; e += kGradThreads) {   // 8 consecutive channels of one token
        const int r = e >> 4, cc = (e & 15) * 8;
        const uint4 kx = *reinterpret_cast<const uint4 *>(sK + r * kP + cc);
        const uint4 qx = *reinterpret_cast<const uint4 *>(sQ + r * kP + cc);
        const uint32_t *kw = reinterpret_cast<const uint32_t *>(&kx), *qw = reinterpret_cast<const uint32_t *>(&qx);
        uint4 og, orr, om, oq;
        uint32_t *pg = reinterpret_cast<uint32_t *>(&og), *pr = reinterpret_cast<uint32_t *>(&orr),
                 *pm = reinterpret_cast<uint32_t *>(&om), *pq = reinterpret_cast<uint32_t *>(&oq);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int col = cc + 2 * u;
            const float2 G2 = gpair(r, col), k2 = unpack2(kw[u]), q2 = unpack2(qw[u]);
            const float gr0 = sGr[col], gr1 = sGr[col + 1];
            const float fr0 = __expf(G2.x - gr0), fr1 = __expf(G2.y - gr1);
            const float fm0 = __expf(gr0 - G2.x), fm1 = __expf(gr1 - G2.y);
            pg[u] = pack2(k2.x * __expf(G2.x), k2.y * __expf(G2.y));
            pr[u] = pack2(k2.x * fr0, k2.y * fr1);
            pm[u] = pack2(k2.x * fm0, k2.y * fm1);
            pq[u] = pack2(q2.x * fr0, q2.y * fr1);
        }
        *reinterpret_cast<uint4 *>(sKG + r * kP + cc) = og;
        *reinterpret_cast<uint4 *>(sKR + r * kP + cc) = orr;
        *reinterpret_cast<uint4 *>(sKM + r * kP + cc) = om;
        *reinterpret_cast<uint4 *>(sQR + r * kP + cc) = oq;
    }
    __syncthreads();

    // ---- phase 2: dXK = T^T dW -> dk, dG, dbeta part;  dXV = T^T dE -> dv, dbeta part;  dT;  P
    zero(tmp[0]);
    zero(tmp[1]);
    gemm_k2<2, 4, 4, true, true>(tmp, sptr(sT), kPs, r1, 0, sptr(sDW), kP, c1, 0, lane);
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = row1(mi, hh);
            const float bt = cg[kC + r];
            float rsum = 0.f;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int col = col1(ni);
                const float2 G2 = gpair(r, col), k2 = ld_pair(sK, kP, r, col);
                const float eg0 = __expf(G2.x), eg1 = __expf(G2.y);
                const float kg0 = k2.x * eg0, kg1 = k2.y * eg1;   // K_g
                const float x0 = tmp[mi][ni][2 * hh], x1 = tmp[mi][ni][2 * hh + 1];
                rsum = fmaf(x0, kg0, fmaf(x1, kg1, rsum));
                dg[mi][ni][2 * hh] = fmaf(bt * x0, kg0, dg[mi][ni][2 * hh]);
                dg[mi][ni][2 * hh + 1] = fmaf(bt * x1, kg1, dg[mi][ni][2 * hh + 1]);
                dk[mi][ni][2 * hh] = fmaf(bt * eg0, x0, dk[mi][ni][2 * hh]);
                dk[mi][ni][2 * hh + 1] = fmaf(bt * eg1, x1, dk[mi][ni][2 * hh + 1]);
            }
            put_row(RB_XK, cb1, r, rsum);
        }
    zero(tmp[0]);
    zero(tmp[1]);
    gemm_k2<2, 4, 4, true, true>(tmp, sptr(sT), kPs, r1, 0, sptr(sDE), kP, c1, 0, lane);
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = row1(mi, hh);
            const float bt = cg[kC + r];
            float rsum = 0.f;
            float *dst = p.dv + (tok0 + static_cast<size_t>(r) * p.H) * kD;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int col = col1(ni);
                const float2 v2 = ld_pair(sV, kP, r, col);
                rsum = fmaf(tmp[mi][ni][2 * hh], v2.x, fmaf(tmp[mi][ni][2 * hh + 1], v2.y, rsum));
                if (r < L)
                    *reinterpret_cast<float2 *>(dst + col) =
                        make_float2(bt * tmp[mi][ni][2 * hh], bt * tmp[mi][ni][2 * hh + 1]);
            }
            put_row(RB_XV, cb1, r, rsum);
        }
    {   // dT = (dW K_g^T + dE V^T) diag(beta)  (over Q)
        float a1[1][4][4];
        zero(a1[0]);
        gemm_k2<1, 4, 8, false, false>(a1, sptr(sDW), kP, r2, 0, sptr(sKG), kP, c2, 0, lane);
        gemm_k2<1, 4, 8, false, false>(a1, sptr(sDE), kP, r2, 0, sptr(sV), kP, c2, 0, lane);
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int j = c2 + 8 * ni + 2 * q4;
            const float bj0 = cg[kC + j], bj1 = cg[kC + j + 1];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                st_pair(sDT, kPs, row2(hh), j, bj0 * a1[0][ni][2 * hh], bj1 * a1[0][ni][2 * hh + 1]);
        }
    }
    __syncthreads();   // dT is visible; V and dE are no longer read

    // ---- phase 3: Y = T^T dT (over V);  dR = -strict_lower(Y T^T), dP = beta dR (over dE);  dQr -> dq
    {
        float y[1][4][4];
        zero(y[0]);
        gemm_k2<1, 4, 4, true, true>(y, sptr(sT), kPs, r2, 0, sptr(sDT), kPs, c2, 0, lane);
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                st_pair(sY, kPs, row2(hh), c2 + 8 * ni + 2 * q4, y[0][ni][2 * hh], y[0][ni][2 * hh + 1]);
    }
    __syncthreads();
    {
        float pk[1][4][4];   // P = K_r K_m^T for the dR . P sums
        zero(pk[0]);
        gemm_k2<1, 4, 8, false, false>(pk, sptr(sKR), kP, r2, 0, sptr(sKM), kP, c2, 0, lane);
        float dr[1][4][4];
        zero(dr[0]);
        gemm_k2<1, 4, 4, false, false>(dr, sptr(sY), kPs, r2, 0, sptr(sT), kPs, c2, 0, lane);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int i = row2(hh);
            const float bi = cg[kC + i];
            float rsum = 0.f;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int j = c2 + 8 * ni + 2 * q4;
                const float x0 = j < i ? -dr[0][ni][2 * hh] : 0.f, x1 = j + 1 < i ? -dr[0][ni][2 * hh + 1] : 0.f;
                rsum = fmaf(x0, pk[0][ni][2 * hh], fmaf(x1, pk[0][ni][2 * hh + 1], rsum));
                st_pair(sDP, kPs, i, j, bi * x0, bi * x1);
            }
            put_row(RB_R, cb2, i, rsum);
        }
    }
    // dQr = dA K_m: dq += dQr e^{G - G_r}, dG += dQr Q_r (the bf16 Q_r of dA^T Q_r); dq is complete
    zero(tmp[0]);
    zero(tmp[1]);
    gemm_k2<2, 4, 4, false, true>(tmp, sptr(sDA), kPs, r1, 0, sptr(sKM), kP, c1, 0, lane);
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = row1(mi, hh);
            float *dst = p.dq + (tok0 + static_cast<size_t>(r) * p.H) * kD;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int col = col1(ni);
                const float2 G2 = gpair(r, col), qr = ld_pair(sQR, kP, r, col);
                const float x0 = tmp[mi][ni][2 * hh], x1 = tmp[mi][ni][2 * hh + 1];
                dg[mi][ni][2 * hh] = fmaf(x0, qr.x, dg[mi][ni][2 * hh]);
                dg[mi][ni][2 * hh + 1] = fmaf(x1, qr.y, dg[mi][ni][2 * hh + 1]);
                if (r < L) {
                    const float2 d = *reinterpret_cast<const float2 *>(dst + col);
                    *reinterpret_cast<float2 *>(dst + col) = make_float2(fmaf(x0, __expf(G2.x - sGr[col]), d.x),
                                                                         fmaf(x1, __expf(G2.y - sGr[col + 1]), d.y));
                }
            }
        }
    __syncthreads();   // dP is visible

    // ---- phase 4: dKr = dP K_m -> dk, dG;  dKm = dP^T K_r + dA^T Q_r -> dk, dG
    zero(tmp[0]);
    zero(tmp[1]);
    gemm_k2<2, 4, 4, false, true>(tmp, sptr(sDP), kPs, r1, 0, sptr(sKM), kP, c1, 0, lane);
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int r = row1(mi, hh), col = col1(ni);
                const float2 G2 = gpair(r, col), kr = ld_pair(sKR, kP, r, col);
                const float x0 = tmp[mi][ni][2 * hh], x1 = tmp[mi][ni][2 * hh + 1];
                dg[mi][ni][2 * hh] = fmaf(x0, kr.x, dg[mi][ni][2 * hh]);
                dg[mi][ni][2 * hh + 1] = fmaf(x1, kr.y, dg[mi][ni][2 * hh + 1]);
                dk[mi][ni][2 * hh] = fmaf(x0, __expf(G2.x - sGr[col]), dk[mi][ni][2 * hh]);
                dk[mi][ni][2 * hh + 1] = fmaf(x1, __expf(G2.y - sGr[col + 1]), dk[mi][ni][2 * hh + 1]);
            }
    zero(tmp[0]);
    zero(tmp[1]);
    gemm_k2<2, 4, 4, true, true>(tmp, sptr(sDP), kPs, r1, 0, sptr(sKR), kP, c1, 0, lane);
    gemm_k2<2, 4, 4, true, true>(tmp, sptr(sDA), kPs, r1, 0, sptr(sQR), kP, c1, 0, lane);
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int r = row1(mi, hh), col = col1(ni);
                const float2 G2 = gpair(r, col), km = ld_pair(sKM, kP, r, col);
                const float x0 = tmp[mi][ni][2 * hh], x1 = tmp[mi][ni][2 * hh + 1];
                dg[mi][ni][2 * hh] = fmaf(-x0, km.x, dg[mi][ni][2 * hh]);
                dg[mi][ni][2 * hh + 1] = fmaf(-x1, km.y, dg[mi][ni][2 * hh + 1]);
                dk[mi][ni][2 * hh] = fmaf(x0, __expf(sGr[col] - G2.x), dk[mi][ni][2 * hh]);
                dk[mi][ni][2 * hh + 1] = fmaf(x1, __expf(sGr[col + 1] - G2.y), dk[mi][ni][2 * hh + 1]);
            }
    // dG to shared memory (over dW | K_g, read last in phase 2)
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int ni = 0; ni < 4; ++ni)
                *reinterpret_cast<float2 *>(sDG + row1(mi, hh) * kPG + col1(ni)) =
                    make_float2(dg[mi][ni][2 * hh], dg[mi][ni][2 * hh + 1]);
    __syncthreads();   // dG and every row partial are in shared memory

    // per token (threads 0-63): dbeta, deta, the k coefficient
    if (tid < kC) {
        const int t = tid;
        const float xk = rrow[RB_XK][0][t] + rrow[RB_XK][1][t] + rrow[RB_XK][2][t] + rrow[RB_XK][3][t];
        const float xv = rrow[RB_XV][0][t] + rrow[RB_XV][1][t] + rrow[RB_XV][2][t] + rrow[RB_XV][3][t];
        const float xr = rrow[RB_R][0][t] + rrow[RB_R][1][t];
        const float dbeta = xk + xv + xr, bt = cg[kC + t], den = cg[2 * kC + t];
        float deta = dbeta, kc = 0.f;
        if (!p.beta_raw) {
            const bool flows = den != 0.f;
            deta = flows ? dbeta / den : 0.f;
            kc = flows ? -2.f * bt * dbeta / den : 0.f;
        }
        kcoef[t] = kc;
        if (t < L) p.deta[tok0 + static_cast<size_t>(t) * p.H] = deta;
    }
    // reverse prefix of dG per channel, in two halves of 32 tokens: the half sums first
    const int ch = tid & (kD - 1), hf = tid >> 7;
    {
        float sum = 0.f;
#pragma unroll 8
        for (int u = 0; u < 32; ++u) sum += sDG[(32 * hf + u) * kPG + ch];
        shalf[hf * kD + ch] = sum;
    }
    __syncthreads();   // kcoef and the half sums are visible

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
                const int col = col1(ni);
                const float2 kx = ld_pair(sK, kP, r, col);
                *reinterpret_cast<float2 *>(dst + col) =
                    make_float2(fmaf(kc, kx.x, dk[mi][ni][2 * hh]), fmaf(kc, kx.y, dk[mi][ni][2 * hh + 1]));
            }
        }
    {   // the end decay's terms join the last row: sum_i dKe K_e + Gamma <S, dS'>
        float run = sColK[ch] + sColK[kD + ch] + __expf(sGe[ch]) * sDGam[ch];
        if (hf == 0) run += shalf[kD + ch];
        for (int u = 31; u >= 0; --u) {
            const int t = 32 * hf + u;
            run += sDG[t * kPG + ch];
            if (t < L) {
                const size_t o = (tok0 + static_cast<size_t>(t) * p.H) * kD + ch;
                p.dalpha[o] = run / p.alpha[o];
            }
        }
    }
}

}  // namespace

cudaError_t launch_bwd_prep_ch(const ChBwd &p, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(bwd_prep_ch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PC_BYTES);
    if (e != cudaSuccess) return e;
    bwd_prep_ch_kernel<<<dim3(p.nc, p.B * p.H), kPrepThreads, PC_BYTES, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_grad_ch(const ChBwd &p, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(bwd_grad_ch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GC_BYTES);
    if (e != cudaSuccess) return e;
    bwd_grad_ch_kernel<<<dim3(p.nc, p.B * p.H), kGradThreads, GC_BYTES, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace bwdc
}  // namespace kla
