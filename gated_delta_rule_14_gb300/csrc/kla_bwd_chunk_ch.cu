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
#include "sm103_ptx.cuh"

namespace kla {
namespace bwdc {
namespace {

// Log-gates of key channels 2 cp and 2 cp + 1 over the 16 tokens [16 qt, 16 qt + 16) of the chunk
// (tokens at or past L count as alpha = 1), clamped at kMinLogGate; their sums go to
// squart[qt][2 cp], squart[qt][2 cp + 1] (fp32 [4][128]).
__device__ __forceinline__ void gate_logs(const float *alpha, size_t tok0, int H, int L, int cp, int qt,
                                          float (&lg)[2][16], float *squart) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const int t = 16 * qt + u;
        float2 a = make_float2(1.f, 1.f);
        if (t < L) a = *reinterpret_cast<const float2 *>(alpha + (tok0 + static_cast<size_t>(t) * H) * kD + 2 * cp);
        lg[0][u] = fmaxf(logf(a.x), kMinLogGate);
        lg[1][u] = fmaxf(logf(a.y), kMinLogGate);
        s0 += lg[0][u];
        s1 += lg[1][u];
    }
    *reinterpret_cast<float2 *>(squart + qt * kD + 2 * cp) = make_float2(s0, s1);
}
// After every quarter sum is in squart: the inclusive prefix G at the start of quarter qt (its
// offset), the reference G_r (tokens 0-31) and G_end, for channel c. Every kernel forms them in this
// order of summation.
struct GateRef {
    float off, Gr, Gend;
};
__device__ __forceinline__ GateRef gate_ref(const float *squart, int c, int qt) {
    const float s0 = squart[c], s1 = squart[kD + c], s2 = squart[2 * kD + c], s3 = squart[3 * kD + c];
    GateRef r;
    r.Gr = s0 + s1;
    r.Gend = (r.Gr + s2) + s3;
    r.off = qt == 0 ? 0.f : qt == 1 ? s0 : qt == 2 ? r.Gr : r.Gr + s2;
    return r;
}

// ============================================================== prep: per-chunk operands
// One CTA of 8 warps per chunk, two per SM, on the tensor cores. The q, k, v tiles land by TMA in
// the 128-byte-swizzled layout; threads (channel pair, quarter) rewrite K and Q in place as the
// factor tiles K_r, Q_r and write K_m, storing the K_e, s Q_g and e^{G_end} records on the way; one
// M = 128 product gives P = K_r K_m^T (rows 0-63) and Q_r K_m^T (rows 64-127) in TMEM, whose rows
// become R = beta P (strictly lower, fp32) and A (lower, bf16, stored); T = (I + R)^{-1} in fp32;
// T_V = T diag(beta) enters W_r^T = K_r^T T_V^T and U^T = V^T T_V^T (M = 128 channels), and
// W = W_r diag(e^{G_r}) is one factor per TMEM lane on the way to the records.
namespace pc {
constexpr int kThreads = 256;
constexpr uint32_t kHalf = 8192;                    // 64 rows x 128 bytes
constexpr uint32_t OFF_QK = 0;                      // [K_r half 0 | Q_r half 0 | K_r half 1 | Q_r half 1]; W, U staging
constexpr uint32_t OFF_TV = OFF_QK + kHalf;         // T_V over Q_r half 0 (read by the first product only)
constexpr uint32_t OFF_V = 4 * kHalf;               // V [half][64 t][64 v]
constexpr uint32_t OFF_KM = OFF_V + 2 * kHalf;      // K_m [half][64 t][64 k], K-major
constexpr uint32_t OFF_R = OFF_KM + 2 * kHalf;      // fp32 [64][kPR]: R, then T
constexpr uint32_t OFF_X = OFF_R + kC * kPR * 4;    // solve scratch fp32 [32][kPX]
constexpr uint32_t OFF_VEC = OFF_X + 32 * kPX * 4;  // eta, beta [64]; quarter sums [4][128]; e^{G_r} [128]
constexpr uint32_t OFF_BAR = OFF_VEC + (2 * kC + 5 * kD) * 4;
constexpr uint32_t kBytes = OFF_BAR + 64 + 1024;
static_assert(OFF_R % 16 == 0 && 2 * kBytes <= 232448, "two prep CTAs per SM");
constexpr uint32_t TM_P = 0, TM_W = 0, TM_U = 64, kTmemCols = 128;   // W^T over P once read
constexpr uint32_t kWaitLimit = 100000;                                // x 20 us: ~2 s
}  // namespace pc


__global__ void __launch_bounds__(pc::kThreads, 2)
bwd_prep_ch_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                   const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mW,
                   const __grid_constant__ CUtensorMap mU, const ChBwd p) {
    using namespace pc;
    using namespace ptx;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
    if (p.skip && p.skip[bh]) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    float(*sR)[kPR] = reinterpret_cast<float(*)[kPR]>(smem + OFF_R);
    float *sX = reinterpret_cast<float *>(smem + OFF_X);
    float *seta = reinterpret_cast<float *>(smem + OFF_VEC), *sb = seta + kC, *squart = sb + kC, *segr = squart + 4 * kD;
    const uint32_t bar_full = sbase + OFF_BAR, bar_mma = bar_full + 8;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + 16);
    const int row = 32 * (warp & 3) + lane, half = warp >> 2;   // TMEM lane, column half
    const int t0 = c * kC, L = min(kC, p.T - t0);
    const size_t n = static_cast<size_t>(bh) * p.nc + c;
    const size_t tok0 = (static_cast<size_t>(b) * p.T + t0) * p.H + h;

    if (tid == 0) {
        mbar_init(bar_full, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_full, 6 * kHalf);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            tma_load_4d(sbase + OFF_QK + 2 * kHalf * hh, &mK, bar_full, 64 * hh, h, t0, b);
            tma_load_4d(sbase + OFF_QK + 2 * kHalf * hh + kHalf, &mQ, bar_full, 64 * hh, h, t0, b);
            tma_load_4d(sbase + OFF_V + kHalf * hh, &mV, bar_full, 64 * hh, h, t0, b);
        }
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kTmemCols);
        tmem_relinquish();
    }
    // log-gates while the tiles land: thread (channel pair cp, quarter qt of the chunk)
    const int cp = tid & 63, qt = tid >> 6;
    float lg[2][16];
    gate_logs(p.alpha, tok0, p.H, L, cp, qt, lg, squart);
    if (tid < kC) seta[tid] = tid < L ? p.eta[tok0 + static_cast<size_t>(tid) * p.H] : 0.f;
    bool ok = mbar_wait_bounded(bar_full, 0, kWaitLimit);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t tl = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);

    // ||k||^2 from the raw K tile, beta and the cg record: warp w takes tokens 8 w .. 8 w + 7, a
    // lane 4 channels (4 lane .. 4 lane + 3: k half lane / 16, bytes 8 (lane % 16) of the row)
    float *cg = p.ws.cg + n * kCgFloats;
    for (int u = 0; u < 8; ++u) {
        const int i = 8 * warp + u;
        const uint2 x = *reinterpret_cast<const uint2 *>(smem + OFF_QK + 2 * kHalf * (lane >> 4) +
                                                        sw128_off(i, 8 * (lane & 15)));
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
    __syncthreads();   // every read of the raw K is done; the quarter sums are visible

    // factor tiles, in place: K_r, Q_r (over K, Q) and K_m; the records K_e, s Q_g and e^{G_end}
    {
        const GateRef g0 = gate_ref(squart, 2 * cp, qt), g1 = gate_ref(squart, 2 * cp + 1, qt);
        float G0 = g0.off, G1 = g1.off;
        uint32_t *ke = reinterpret_cast<uint32_t *>(p.ws.Ke + n * kC * kD) + cp;
        uint32_t *qg = reinterpret_cast<uint32_t *>(p.ws.Qg + n * kC * kD) + cp;
        if (qt == 0) *reinterpret_cast<float2 *>(segr + 2 * cp) = make_float2(__expf(g0.Gr), __expf(g1.Gr));
        if (qt == 3)
            *reinterpret_cast<float2 *>(p.ws.gend + n * kD + 2 * cp) = make_float2(__expf(g0.Gend), __expf(g1.Gend));
        const uint32_t cb = 4 * (cp & 31);   // byte column of the channel pair in its 64-channel half
        uint8_t *kt = smem + OFF_QK + 2 * kHalf * (cp >> 5), *qtl = kt + kHalf;
        uint8_t *km = smem + OFF_KM + kHalf * (cp >> 5);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = 16 * qt + u;
            G0 += lg[0][u];
            G1 += lg[1][u];
            const float fr0 = __expf(G0 - g0.Gr), fm0 = __expf(g0.Gr - G0), eg0 = __expf(G0), ee0 = __expf(g0.Gend - G0);
            const float fr1 = __expf(G1 - g1.Gr), fm1 = __expf(g1.Gr - G1), eg1 = __expf(G1), ee1 = __expf(g1.Gend - G1);
            const uint32_t off = sw128_off(i, cb);
            uint32_t *pk = reinterpret_cast<uint32_t *>(kt + off), *pq = reinterpret_cast<uint32_t *>(qtl + off);
            const float2 kv = unpack2(*pk), qv = unpack2(*pq);
            *pk = pack2(kv.x * fr0, kv.y * fr1);
            *pq = pack2(qv.x * fr0, qv.y * fr1);
            *reinterpret_cast<uint32_t *>(km + off) = pack2(kv.x * fm0, kv.y * fm1);
            ke[i * (kD / 2)] = pack2(kv.x * ee0, kv.y * ee1);
            qg[i * (kD / 2)] = pack2(p.q_scale * qv.x * eg0, p.q_scale * qv.y * eg1);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {   // [K_r; Q_r] K_m^T
        tc_fence_after();
        if (__all_sync(0xffffffffu, ok) && elect_one()) {
            const uint64_t da = sw128_desc(sbase + OFF_QK, 16, 1024), db = sw128_desc(sbase + OFF_KM, 16, 1024);
            const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tbase + TM_P, desc_add(da, (s >> 2) * 2 * kHalf + (s & 3) * 32),
                         desc_add(db, (s >> 2) * kHalf + (s & 3) * 32), id, s);
            mma_commit(bar_mma);
        }
        __syncwarp();
    }
    if (!mbar_wait_bounded(bar_mma, 0, kWaitLimit)) ok = false;
    tc_fence_after();
    {   // this thread's half-row: R = beta P (strictly lower) or A (lower, to its record)
        uint32_t xr[32];
        tmem_ld32(tl + TM_P + 32 * half, xr);
        tmem_ld_wait();
        const int i = row & (kC - 1);
        const bool key_row = row < kC;
        const float scale = key_row ? sb[i] : 1.f;
        float v[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int j = 32 * half + jj;
            v[jj] = (key_row ? j < i : j <= i) ? scale * __uint_as_float(xr[jj]) : 0.f;
        }
        if (key_row) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4 *>(&sR[i][32 * half + 4 * q]) =
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
            bf16 *dst = p.ws.A + (n * kC + i) * kC + 32 * half;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4 *>(dst + 8 * q) =
                    make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
        }
    }
    __syncthreads();   // R complete
    unit_lower_inverse64(sR, sX, warp, lane);   // T over R; ends with a block barrier
    {   // T (bf16 record) and T_V = T diag(beta) (bf16, K-major, 128-byte swizzle)
        const int r = tid >> 2, kq = tid & 3;
        bf16 *trec = p.ws.Tm + (n * kC + r) * kC + 16 * kq;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float tv[8], tt[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = 16 * kq + 8 * hh + u;
                tt[u] = j <= r ? sR[r][j] : 0.f;
                tv[u] = tt[u] * sb[j];
            }
            *reinterpret_cast<uint4 *>(trec + 8 * hh) =
                make_uint4(pack_bf16(tt[0], tt[1]), pack_bf16(tt[2], tt[3]), pack_bf16(tt[4], tt[5]),
                           pack_bf16(tt[6], tt[7]));
            st_shared_v4(sbase + OFF_TV + sw128_off(r, 32 * kq + 16 * hh), pack_bf16(tv[0], tv[1]),
                         pack_bf16(tv[2], tv[3]), pack_bf16(tv[4], tv[5]), pack_bf16(tv[6], tv[7]));
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {   // W_r^T = K_r^T T_V^T and U^T = V^T T_V^T (M = 128 channels, N = 64, K = 64)
        tc_fence_after();
        if (elect_one()) {
            const uint32_t id = idesc_bf16(128, 64, 1, 0);
            const uint64_t dk = sw128_desc(sbase + OFF_QK, 2 * kHalf, 1024), dv = sw128_desc(sbase + OFF_V, kHalf, 1024);
            const uint64_t dt = sw128_desc(sbase + OFF_TV, 16, 1024);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tbase + TM_W, desc_add(dk, s * 2048), desc_add(dt, s * 32), id, s);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tbase + TM_U, desc_add(dv, s * 2048), desc_add(dt, s * 32), id, s);
            mma_commit(bar_mma);
        }
        __syncwarp();
    }
    if (!mbar_wait_bounded(bar_mma, 1, kWaitLimit)) ok = false;
    tc_fence_after();
    {   // rows of W^T (times e^{G_r} of the channel) and U^T -> record-layout staging tiles over the q/k area
        const uint32_t cb = (row & 63) * 2, hb = (row >> 6) * kHalf;
        unsigned short *wst = reinterpret_cast<unsigned short *>(smem + OFF_QK + hb);
        unsigned short *ust = reinterpret_cast<unsigned short *>(smem + OFF_QK + 2 * kHalf + hb);
        const float fw = segr[row];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            uint32_t d[32];
            tmem_ld32(tl + (m ? TM_U : TM_W) + 32 * half, d);
            tmem_ld_wait();
            unsigned short *st = m ? ust : wst;
            const float f = m ? 1.f : fw;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) st[sw128_off(32 * half + jj, cb) >> 1] = bf16_bits(f * __uint_as_float(d[jj]));
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        const int y = static_cast<int>(n) * kC;
        tma_store_2d(&mW, sbase + OFF_QK, 0, y);
        tma_store_2d(&mW, sbase + OFF_QK + kHalf, 64, y);
        tma_store_2d(&mU, sbase + OFF_QK + 2 * kHalf, 0, y);
        tma_store_2d(&mU, sbase + OFF_QK + 3 * kHalf, 64, y);
        tma_store_commit();
        tma_store_wait_all();
        if (!ok && p.err) atomicOr(p.err, kErrTimeout);
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
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
// One CTA of 16 warps per chunk. Warp w owns the 16 x 32 block (rows 16 (w & 3), columns
// 32 (w >> 2)) of every 64 x 128 quantity and keeps dk, dq and dG for it in registers, so every
// elementwise step is local; 64 x 64 products give a warp 16 x 16 (rows
// 16 (w & 3), columns 16 (w >> 2)). Phases (block barriers between them):
//   1  <S, dS'> per channel; dKe = E dS'^T; dQg = s dO S^T; dW = -dE S^T; dA = s lower(dO E^T)
//   1b dW and dA stored; the bf16 factor tiles K_g, K_r, K_m, Q_r built over S, dS' and E
//   2  dQr = dA K_m -> dq; dXK = T^T dW; dXV = T^T dE -> dv; dT
//   3  Y = T^T dT; P = K_r K_m^T, dR and dP = beta dR
//   4  dKr = dP K_m; dKm = dP^T K_r + dA^T Q_r; then per token dbeta, deta, the k coefficient,
//      dk, and the reverse prefix of dG per channel -> dalpha.
constexpr int kGradThreads = 512;
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
constexpr int GC_COLK = GC_DGAM + kD * 4;                     // fp32 [4][128] column sums of dKe K_e
constexpr int GC_RROW = GC_COLK + 4 * kD * 4;                 // fp32 [3][4][64] row partials
constexpr int GC_KC = GC_RROW + 3 * 4 * kC * 4;               // fp32 [64] k coefficient
constexpr int GC_QS = GC_KC + kC * 4;                         // fp32 [4][128] partial sums of the gates / of dG
constexpr int GC_BYTES = GC_QS + 4 * kD * 4;
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
          *kcoef = reinterpret_cast<float *>(smem + GC_KC), *squart = reinterpret_cast<float *>(smem + GC_QS);
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
    load_dense<kD>(sDE, p.ws.dE + n * kC * kD, kC, tid, kGradThreads);
    load_dense<kD>(sS, p.ws.S + n * kD * kD, kD, tid, kGradThreads);
    load_dense<kD>(sDS, p.ws.dS + n * kD * kD, kD, tid, kGradThreads);
    load_dense<kC>(sT, p.ws.Tm + n * kC * kC, kC, tid, kGradThreads);
    if (tid < static_cast<int>(kCgFloats) / 4)
        cp16(smem + GC_CG + 16 * tid, p.ws.cg + n * kCgFloats + 4 * tid, true);
    cp_commit();
    // G per (token, channel) while the tiles land, in the prep kernel's order of summation:
    // threads 0-255 as (channel pair, quarter of the chunk)
    {
        const int cp = tid & 63, qt = (tid >> 6) & 3;
        float lg[2][16];
        if (tid < 4 * 64) gate_logs(p.alpha, tok0, p.H, L, cp, qt, lg, squart);
        __syncthreads();
        if (tid < 4 * 64) {
            const GateRef g0 = gate_ref(squart, 2 * cp, qt), g1 = gate_ref(squart, 2 * cp + 1, qt);
            float G0 = g0.off, G1 = g1.off;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                G0 += lg[0][u];
                G1 += lg[1][u];
                *reinterpret_cast<float2 *>(sG + (16 * qt + u) * kPG + 2 * cp) = make_float2(G0, G1);
            }
            if (qt == 0) {
                *reinterpret_cast<float2 *>(sGr + 2 * cp) = make_float2(g0.Gr, g1.Gr);
                *reinterpret_cast<float2 *>(sGe + 2 * cp) = make_float2(g0.Gend, g1.Gend);
            }
        }
    }
    cp_wait<0>();
    __syncthreads();

    const int r1 = 16 * (warp & 3), c1 = 32 * (warp >> 2), cb = warp >> 2;   // 64 x 128: 16 x 32 per warp
    const int c2 = 16 * (warp >> 2);                                         // 64 x 64: 16 x 16 per warp
    auto row1 = [&](int hh) { return r1 + g + 8 * hh; };
    auto col1 = [&](int ni) { return c1 + 8 * ni + 2 * q4; };
    auto col2 = [&](int ni) { return c2 + 8 * ni + 2 * q4; };
    auto gpair = [&](int r, int col) { return *reinterpret_cast<const float2 *>(sG + r * kPG + col); };
    auto put_row = [&](int qi, int row, float x) {   // sum over the 4 lanes of a row, into column block cb
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        if (q4 == 0) rrow[qi][cb][row] = x;
    };
    auto dq_row = [&](int r) { return p.dq + (tok0 + static_cast<size_t>(r) * p.H) * kD; };

    float dk[1][4][4], dq[1][4][4], dg[1][4][4], tmp[1][4][4];
    float da[1][2][4];
    // ---- phase 1
    {   // <S, dS'> per key channel (row of S): four threads per row
        const int r = tid >> 2, h0 = (tid & 3) * 32;
        float sum = 0.f;
#pragma unroll
        for (int cc = 0; cc < 32; cc += 8) {
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
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if ((tid & 3) == 0) sDGam[r] = sum;
    }
    // dKe = E dS'^T: dk = dKe e^{G_end - G}, dG = -dKe K_e, column sums of dKe K_e for the last row
    zero(dk[0]);
    gemm_k2<1, 4, 8, false, false>(dk, sptr(sE), kP, r1, 0, sptr(sDS), kP, c1, 0, lane);
    {
        float colk[4][2] = {};
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int col = col1(ni);
            const float ge0 = sGe[col], ge1 = sGe[col + 1];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = row1(hh);
                const float2 G2 = gpair(r, col), k2 = ld_pair(sK, kP, r, col);
                const float x0 = dk[0][ni][2 * hh] * __expf(ge0 - G2.x), x1 = dk[0][ni][2 * hh + 1] * __expf(ge1 - G2.y);
                const float m0 = x0 * k2.x, m1 = x1 * k2.y;   // dKe . K_e
                dg[0][ni][2 * hh] = -m0;
                dg[0][ni][2 * hh + 1] = -m1;
                colk[ni][0] += m0;
                colk[ni][1] += m1;
                dk[0][ni][2 * hh] = x0;
                dk[0][ni][2 * hh + 1] = x1;
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
                if (g == 0) sColK[(warp & 3) * kD + col1(ni) + e] = y;
            }
    }
    // dQg = s dO S^T: dq = dQg e^{G}, dG += dQg Q_g
    zero(dq[0]);
    gemm_k2<1, 4, 8, false, false>(dq, sptr(sDO), kP, r1, 0, sptr(sS), kP, c1, 0, lane);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int r = row1(hh);
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int col = col1(ni);
            const float2 G2 = gpair(r, col), q2 = ld_pair(sQ, kP, r, col);
            const float x0 = dq[0][ni][2 * hh] * s * __expf(G2.x), x1 = dq[0][ni][2 * hh + 1] * s * __expf(G2.y);
            dg[0][ni][2 * hh] = fmaf(x0, q2.x, dg[0][ni][2 * hh]);
            dg[0][ni][2 * hh + 1] = fmaf(x1, q2.y, dg[0][ni][2 * hh + 1]);
            dq[0][ni][2 * hh] = x0;
            dq[0][ni][2 * hh + 1] = x1;
        }
    }
    // dW = -dE S^T (stored after the barrier, over S)
    zero(tmp[0]);
    gemm_k2<1, 4, 8, false, false>(tmp, sptr(sDE), kP, r1, 0, sptr(sS), kP, c1, 0, lane);
    // dA = s lower(dO E^T) (stored after the barrier, over dO)
    da[0][0][0] = da[0][0][1] = da[0][0][2] = da[0][0][3] = 0.f;
    da[0][1][0] = da[0][1][1] = da[0][1][2] = da[0][1][3] = 0.f;
    gemm_k2<1, 2, 8, false, false>(da, sptr(sDO), kP, r1, 0, sptr(sE), kP, c2, 0, lane);
    __syncthreads();   // every read of S, dS', E and dO is done

    // ---- phase 1b: dW, dA; the factor tiles
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
            st_pair(sDW, kP, row1(hh), col1(ni), -tmp[0][ni][2 * hh], -tmp[0][ni][2 * hh + 1]);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int i = row1(hh);
#pragma unroll
        for (int ni = 0; ni < 2; ++ni) {
            const int j = col2(ni);
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

    // ---- phase 2: dQr -> dq;  dXK = T^T dW -> dk, dG, dbeta part;  dXV = T^T dE -> dv, dbeta part;  dT
    // dQr = dA K_m: dq += dQr e^{G - G_r}, dG += dQr Q_r (the bf16 Q_r of dA^T Q_r); dq is complete
    zero(tmp[0]);
    gemm_m<1, 4, 4, false, true>(tmp, sptr(sDA), kPs, r1, 0, sptr(sKM), kP, c1, 0, lane);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int r = row1(hh);
        float *dst = dq_row(r);
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int col = col1(ni);
            const float2 G2 = gpair(r, col), qr = ld_pair(sQR, kP, r, col);
            const float x0 = tmp[0][ni][2 * hh], x1 = tmp[0][ni][2 * hh + 1];
            dg[0][ni][2 * hh] = fmaf(x0, qr.x, dg[0][ni][2 * hh]);
            dg[0][ni][2 * hh + 1] = fmaf(x1, qr.y, dg[0][ni][2 * hh + 1]);
            if (r < L)
                *reinterpret_cast<float2 *>(dst + col) =
                    make_float2(fmaf(x0, __expf(G2.x - sGr[col]), dq[0][ni][2 * hh]),
                                fmaf(x1, __expf(G2.y - sGr[col + 1]), dq[0][ni][2 * hh + 1]));
        }
    }
    zero(tmp[0]);
    gemm_k2<1, 4, 4, true, true>(tmp, sptr(sT), kPs, r1, 0, sptr(sDW), kP, c1, 0, lane);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int r = row1(hh);
        const float bt = cg[kC + r];
        float rsum = 0.f;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int col = col1(ni);
            const float2 G2 = gpair(r, col), k2 = ld_pair(sK, kP, r, col);
            const float eg0 = __expf(G2.x), eg1 = __expf(G2.y);
            const float kg0 = k2.x * eg0, kg1 = k2.y * eg1;   // K_g
            const float x0 = tmp[0][ni][2 * hh], x1 = tmp[0][ni][2 * hh + 1];
            rsum = fmaf(x0, kg0, fmaf(x1, kg1, rsum));
            dg[0][ni][2 * hh] = fmaf(bt * x0, kg0, dg[0][ni][2 * hh]);
            dg[0][ni][2 * hh + 1] = fmaf(bt * x1, kg1, dg[0][ni][2 * hh + 1]);
            dk[0][ni][2 * hh] = fmaf(bt * eg0, x0, dk[0][ni][2 * hh]);
            dk[0][ni][2 * hh + 1] = fmaf(bt * eg1, x1, dk[0][ni][2 * hh + 1]);
        }
        put_row(RB_XK, r, rsum);
    }
    zero(tmp[0]);
    gemm_k2<1, 4, 4, true, true>(tmp, sptr(sT), kPs, r1, 0, sptr(sDE), kP, c1, 0, lane);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int r = row1(hh);
        const float bt = cg[kC + r];
        float rsum = 0.f;
        float *dst = p.dv + (tok0 + static_cast<size_t>(r) * p.H) * kD;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int col = col1(ni);
            const float2 v2 = ld_pair(sV, kP, r, col);
            rsum = fmaf(tmp[0][ni][2 * hh], v2.x, fmaf(tmp[0][ni][2 * hh + 1], v2.y, rsum));
            if (r < L)
                *reinterpret_cast<float2 *>(dst + col) = make_float2(bt * tmp[0][ni][2 * hh], bt * tmp[0][ni][2 * hh + 1]);
        }
        put_row(RB_XV, r, rsum);
    }
    {   // dT = (dW K_g^T + dE V^T) diag(beta)  (over Q)
        float a1[1][2][4] = {};
        gemm_k2<1, 2, 8, false, false>(a1, sptr(sDW), kP, r1, 0, sptr(sKG), kP, c2, 0, lane);
        gemm_k2<1, 2, 8, false, false>(a1, sptr(sDE), kP, r1, 0, sptr(sV), kP, c2, 0, lane);
#pragma unroll
        for (int ni = 0; ni < 2; ++ni) {
            const int j = col2(ni);
            const float bj0 = cg[kC + j], bj1 = cg[kC + j + 1];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                st_pair(sDT, kPs, row1(hh), j, bj0 * a1[0][ni][2 * hh], bj1 * a1[0][ni][2 * hh + 1]);
        }
    }
    __syncthreads();   // dT is visible; V and dE are no longer read

    // ---- phase 3: Y = T^T dT (over V);  P, dR = -strict_lower(Y T^T), dP = beta dR (over dE);  dQr -> dq
    {
        float y[1][2][4] = {};
        gemm_k2<1, 2, 4, true, true>(y, sptr(sT), kPs, r1, 0, sptr(sDT), kPs, c2, 0, lane);
#pragma unroll
        for (int ni = 0; ni < 2; ++ni)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                st_pair(sY, kPs, row1(hh), col2(ni), y[0][ni][2 * hh], y[0][ni][2 * hh + 1]);
    }
    __syncthreads();
    {
        float pk[1][2][4] = {};   // P = K_r K_m^T for the dR . P sums
        gemm_k2<1, 2, 8, false, false>(pk, sptr(sKR), kP, r1, 0, sptr(sKM), kP, c2, 0, lane);
        float dr[1][2][4] = {};
        gemm_k2<1, 2, 4, false, false>(dr, sptr(sY), kPs, r1, 0, sptr(sT), kPs, c2, 0, lane);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int i = row1(hh);
            const float bi = cg[kC + i];
            float rsum = 0.f;
#pragma unroll
            for (int ni = 0; ni < 2; ++ni) {
                const int j = col2(ni);
                const float x0 = j < i ? -dr[0][ni][2 * hh] : 0.f, x1 = j + 1 < i ? -dr[0][ni][2 * hh + 1] : 0.f;
                rsum = fmaf(x0, pk[0][ni][2 * hh], fmaf(x1, pk[0][ni][2 * hh + 1], rsum));
                st_pair(sDP, kPs, i, j, bi * x0, bi * x1);
            }
            put_row(RB_R, i, rsum);
        }
    }
    __syncthreads();   // dP is visible

    // ---- phase 4: dKr = dP K_m -> dk, dG;  dKm = dP^T K_r + dA^T Q_r -> dk, dG
    // alpha of the chunk's tokens for the last step, rows 0-31 over dT and rows 32-63 over Y (both read
    // last in phase 3)
    {
        float *sAl0 = reinterpret_cast<float *>(sDT), *sAl1 = reinterpret_cast<float *>(sY);
        for (int e = tid; e < kC * kD / 4; e += kGradThreads) {
            const int t = e >> 5, cc = (e & 31) * 4;
            if (t < L) cp16((t < 32 ? sAl0 + t * kD : sAl1 + (t - 32) * kD) + cc,
                            p.alpha + (tok0 + static_cast<size_t>(t) * p.H) * kD + cc, true);
        }
        cp_commit();
    }
    zero(tmp[0]);
    gemm_k2<1, 4, 4, false, true>(tmp, sptr(sDP), kPs, r1, 0, sptr(sKM), kP, c1, 0, lane);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int r = row1(hh), col = col1(ni);
            const float2 G2 = gpair(r, col), kr = ld_pair(sKR, kP, r, col);
            const float x0 = tmp[0][ni][2 * hh], x1 = tmp[0][ni][2 * hh + 1];
            dg[0][ni][2 * hh] = fmaf(x0, kr.x, dg[0][ni][2 * hh]);
            dg[0][ni][2 * hh + 1] = fmaf(x1, kr.y, dg[0][ni][2 * hh + 1]);
            dk[0][ni][2 * hh] = fmaf(x0, __expf(G2.x - sGr[col]), dk[0][ni][2 * hh]);
            dk[0][ni][2 * hh + 1] = fmaf(x1, __expf(G2.y - sGr[col + 1]), dk[0][ni][2 * hh + 1]);
        }
    zero(tmp[0]);
    gemm_k2<1, 4, 4, true, true>(tmp, sptr(sDP), kPs, r1, 0, sptr(sKR), kP, c1, 0, lane);
    gemm_k2<1, 4, 4, true, true>(tmp, sptr(sDA), kPs, r1, 0, sptr(sQR), kP, c1, 0, lane);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int r = row1(hh), col = col1(ni);
            const float2 G2 = gpair(r, col), km = ld_pair(sKM, kP, r, col);
            const float x0 = tmp[0][ni][2 * hh], x1 = tmp[0][ni][2 * hh + 1];
            dg[0][ni][2 * hh] = fmaf(-x0, km.x, dg[0][ni][2 * hh]);
            dg[0][ni][2 * hh + 1] = fmaf(-x1, km.y, dg[0][ni][2 * hh + 1]);
            dk[0][ni][2 * hh] = fmaf(x0, __expf(sGr[col] - G2.x), dk[0][ni][2 * hh]);
            dk[0][ni][2 * hh + 1] = fmaf(x1, __expf(sGr[col + 1] - G2.y), dk[0][ni][2 * hh + 1]);
        }
    // dG to shared memory (over dW | K_g, read last in phase 2)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
            *reinterpret_cast<float2 *>(sDG + row1(hh) * kPG + col1(ni)) =
                make_float2(dg[0][ni][2 * hh], dg[0][ni][2 * hh + 1]);
    __syncthreads();   // dG and every row partial are in shared memory

    cp_wait<0>();
    // per token (threads 0-63): dbeta, deta, the k coefficient
    if (tid < kC) {
        const int t = tid;
        auto rsum4 = [&](int qi) { return rrow[qi][0][t] + rrow[qi][1][t] + rrow[qi][2][t] + rrow[qi][3][t]; };
        const float dbeta = rsum4(RB_XK) + rsum4(RB_XV) + rsum4(RB_R), bt = cg[kC + t], den = cg[2 * kC + t];
        float deta = dbeta, kc = 0.f;
        if (!p.beta_raw) {
            const bool flows = den != 0.f;
            deta = flows ? dbeta / den : 0.f;
            kc = flows ? -2.f * bt * dbeta / den : 0.f;
        }
        kcoef[t] = kc;
        if (t < L) p.deta[tok0 + static_cast<size_t>(t) * p.H] = deta;
    }
    // reverse prefix of dG per channel, in quarters of 16 tokens: the quarter sums first
    const int ch = tid & (kD - 1), qt = tid >> 7;
    {
        float sum = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) sum += sDG[(16 * qt + u) * kPG + ch];
        squart[qt * kD + ch] = sum;
    }
    __syncthreads();   // kcoef, the quarter sums and alpha are visible

#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int r = row1(hh);
        if (r >= L) continue;
        const float kc = kcoef[r];
        float *dst = p.dk + (tok0 + static_cast<size_t>(r) * p.H) * kD;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int col = col1(ni);
            const float2 kx = ld_pair(sK, kP, r, col);
            *reinterpret_cast<float2 *>(dst + col) =
                make_float2(fmaf(kc, kx.x, dk[0][ni][2 * hh]), fmaf(kc, kx.y, dk[0][ni][2 * hh + 1]));
        }
    }
    {   // the end decay's terms join the last row: sum_i dKe K_e + Gamma <S, dS'>
        float run = sColK[ch] + sColK[kD + ch] + sColK[2 * kD + ch] + sColK[3 * kD + ch] +
                    __expf(sGe[ch]) * sDGam[ch];
        for (int q = 3; q > qt; --q) run += squart[q * kD + ch];
#pragma unroll 4
        for (int u = 15; u >= 0; --u) {
            const int t = 16 * qt + u;
            run += sDG[t * kPG + ch];
            if (t < L) {
                const float a = t < 32 ? reinterpret_cast<const float *>(sDT)[t * kD + ch]
                                       : reinterpret_cast<const float *>(sY)[(t - 32) * kD + ch];
                p.dalpha[(tok0 + static_cast<size_t>(t) * p.H) * kD + ch] = run / a;
            }
        }
    }
}

}  // namespace

cudaError_t launch_bwd_prep_ch(const ChBwd &p, cudaStream_t stream) {
    const uint64_t N = static_cast<uint64_t>(p.B) * p.H * p.nc;
    CUtensorMap mQ, mK, mV, mW, mU;
    if (!map_tokens(&mQ, p.q, p.B, p.T, p.H) || !map_tokens(&mK, p.k, p.B, p.T, p.H) ||
        !map_tokens(&mV, p.v, p.B, p.T, p.H) || !map_record(&mW, p.ws.W, kD, N * kC, kC) ||
        !map_record(&mU, p.ws.UdE, kD, N * kC, kC))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(bwd_prep_ch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(pc::kBytes));
    if (e != cudaSuccess) return e;
    bwd_prep_ch_kernel<<<dim3(p.nc, p.B * p.H), pc::kThreads, pc::kBytes, stream>>>(mQ, mK, mV, mW, mU, p);
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
