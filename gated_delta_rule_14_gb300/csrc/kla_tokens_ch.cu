// kla_tokens_ch.cu -- several tokens per call with the per-key-channel gate: the call's T tokens
// (9 <= T <= 16) as one chunk of the chunk form, bf16, d_k = d_v = 128.
//
// The chunk algebra of GeekNews, "Revisando las variantes de atencion lineal de la familia
// DeltaNet", section "KDA por chunks", with C = T and the per-channel decay of section "Kimi
// Delta Attention". With G_t[k] the in-call prefix of log alpha of key channel k (inclusive of
// token t) and beta_t the step size:
//   R_im = beta_i sum_k k_i[k] k_m[k] e^{G_i[k] - G_m[k]}   (m < i)     strictly lower
//   A_im =        sum_k q_i[k] k_m[k] e^{G_i[k] - G_m[k]}   (m <= i)    lower
//   Y    = diag(beta) (V - (K . e^G) S),   E = (I + R)^{-1} Y           (the page's order)
//   O    = s ((Q . e^G) S + A E)
//   S'   = diag(e^{G_end}) S + (K . e^{G_end - G})^T E
// where (X . e^G) scales element [t][k] of X by e^{G_t[k]} and diag(e^{G_end}) scales the state's
// key rows. No factor may overflow whatever the gates: the two 8 x 8 diagonal blocks of R and A
// are formed exactly on the CUDA cores (e^{G_i[k] - G_m[k]} <= 1 for m <= i), and the block of
// rows 8-15 and columns 0-7 is factorised around token 8, where both factors e^{G_i - G_8} and
// e^{G_8 - G_m} are at most 1 (a single reference token for the whole call, as on the 64-token
// chunk path, would bound the gates' range). The contractions with the state and that block run
// on warp-level bf16 tensor cores with fp32 accumulation, the small T x T ones in tf32.
//
// One CTA of 256 threads per head at a time (persistent over heads; two CTAs per SM, so one
// CTA's loads overlap the other's arithmetic); warp w owns value columns 16 w .. 16 w + 15.
// The state is read once from shared memory into the fp32 accumulators of the last
// contraction and written back as bf16 over the consumed words, as the B operand of
// [K;Q] S (the scalar-gate kernel of kla_decode.cu does the same).
#include <algorithm>

#include "kla_internal.cuh"
#include "warp_mma.cuh"

namespace kla {
namespace {

namespace tch {
constexpr int kThreads = 256;
constexpr int kPs = 136;   // fp32 state row pitch (words)
constexpr int kPb = 136;   // bf16 token-tile row pitch (elements): conflict-free ldmatrix
constexpr int kPe = 136;   // fp32 Y / E row pitch
constexpr int kMp = 17;    // 16 x 16 matrices
constexpr int kOffS = 0;                                  // state [128][kPs] f32
constexpr int kOffK = kOffS + 128 * kPs * 4;              // k [16][kPb] bf16, then K . e^G
constexpr int kOffQ = kOffK + 16 * kPb * 2;               // q [16][kPb] bf16, then Q . e^G
constexpr int kOffKe = kOffQ + 16 * kPb * 2;              // K . e^{G_end - G} [16][kPb] bf16
constexpr int kOffEc = kOffKe + 16 * kPb * 2;             // E [16][kPb] bf16
constexpr int kOffV = kOffEc + 16 * kPb * 2;              // v [16][128] bf16
constexpr int kOffG = kOffV + 16 * 128 * 2;               // alpha, then G [16][128] f32
constexpr int kOffE = kOffG + 16 * 128 * 4;               // Y, then E [16][kPe] f32
constexpr int kOffM = kOffE + 16 * kPe * 4;               // R, A, T [3][16][kMp] f32
constexpr int kOffVec = kOffM + 3 * 16 * kMp * 4;         // eta, beta [2][16] f32; e^{G_end} [128] f32
constexpr int kBytes = kOffVec + (32 + 128) * 4;
static_assert(kOffK % 16 == 0 && kOffQ % 16 == 0 && kOffKe % 16 == 0 && kOffEc % 16 == 0 && kOffV % 16 == 0 &&
                  kOffG % 16 == 0 && kOffE % 16 == 0 && kOffM % 16 == 0 && kOffVec % 16 == 0,
              "16-byte aligned regions");
static_assert(2 * (kBytes + 1024) <= 233472, "two CTAs per SM");
constexpr float kMinLogGate = -80.0f;   // log-gates below are clamped (e^-80 is below every fp32 contribution)
// Byte offset, within row `key` of the state buffer, of the bf16 copy of 8-column tile nt of the
// warp's 16 columns (starting at column nb): keys 4..7 of every 8 are shifted by 16 bytes so
// that eight consecutive keys fall in distinct groups of four banks.
__device__ __forceinline__ int bf16_slot(int key, int nb, int nt) {
    return key * kPs * 4 + nb * 4 + 16 * ((key >> 2) & 1) + 16 * nt;
}
}  // namespace tch

struct TokChParams {
    const __nv_bfloat16 *q, *k, *v;
    const float *alpha, *eta;   // alpha [B, T, H, 128]; eta [B, T, H]
    float eps;
    const float *S0;            // NULL: zeros
    float *S_T;                 // NULL: not written; may alias S0
    __nv_bfloat16 *o;
    int B, T, H;
    int beta_raw;
    float q_scale;
};

__device__ __forceinline__ void cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(wmma16::sptr(dst)), "l"(src) : "memory");
}

__global__ void __launch_bounds__(tch::kThreads, 2) tokens_ch_kernel(const TokChParams p) {
    using namespace wmma16;
    typedef __nv_bfloat16 bf16;
    constexpr int DK = 128, DV = 128, MP = tch::kMp;
    extern __shared__ __align__(16) unsigned char dsm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, q4 = lane & 3;
    const int T = p.T, nheads = p.B * p.H, nb = 16 * warp;
    float *sS = reinterpret_cast<float *>(dsm + tch::kOffS);
    bf16 *sk = reinterpret_cast<bf16 *>(dsm + tch::kOffK), *sq = reinterpret_cast<bf16 *>(dsm + tch::kOffQ);
    bf16 *sKe = reinterpret_cast<bf16 *>(dsm + tch::kOffKe), *sEc = reinterpret_cast<bf16 *>(dsm + tch::kOffEc);
    bf16 *sv = reinterpret_cast<bf16 *>(dsm + tch::kOffV);
    float *sG = reinterpret_cast<float *>(dsm + tch::kOffG), *sE = reinterpret_cast<float *>(dsm + tch::kOffE);
    float *sR = reinterpret_cast<float *>(dsm + tch::kOffM), *sAm = sR + 16 * MP, *sT = sAm + 16 * MP;
    float *seta = reinterpret_cast<float *>(dsm + tch::kOffVec), *sbeta = seta + 16, *sgend = seta + 32;
    const uint32_t sS_u32 = sptr(sS);
    const unsigned full = 0xffffffffu;

    for (int head = blockIdx.x; head < nheads; head += gridDim.x) {
        const int b = head / p.H, h = head - b * p.H;
        const size_t row0 = static_cast<size_t>(b) * T * p.H + h;   // [B, T, H] row of the first token
        // (0) the state; 16 rows of k, q, v and of the per-channel gates (tokens past T: zeros and
        // gates of 1); eta (0 past T)
        if (p.S0) {
            const float *Sg = p.S0 + static_cast<size_t>(head) * DK * DV;
            for (int c = tid; c < DK * (DV / 4); c += tch::kThreads) cp16(sS + (c >> 5) * tch::kPs + (c & 31) * 4, Sg + c * 4);
        } else {
            for (int c = tid; c < DK * (DV / 4); c += tch::kThreads)
                *reinterpret_cast<float4 *>(sS + (c >> 5) * tch::kPs + (c & 31) * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        {
            const int u = tid >> 4, ch = tid & 15;
            bf16 *dk = sk + u * tch::kPb + ch * 8, *dq = sq + u * tch::kPb + ch * 8, *dv = sv + u * DV + ch * 8;
            if (u < T) {
                const size_t r = row0 + static_cast<size_t>(u) * p.H;
                cp16(dk, p.k + r * DK + ch * 8);
                cp16(dq, p.q + r * DK + ch * 8);
                cp16(dv, p.v + r * DV + ch * 8);
                cp16(sG + u * DK + ch * 8, p.alpha + r * DK + ch * 8);
                cp16(sG + u * DK + ch * 8 + 4, p.alpha + r * DK + ch * 8 + 4);
            } else {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(dk) = z;
                *reinterpret_cast<uint4 *>(dq) = z;
                *reinterpret_cast<uint4 *>(dv) = z;
                *reinterpret_cast<float4 *>(sG + u * DK + ch * 8) = make_float4(1.f, 1.f, 1.f, 1.f);
                *reinterpret_cast<float4 *>(sG + u * DK + ch * 8 + 4) = make_float4(1.f, 1.f, 1.f, 1.f);
            }
            if (tid < 16) seta[tid] = tid < T ? p.eta[row0 + static_cast<size_t>(tid) * p.H] : 0.f;
        }
        asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
        __syncthreads();   // (A) inputs visible

        // (1) threads 0-127: G of key channel tid over the tokens (in place of alpha) and
        // e^{G_end}; threads 128-255: ||k_t||^2 (8 threads per token) and the step sizes
        if (tid < DK) {
            float G = 0.f;
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                G += fmaxf(__logf(sG[t * DK + tid]), tch::kMinLogGate);
                sG[t * DK + tid] = G;   // tokens past T have gates of 1: G stays G_end
            }
            sgend[tid] = __expf(G);
        } else {
            const int t = (tid - DK) >> 3, part = tid & 7;
            float n2 = 0.f;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint4 x = *reinterpret_cast<const uint4 *>(sk + t * tch::kPb + 16 * part + 8 * j);
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 f = unpack2(w[u]);
                    n2 = fmaf(f.x, f.x, n2);
                    n2 = fmaf(f.y, f.y, n2);
                }
            }
            n2 += __shfl_xor_sync(full, n2, 1);
            n2 += __shfl_xor_sync(full, n2, 2);
            n2 += __shfl_xor_sync(full, n2, 4);
            if (part == 0) sbeta[t] = t < T ? kla_beta(seta[t], n2, p.eps, p.beta_raw) : 0.f;
        }
        __syncthreads();   // (B) G, e^{G_end} and beta visible

        // (2) R and A. Block (rows 8-15, columns 0-7) factorises around token 8 with both factors at
        // most 1 (m < 8 <= i: e^{G_i - G_8} and e^{G_8 - G_m}, so nothing overflows and an underflow
        // only loses a term below e^-87): one warp MMA over [K_hi; Q_hi] e^{G - G_8} and
        // K_lo e^{G_8 - G}, in bf16 like the contractions with the state. The two 8 x 8 diagonal
        // blocks are formed exactly per channel: warp w takes rows w and 15 - w (9 entries), lane =
        // 4 key channels. K . e^{G_end - G} from the raw keys meanwhile.
        bf16 *sHi = sEc;                                 // [K_hi; Q_hi] e^{G - G_8}: 16 rows
        bf16 *sLo = reinterpret_cast<bf16 *>(sE);        // K_lo e^{G_8 - G}: rows 0-7 (8-15 zero)
        {
            const int t = tid >> 4, cc = 8 * (tid & 15);   // row t of [K_hi; Q_hi], 8 channels
            const int i = 8 + (t & 7);
            const uint4 x = *reinterpret_cast<const uint4 *>((t < 8 ? sk : sq) + i * tch::kPb + cc);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            uint32_t o4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = unpack2(w[u]);
                const int k0 = cc + 2 * u;
                o4[u] = pack2(f.x * __expf(sG[i * DK + k0] - sG[8 * DK + k0]),
                              f.y * __expf(sG[i * DK + k0 + 1] - sG[8 * DK + k0 + 1]));
            }
            *reinterpret_cast<uint4 *>(sHi + t * tch::kPb + cc) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            if (t < 8) {
                const uint4 y = *reinterpret_cast<const uint4 *>(sk + t * tch::kPb + cc);
                const uint32_t wy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 f = unpack2(wy[u]);
                    const int k0 = cc + 2 * u;
                    o4[u] = pack2(f.x * __expf(sG[8 * DK + k0] - sG[t * DK + k0]),
                                  f.y * __expf(sG[8 * DK + k0 + 1] - sG[t * DK + k0 + 1]));
                }
                *reinterpret_cast<uint4 *>(sLo + t * tch::kPb + cc) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            } else {
                *reinterpret_cast<uint4 *>(sLo + t * tch::kPb + cc) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        __syncthreads();
        {
            if (warp == 7) {   // the off-diagonal block on the tensor cores
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks) {
                    uint32_t a[4], bb[4];
                    frag_a_rk(sptr(sHi), tch::kPb, 0, 16 * ks, lane, a);
                    frag_b_rk(sptr(sLo), tch::kPb, 0, 16 * ks, lane, bb);
                    mma(acc, a, bb[0], bb[1]);
                }
                const int i = 8 + g, m = 2 * q4;
                const float bi = sbeta[i];
                sR[i * MP + m] = bi * acc[0];
                sR[i * MP + m + 1] = bi * acc[1];
                sAm[i * MP + m] = acc[2];
                sAm[i * MP + m + 1] = acc[3];
            }
            const int c0 = 4 * lane;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int i = rr ? 15 - warp : warp, mlo = i < 8 ? 0 : 8;
                const float2 ki01 = unpack2(*reinterpret_cast<const uint32_t *>(sk + i * tch::kPb + c0));
                const float2 ki23 = unpack2(*reinterpret_cast<const uint32_t *>(sk + i * tch::kPb + c0 + 2));
                const float2 qi01 = unpack2(*reinterpret_cast<const uint32_t *>(sq + i * tch::kPb + c0));
                const float2 qi23 = unpack2(*reinterpret_cast<const uint32_t *>(sq + i * tch::kPb + c0 + 2));
                const float4 Gi = *reinterpret_cast<const float4 *>(sG + i * DK + c0);
                const float bi = sbeta[i];
                constexpr int kGrp = 2;
                // columns mlo <= m <= i in groups of kGrp: the 2 kGrp reductions of a group run level
                // by level together, so a group costs one chain of five shuffle latencies
                for (int m0 = mlo; m0 <= i; m0 += kGrp) {
                    float r[kGrp], a[kGrp];
#pragma unroll
                    for (int u = 0; u < kGrp; ++u) {
                        const int m = min(m0 + u, 15);
                        const float2 km01 = unpack2(*reinterpret_cast<const uint32_t *>(sk + m * tch::kPb + c0));
                        const float2 km23 = unpack2(*reinterpret_cast<const uint32_t *>(sk + m * tch::kPb + c0 + 2));
                        const float4 Gm = *reinterpret_cast<const float4 *>(sG + m * DK + c0);
                        const float d0 = __expf(Gi.x - Gm.x), d1 = __expf(Gi.y - Gm.y), d2 = __expf(Gi.z - Gm.z),
                                    d3 = __expf(Gi.w - Gm.w);
                        const float w0 = km01.x * d0, w1 = km01.y * d1, w2 = km23.x * d2, w3 = km23.y * d3;
                        r[u] = ki01.x * w0 + ki01.y * w1 + ki23.x * w2 + ki23.y * w3;
                        a[u] = qi01.x * w0 + qi01.y * w1 + qi23.x * w2 + qi23.y * w3;
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                        for (int u = 0; u < kGrp; ++u) {
                            r[u] += __shfl_xor_sync(full, r[u], o);
                            a[u] += __shfl_xor_sync(full, a[u], o);
                        }
                    }
                    if (lane == 0) {
#pragma unroll
                        for (int u = 0; u < kGrp; ++u) {
                            const int m = m0 + u;
                            if (m <= i) {
                                sR[i * MP + m] = m < i ? bi * r[u] : 0.f;
                                sAm[i * MP + m] = a[u];
                            }
                        }
                    }
                }
                if (lane < 16 - (i + 1)) {   // the upper triangle is zero
                    sR[i * MP + i + 1 + lane] = 0.f;
                    sAm[i * MP + i + 1 + lane] = 0.f;
                }
            }
            // K . e^{G_end - G}: thread = (token tid / 16, 8 channels)
            const int t = tid >> 4, cc = 8 * (tid & 15);
            const uint4 x = *reinterpret_cast<const uint4 *>(sk + t * tch::kPb + cc);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            uint32_t o4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {   // G_end is row 15 of G (tokens past T have gates of 1)
                const float2 f = unpack2(w[u]);
                const int k0 = cc + 2 * u;
                const float d0 = __expf(sG[15 * DK + k0] - sG[t * DK + k0]);
                const float d1 = __expf(sG[15 * DK + k0 + 1] - sG[t * DK + k0 + 1]);
                o4[u] = pack2(f.x * d0, f.y * d1);
            }
            *reinterpret_cast<uint4 *>(sKe + t * tch::kPb + cc) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
        __syncthreads();   // (C) R, A and K . e^{G_end - G} written; raw k and q read for the last time

        // (3) K . e^G and Q . e^G in place (thread = (token, 8 channels)); warp 0 then solves T
        {
            const int t = tid >> 4, cc = 8 * (tid & 15);
            float eg[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) eg[u] = __expf(sG[t * DK + cc + u]);
            bf16 *tiles[2] = {sk + t * tch::kPb + cc, sq + t * tch::kPb + cc};
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const uint4 x = *reinterpret_cast<const uint4 *>(tiles[s]);
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
                uint32_t o4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 f = unpack2(w[u]);
                    o4[u] = pack2(f.x * eg[2 * u], f.y * eg[2 * u + 1]);
                }
                *reinterpret_cast<uint4 *>(tiles[s]) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
        }
        // every warp: its state columns into fp32 accumulators, back as bf16 (B operand of [K;Q] S)
        float sacc[8][2][4];   // rows (keys) 16 mt + g (+ 8), columns nb + 8 nt + 2 q4 (+ 1)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float *r = sS + (16 * mt + g) * tch::kPs + nb + 8 * nt + 2 * q4;
                const float2 x = *reinterpret_cast<const float2 *>(r), y = *reinterpret_cast<const float2 *>(r + 8 * tch::kPs);
                sacc[mt][nt][0] = x.x; sacc[mt][nt][1] = x.y; sacc[mt][nt][2] = y.x; sacc[mt][nt][3] = y.y;
            }
        __syncwarp();
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int key = 16 * mt + g + 8 * hh;
                    *reinterpret_cast<uint32_t *>(dsm + tch::bf16_slot(key, nb, nt) + 4 * q4) =
                        pack2(sacc[mt][nt][2 * hh], sacc[mt][nt][2 * hh + 1]);
                }
        if (warp == 0 && lane < 16) {   // column lane of T = (I + R)^{-1} by forward substitution
            float tc[16];
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) tc[i2] = i2 == lane ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < 15; ++m)
#pragma unroll
                for (int i2 = m + 1; i2 < 16; ++i2) tc[i2] = fmaf(-sR[i2 * MP + m], tc[m], tc[i2]);
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) sT[i2 * MP + lane] = tc[i2];
        }
        __syncthreads();   // (D) scaled K, Q and T visible

        // (4) [K . e^G; Q . e^G] S over the warp's 16 columns
        float pk[2][4] = {}, pq[2][4] = {};   // [n tile]: rows = tokens g, g + 8
        {
            const int m = lane >> 3, r = lane & 7;
            const uint32_t bbase = sS_u32 + tch::bf16_slot(8 * (m & 1) + r, nb, m >> 1);
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks) {
                uint32_t bb[4], ak[4], aq[4];
                ldsm4t(bbase + 16 * ks * tch::kPs * 4, bb);
                frag_a_rk(sptr(sk), tch::kPb, 0, 16 * ks, lane, ak);
                frag_a_rk(sptr(sq), tch::kPb, 0, 16 * ks, lane, aq);
                mma(pk[0], ak, bb[0], bb[1]);
                mma(pk[1], ak, bb[2], bb[3]);
                mma(pq[0], aq, bb[0], bb[1]);
                mma(pq[1], aq, bb[2], bb[3]);
            }
        }
        // Y = diag(beta) (V - (K . e^G) S) into sE (the warp's columns)
        {
            const float b0 = sbeta[g], b1 = sbeta[g + 8];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int u = g + 8 * hh;
                const float bu = hh ? b1 : b0;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float2 vv = unpack2(*reinterpret_cast<const uint32_t *>(sv + u * DV + nb + 8 * nt + 2 * q4));
                    *reinterpret_cast<float2 *>(sE + u * tch::kPe + nb + 8 * nt + 2 * q4) =
                        make_float2(bu * (vv.x - pk[nt][2 * hh]), bu * (vv.y - pk[nt][2 * hh + 1]));
                }
            }
        }
        __syncwarp();
        // (5) E = T Y (tf32 over the tokens); E in place of Y, and as bf16
        float eacc[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int k0 = 8 * ks;
            const uint32_t a[4] = {tf32(sT[g * MP + k0 + q4]), tf32(sT[(g + 8) * MP + k0 + q4]),
                                   tf32(sT[g * MP + k0 + q4 + 4]), tf32(sT[(g + 8) * MP + k0 + q4 + 4])};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                mma_tf32(eacc[nt], a, tf32(sE[(k0 + q4) * tch::kPe + nb + 8 * nt + g]),
                         tf32(sE[(k0 + q4 + 4) * tch::kPe + nb + 8 * nt + g]));
        }
        __syncwarp();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int u = g + 8 * hh;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int col = nb + 8 * nt + 2 * q4;
                *reinterpret_cast<float2 *>(sE + u * tch::kPe + col) = make_float2(eacc[nt][2 * hh], eacc[nt][2 * hh + 1]);
                *reinterpret_cast<uint32_t *>(sEc + u * tch::kPb + col) = pack2(eacc[nt][2 * hh], eacc[nt][2 * hh + 1]);
            }
        }
        __syncwarp();
        // (6) O = s ((Q . e^G) S + A E)
        {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int k0 = 8 * ks;
                const uint32_t a[4] = {tf32(sAm[g * MP + k0 + q4]), tf32(sAm[(g + 8) * MP + k0 + q4]),
                                       tf32(sAm[g * MP + k0 + q4 + 4]), tf32(sAm[(g + 8) * MP + k0 + q4 + 4])};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    mma_tf32(pq[nt], a, tf32(sE[(k0 + q4) * tch::kPe + nb + 8 * nt + g]),
                             tf32(sE[(k0 + q4 + 4) * tch::kPe + nb + 8 * nt + g]));
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int u = g + 8 * hh;
                if (u < T) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        *reinterpret_cast<__nv_bfloat162 *>(p.o + (row0 + static_cast<size_t>(u) * p.H) * DV + nb + 8 * nt + 2 * q4) =
                            __floats2bfloat162_rn(p.q_scale * pq[nt][2 * hh], p.q_scale * pq[nt][2 * hh + 1]);
                }
            }
        }
        // (7) S' = diag(e^{G_end}) S + (K . e^{G_end - G})^T E over 16 tokens (rows past T are zero)
        {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const float ga = sgend[16 * mt + g], gb = sgend[16 * mt + g + 8];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    sacc[mt][nt][0] *= ga; sacc[mt][nt][1] *= ga;
                    sacc[mt][nt][2] *= gb; sacc[mt][nt][3] *= gb;
                }
            }
            uint32_t bb[4];
            frag_b_kr(sptr(sEc), tch::kPb, nb, 0, lane, bb);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                uint32_t a[4];
                frag_a_kr(sptr(sKe), tch::kPb, 16 * mt, 0, lane, a);
                mma(sacc[mt][0], a, bb[0], bb[1]);
                mma(sacc[mt][1], a, bb[2], bb[3]);
            }
        }
        if (p.S_T) {
            float *Sh = p.S_T + static_cast<size_t>(head) * DK * DV;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    float *r = Sh + (16 * mt + g) * DV + nb + 8 * nt + 2 * q4;
                    *reinterpret_cast<float2 *>(r) = make_float2(sacc[mt][nt][0], sacc[mt][nt][1]);
                    *reinterpret_cast<float2 *>(r + 8 * DV) = make_float2(sacc[mt][nt][2], sacc[mt][nt][3]);
                }
        }
        __syncthreads();   // (E) every buffer is read: the next head may overwrite them
    }
}

}  // namespace

bool tokens_ch_supports(const ChunkArgs &a) {
    auto al = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
    // from 9 tokens: measured on GB300 at 64 x 16 heads, a flat ~54 us per call against the token
    // loop's 52.8 us at T = 8, 71.6 us at T = 10 and 102.7 us at T = 16
    return a.dtype == KLA_DTYPE_BF16 && a.gate == KLA_GATE_CHANNEL && a.d_k == 128 && a.d_v == 128 && a.T >= 9 &&
           a.T <= kShortSeqMaxT && al(a.q) && al(a.k) && al(a.v) && al(a.o) && al(a.alpha) &&
           (!a.S0 || al(a.S0)) && (!a.S_T || al(a.S_T));
}

cudaError_t launch_tokens_ch(const ChunkArgs &a) {
    // Cached per device: the shared-memory limit, the SM count and the resident CTAs per SM.
    static bool attr_set[64] = {};
    static int sms_of[64] = {}, per_sm[64] = {};
    int dev = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        if ((e = cudaFuncSetAttribute(tokens_ch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tch::kBytes)) !=
            cudaSuccess)
            return e;
        attr_set[dev] = true;
    }
    if (sms_of[dev] == 0 &&
        (e = cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if (per_sm[dev] == 0) {
        int n = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tokens_ch_kernel, tch::kThreads, tch::kBytes)) !=
            cudaSuccess)
            return e;
        per_sm[dev] = std::max(1, n);
    }
    TokChParams p{static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
                  static_cast<const __nv_bfloat16 *>(a.v), a.alpha, a.eta, a.eps, a.S0, a.S_T,
                  static_cast<__nv_bfloat16 *>(a.o), a.B, a.T, a.H, a.beta_raw, a.q_scale};
    const int nheads = a.B * a.H;
    const int grid = std::min(nheads, per_sm[dev] * sms_of[dev]);
    tokens_ch_kernel<<<grid, tch::kThreads, tch::kBytes, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kla
