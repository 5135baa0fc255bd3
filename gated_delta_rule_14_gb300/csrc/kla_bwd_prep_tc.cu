// kla_bwd_prep_tc.cu -- the per-chunk operands of the chunkwise backward, scalar gate, on the
// tensor cores (tcgen05 with TMEM accumulators, tiles staged by TMA): for every 64-token chunk of
// every (b, h) chain, from q, k, v, alpha and eta, the records the carries and the gradient
// kernel read: G (in-chunk prefix of log alpha), beta, ||k||^2 + eps, A = lower(ratio . Q K^T),
// T = (I + R)^{-1}, W = T diag(beta e^G) K and U = T diag(beta) V (GeekNews, "Revisando las
// variantes de atencion lineal de la familia DeltaNet", section "KDA por chunks").
//
// One CTA of 8 warps per chunk, three per SM. The q and k tiles are stacked as the 128 rows of one
// operand, so a single M = 128 product gives K K^T (rows 0-63) and Q K^T (rows 64-127) in TMEM;
// thread (row, half) turns its half-row into R (fp32, for the solve) or A (bf16, stored
// directly), with beta_i taken from the diagonal ||k_i||^2. T comes from the shared 64 x 64
// unit-lower inverse in fp32; T_K = T diag(beta e^G) and T_V = T diag(beta) enter as K-major bf16
// operands of W^T = K^T T_K^T and U^T = V^T T_V^T (M = 128 key or value channels), whose rows go
// back out through MN-major staging tiles and TMA stores as the row-major W and U records.
#include <cuda.h>

#include "kla_bwd_chunk.cuh"
#include "sm103_ptx.cuh"

namespace kla {
namespace bwdc {
namespace {

using namespace ptx;

constexpr int kThreads = 256;
constexpr uint32_t kHalf = 8192;                   // 64 rows x 128 bytes
constexpr uint32_t OFF_QK = 0;                     // [K half 0 | Q half 0 | K half 1 | Q half 1]; later W, U staging
constexpr uint32_t OFF_TK = OFF_QK + kHalf;        // T_K bf16, K-major [64 t][64 t'], over Q half 0 (read by [K;Q] K^T only)
constexpr uint32_t OFF_TV = OFF_QK + 3 * kHalf;    // T_V, over Q half 1
constexpr uint32_t OFF_V = 4 * kHalf;              // V [half][64 t][64 v]
constexpr uint32_t OFF_R = OFF_V + 2 * kHalf;      // R, then T: fp32 [64][kPR]
constexpr uint32_t OFF_X = OFF_R + kC * kPR * 4;   // solve scratch fp32 [32][kPX]
constexpr uint32_t OFF_VEC = OFF_X + 32 * kPX * 4; // eta, G, beta, beta e^G: fp32 [4][64]
constexpr uint32_t OFF_BAR = OFF_VEC + 4 * kC * 4; // full, mma, TMEM base
constexpr uint32_t kSmemBytes = OFF_BAR + 64 + 1024;
static_assert(OFF_R % 16 == 0 && OFF_X % 16 == 0 && kSmemBytes <= 232448 / 3, "three CTAs per SM");
// TMEM columns: [K;Q] K^T, then W^T over it once read; U^T (128 columns a CTA, three CTAs an SM)
constexpr uint32_t TM_A = 0, TM_W = 0, TM_U = 64, kTmemCols = 128;
constexpr uint32_t kWaitLimit = 100000;               // x 20 us: a stuck wait gives up after ~2 s


struct PrepTcParams {
    const float *alpha, *eta;
    float eps;
    int beta_raw;
    int B, T, H, nc;
    Ws ws;
    unsigned *err;
};

__global__ void __launch_bounds__(kThreads, 3)
prep_tc_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mW,
               const __grid_constant__ CUtensorMap mU, const PrepTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    float(*sR)[kPR] = reinterpret_cast<float(*)[kPR]>(smem + OFF_R);
    float *sX = reinterpret_cast<float *>(smem + OFF_X);
    float *seta = reinterpret_cast<float *>(smem + OFF_VEC), *sG = seta + kC, *sb = sG + kC, *sgb = sb + kC;
    const uint32_t bar_full = sbase + OFF_BAR, bar_mma = bar_full + 8;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + 16);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = 32 * (warp & 3) + lane, half = warp >> 2;   // TMEM lane, column half
    const int c = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
    const int t0 = c * kC, L = min(kC, p.T - t0);
    const size_t n = static_cast<size_t>(bh) * p.nc + c;
    const size_t base = (static_cast<size_t>(b) * p.T + t0) * p.H + h;   // (b, t0, h)

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
        // gates while the tiles land (tokens 2 lane, 2 lane + 1): log alpha, its inclusive prefix G, eta
        float x[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = 2 * lane + e;
            const bool ok = t < L;
            x[e] = ok ? fmaxf(logf(p.alpha[base + static_cast<size_t>(t) * p.H]), kMinLogGate) : 0.f;
            seta[t] = ok ? p.eta[base + static_cast<size_t>(t) * p.H] : 0.f;
        }
        float sc = x[0] + x[1];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, sc, o);
            if (lane >= o) sc += y;
        }
        sG[2 * lane + 1] = sc;
        sG[2 * lane] = sc - x[1];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t tl = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    bool ok = true;
    if (warp == 0) {
        ok = mbar_wait_bounded(bar_full, 0, kWaitLimit);
        if (__all_sync(0xffffffffu, ok) && elect_one()) {   // [K; Q] K^T
            tc_fence_after();
            const uint64_t dq = sw128_desc(sbase + OFF_QK, 16, 1024);
            const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * 2 * kHalf + (s & 3) * 32;
                mma_bf16(tbase + TM_A, desc_add(dq, off), desc_add(dq, off), id, s);
            }
            mma_commit(bar_mma);
        }
        __syncwarp();
    }
    if (!mbar_wait_bounded(bar_mma, 0, kWaitLimit)) ok = false;
    tc_fence_after();
    float *cg = p.ws.cg + n * kCgFloats;
    uint32_t xr[32];   // this thread's half-row of K K^T (row < 64) or Q K^T
    tmem_ld32(tl + TM_A + 32 * half, xr);
    tmem_ld_wait();
    const int i = row & (kC - 1);
    const bool key_row = row < kC;
    if (key_row && (i >> 5) == half) {   // ||k_i||^2 is the diagonal of K K^T
        float n2 = 0.f;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj)   // a fixed index keeps the half-row in registers
            if (jj == (i & 31)) n2 = __uint_as_float(xr[jj]);
        const float beta = i < L ? kla_beta(seta[i], n2, p.eps, p.beta_raw) : 0.f;
        sb[i] = beta;
        sgb[i] = beta * __expf(sG[i]);
        cg[i] = sG[i];
        cg[kC + i] = beta;
        cg[2 * kC + i] = n2 + p.eps;
    }
    __syncthreads();   // beta of every row
    {
        const float Gi = sG[i], scale = key_row ? sb[i] : 1.f;
        float v[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int j = 32 * half + jj;
            const bool keep = key_row ? j < i : j <= i;
            v[jj] = keep ? scale * __expf(Gi - sG[j]) * __uint_as_float(xr[jj]) : 0.f;
        }
        if (key_row) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4 *>(&sR[i][32 * half + 4 * q]) =
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {   // A, unscaled by s, straight to its record
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
    {   // T (bf16 record), T_K = T diag(beta e^G), T_V = T diag(beta) (bf16, K-major, 128-byte swizzle)
        const int r = tid >> 2, kq = tid & 3;
        bf16 *trec = p.ws.Tm + (n * kC + r) * kC + 16 * kq;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float tk[8], tv[8], tt[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = 16 * kq + 8 * hh + u;
                const float t = j <= r ? sR[r][j] : 0.f;
                tt[u] = t;
                tv[u] = t * sb[j];
                tk[u] = t * sgb[j];
            }
            *reinterpret_cast<uint4 *>(trec + 8 * hh) =
                make_uint4(pack_bf16(tt[0], tt[1]), pack_bf16(tt[2], tt[3]), pack_bf16(tt[4], tt[5]),
                           pack_bf16(tt[6], tt[7]));
            const uint32_t off = sw128_off(r, 32 * kq + 16 * hh);
            st_shared_v4(sbase + OFF_TK + off, pack_bf16(tk[0], tk[1]), pack_bf16(tk[2], tk[3]),
                         pack_bf16(tk[4], tk[5]), pack_bf16(tk[6], tk[7]));
            st_shared_v4(sbase + OFF_TV + off, pack_bf16(tv[0], tv[1]), pack_bf16(tv[2], tv[3]),
                         pack_bf16(tv[4], tv[5]), pack_bf16(tv[6], tv[7]));
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {   // W^T = K^T T_K^T and U^T = V^T T_V^T (M = 128 channels, N = 64 tokens, K = 64)
        tc_fence_after();
        if (elect_one()) {
            const uint32_t id = idesc_bf16(128, 64, 1, 0);
            const uint64_t dk = sw128_desc(sbase + OFF_QK, 2 * kHalf, 1024), dtk = sw128_desc(sbase + OFF_TK, 16, 1024);
            const uint64_t dv = sw128_desc(sbase + OFF_V, kHalf, 1024), dtv = sw128_desc(sbase + OFF_TV, 16, 1024);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tbase + TM_W, desc_add(dk, s * 2048), desc_add(dtk, s * 32), id, s);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tbase + TM_U, desc_add(dv, s * 2048), desc_add(dtv, s * 32), id, s);
            mma_commit(bar_mma);
        }
        __syncwarp();
    }
    if (!mbar_wait_bounded(bar_mma, 1, kWaitLimit)) ok = false;
    tc_fence_after();
    // W^T / U^T rows (channel `row`, tokens 32 half ..) -> the row-major W and U records through
    // staging tiles laid out as the records' TMA boxes ([channel half][64 t][64 channels], over
    // the q/k tiles, which the finished products no longer read)
    {
        const uint32_t cb = (row & 63) * 2, hb = (row >> 6) * kHalf;
        unsigned short *wst = reinterpret_cast<unsigned short *>(smem + OFF_QK + hb);
        unsigned short *ust = reinterpret_cast<unsigned short *>(smem + OFF_QK + 2 * kHalf + hb);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            uint32_t d[32];
            tmem_ld32(tl + (m ? TM_U : TM_W) + 32 * half, d);
            tmem_ld_wait();
            unsigned short *st = m ? ust : wst;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) st[sw128_off(32 * half + jj, cb) >> 1] = bf16_bits(__uint_as_float(d[jj]));
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

}  // namespace

cudaError_t launch_prep_tc(const bf16 *q, const bf16 *k, const bf16 *v, const float *alpha, const float *eta,
                           float eps, int beta_raw, int B, int T, int H, int nc, const Ws &ws, unsigned *err,
                           cudaStream_t stream) {
    const uint64_t N = static_cast<uint64_t>(B) * H * nc;
    CUtensorMap mQ, mK, mV, mW, mU;
    if (!map_tokens(&mQ, q, B, T, H) || !map_tokens(&mK, k, B, T, H) || !map_tokens(&mV, v, B, T, H) ||
        !map_record(&mW, ws.W, kD, N * kC, kC) || !map_record(&mU, ws.UdE, kD, N * kC, kC))
        return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const PrepTcParams p{alpha, eta, eps, beta_raw, B, T, H, nc, ws, err};
    prep_tc_kernel<<<dim3(nc, B * H), kThreads, kSmemBytes, stream>>>(mQ, mK, mV, mW, mU, p);
    return cudaGetLastError();
}

}  // namespace bwdc
}  // namespace kla
