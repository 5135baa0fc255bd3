// kla_decode.cu -- fused single-token KLA step (decode).
//
// Per (sequence b, head h) and token (GeekNews, "Revisando las variantes de atencion lineal
// de la familia DeltaNet", section "Kernel Triton recurrente fusionado para decodificacion";
// step size from the KLA page, section "La Regola di Aggiornamento KLA"):
//   S~ = alpha (.) S ;  e = v - S~^T k ;  beta = eta / (||k||^2 + eps) ;  S = S~ + beta k e^T ;
//   o = S^T q.
// Expanding the read after the write gives o = S~^T q + beta e (k . q), so both reductions
// over the key rows (S~^T k and S~^T q) come from ONE pass over the old state, and the new
// state is written in the same pass: every state element is read once and written once.
// The step is HBM-bound (8 d_k d_v bytes of state traffic against 7 d_k d_v flops), so it
// runs on the CUDA cores with 128-bit coalesced loads and stores.
//
// Grid: one CTA of 128 threads per (32-column value tile, head, sequence). A CTA keeps its
// d_k x 32 tile of S in registers (8 float4 per thread at d_k = 128) between the reduction
// and the write.
#include <algorithm>

#include "kla_internal.cuh"
#include "warp_mma.cuh"

namespace kla {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxRowsPerThread = 8;
constexpr float kMinLogGateDecode = -80.0f;   // log-gates below are clamped (e^-80 is below every fp32 contribution)

struct DecodeParams {
    const void *q, *k, *v;
    const float *alpha, *eta;
    float eps;
    float *S;
    void *o;
    int B, H, DK, DV, BV;
    int beta_raw;
    float q_scale;
};

template <typename TIn, bool kChannel, int NCG>   // NCG = float4 column groups per tile (BV / 4)
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecodeParams p) {
    constexpr int RG = kThreads / NCG;            // row groups
    __shared__ float sk[128], sq[128], sa[128];
    __shared__ float sred[2][kThreads / 32][NCG * 4];
    __shared__ float snorm[2][kThreads / 32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid % NCG, rg = tid / NCG;
    const int v0 = blockIdx.x * (NCG * 4);
    const int h = blockIdx.y, b = blockIdx.z;
    const size_t bh = static_cast<size_t>(b) * p.H + h;
    const int DK = p.DK;
    float *Sbh = p.S + bh * DK * p.DV;

    // Issue the state loads first: they are the long pole.
    float4 s[kMaxRowsPerThread];
#pragma unroll
    for (int r = 0; r < kMaxRowsPerThread; ++r) {
        const int i = rg + r * RG;
        if (i < DK) s[r] = *reinterpret_cast<const float4 *>(Sbh + static_cast<size_t>(i) * p.DV + v0 + cg * 4);
    }

    const TIn *q = static_cast<const TIn *>(p.q) + bh * DK;
    const TIn *k = static_cast<const TIn *>(p.k) + bh * DK;
    float kk = 0.f, kq = 0.f;
    if (tid < DK) {
        const float kt = to_f32(k[tid]), qt = to_f32(q[tid]);
        sk[tid] = kt;
        sq[tid] = qt;
        sa[tid] = kChannel ? p.alpha[bh * DK + tid] : 0.f;
        kk = kt * kt;
        kq = kt * qt;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        kk += __shfl_xor_sync(0xffffffffu, kk, off);
        kq += __shfl_xor_sync(0xffffffffu, kq, off);
    }
    if (lane == 0) { snorm[0][warp] = kk; snorm[1][warp] = kq; }
    __syncthreads();
    float knorm2 = 0.f, kdotq = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) { knorm2 += snorm[0][w]; kdotq += snorm[1][w]; }
    const float beta = kla_beta(p.eta[bh], knorm2, p.eps, p.beta_raw);
    const float a_scalar = kChannel ? 1.f : p.alpha[bh];

    // Partial reductions over this thread's rows of the decayed state.
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int r = 0; r < kMaxRowsPerThread; ++r) {
        const int i = rg + r * RG;
        if (i < DK) {
            const float a = kChannel ? sa[i] : a_scalar;
            const float ak = a * sk[i], aq = a * sq[i];
            pk.x = fmaf(ak, s[r].x, pk.x); pk.y = fmaf(ak, s[r].y, pk.y);
            pk.z = fmaf(ak, s[r].z, pk.z); pk.w = fmaf(ak, s[r].w, pk.w);
            pq.x = fmaf(aq, s[r].x, pq.x); pq.y = fmaf(aq, s[r].y, pq.y);
            pq.z = fmaf(aq, s[r].z, pq.z); pq.w = fmaf(aq, s[r].w, pq.w);
        }
    }
    // Reduce over the row groups of the warp (lanes sharing a column group).
#pragma unroll
    for (int off = NCG; off < 32; off <<= 1) {
        pk.x += __shfl_xor_sync(0xffffffffu, pk.x, off); pk.y += __shfl_xor_sync(0xffffffffu, pk.y, off);
        pk.z += __shfl_xor_sync(0xffffffffu, pk.z, off); pk.w += __shfl_xor_sync(0xffffffffu, pk.w, off);
        pq.x += __shfl_xor_sync(0xffffffffu, pq.x, off); pq.y += __shfl_xor_sync(0xffffffffu, pq.y, off);
        pq.z += __shfl_xor_sync(0xffffffffu, pq.z, off); pq.w += __shfl_xor_sync(0xffffffffu, pq.w, off);
    }
    if (lane < NCG) {
        *reinterpret_cast<float4 *>(&sred[0][warp][lane * 4]) = pk;
        *reinterpret_cast<float4 *>(&sred[1][warp][lane * 4]) = pq;
    }
    __syncthreads();
    float4 pred = make_float4(0.f, 0.f, 0.f, 0.f), rd = pred;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const float4 x = *reinterpret_cast<const float4 *>(&sred[0][w][cg * 4]);
        const float4 y = *reinterpret_cast<const float4 *>(&sred[1][w][cg * 4]);
        pred.x += x.x; pred.y += x.y; pred.z += x.z; pred.w += x.w;
        rd.x += y.x; rd.y += y.y; rd.z += y.z; rd.w += y.w;
    }
    const TIn *vv = static_cast<const TIn *>(p.v) + bh * p.DV + v0 + cg * 4;
    float4 e;
    e.x = to_f32(vv[0]) - pred.x; e.y = to_f32(vv[1]) - pred.y;
    e.z = to_f32(vv[2]) - pred.z; e.w = to_f32(vv[3]) - pred.w;

    if (rg == 0) {   // o = s (S~^T q + beta e (k . q))
        TIn *o = static_cast<TIn *>(p.o) + bh * p.DV + v0 + cg * 4;
        const float bkq = beta * kdotq, sc = p.q_scale;
        o[0] = from_f32<TIn>(sc * fmaf(bkq, e.x, rd.x));
        o[1] = from_f32<TIn>(sc * fmaf(bkq, e.y, rd.y));
        o[2] = from_f32<TIn>(sc * fmaf(bkq, e.z, rd.z));
        o[3] = from_f32<TIn>(sc * fmaf(bkq, e.w, rd.w));
    }
    // S = S~ + beta k e^T
#pragma unroll
    for (int r = 0; r < kMaxRowsPerThread; ++r) {
        const int i = rg + r * RG;
        if (i < DK) {
            const float a = kChannel ? sa[i] : a_scalar;
            const float bk = beta * sk[i];
            float4 x;
            x.x = fmaf(a, s[r].x, bk * e.x); x.y = fmaf(a, s[r].y, bk * e.y);
            x.z = fmaf(a, s[r].z, bk * e.z); x.w = fmaf(a, s[r].w, bk * e.w);
            *reinterpret_cast<float4 *>(Sbh + static_cast<size_t>(i) * p.DV + v0 + cg * 4) = x;
        }
    }
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Persistent, software-pipelined variant for 32-column tiles with 16-byte aligned vectors: each
// CTA walks tiles (32 value columns of one head) with a grid stride and copies the next tile's
// state, k, q, v and gates into the other half of a double buffer (cp.async) while it reduces,
// updates and writes the current one, so an SM always has loads in flight. Same arithmetic, in
// the same order, as decode_kernel.
template <typename TIn, bool kChannel>
__global__ void __launch_bounds__(kThreads, 5) decode_pipe_kernel(const DecodeParams p, int ntiles) {
    constexpr int NCG = 8, RG = kThreads / NCG, BV = 32;
    __shared__ __align__(16) float sS[2][128 * BV];
    __shared__ __align__(16) TIn skq[2][2][128];
    __shared__ __align__(16) TIn sv[2][BV];
    __shared__ __align__(16) float sal[2][kChannel ? 128 : 4];
    __shared__ __align__(16) float seta[2][4];
    __shared__ float sa[128];
    __shared__ float sred[2][kThreads / 32][NCG * 4];
    __shared__ float snorm[2][kThreads / 32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid % NCG, rg = tid / NCG;
    const int DK = p.DK, DV = p.DV, ctiles = DV / BV;
    auto tile_bh = [&](int t, int &v0) {
        v0 = (t % ctiles) * BV;
        return static_cast<size_t>(t / ctiles);   // = b * H + h
    };
    auto prefetch = [&](int t, int slot) {
        int v0;
        const size_t bh = tile_bh(t, v0);
        const float *Sg = p.S + bh * DK * DV + v0;
        for (int c = tid; c < DK * (BV / 4); c += kThreads) {
            const int row = c >> 3, ch = c & 7;
            cp_async16(&sS[slot][row * BV + ch * 4], Sg + static_cast<size_t>(row) * DV + ch * 4);
        }
        constexpr int per16 = 16 / sizeof(TIn);
        const int nkq = DK / per16;                       // 16-byte chunks of k (and of q)
        const TIn *gk = static_cast<const TIn *>(p.k) + bh * DK, *gq = static_cast<const TIn *>(p.q) + bh * DK;
        if (tid < nkq) cp_async16(&skq[slot][0][tid * per16], gk + tid * per16);
        else if (tid < 2 * nkq) cp_async16(&skq[slot][1][(tid - nkq) * per16], gq + (tid - nkq) * per16);
        const int nv = BV / per16;
        if (tid >= 64 && tid < 64 + nv)
            cp_async16(&sv[slot][(tid - 64) * per16], static_cast<const TIn *>(p.v) + bh * DV + v0 + (tid - 64) * per16);
        if (kChannel) {
            if (tid >= 96 && tid < 96 + DK / 4) cp_async16(&sal[slot][(tid - 96) * 4], p.alpha + bh * DK + (tid - 96) * 4);
        } else if (tid == 96) {
            cp_async4(&sal[slot][0], p.alpha + bh);
        }
        if (tid == 127) cp_async4(&seta[slot][0], p.eta + bh);
    };

    int it = 0;
    if (blockIdx.x < ntiles) prefetch(blockIdx.x, 0);
    cp_async_commit();
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int slot = it & 1;
        if (t + static_cast<int>(gridDim.x) < ntiles) prefetch(t + gridDim.x, slot ^ 1);
        cp_async_commit();
        cp_async_wait_1();   // this thread's copies of tile t have landed
        __syncthreads();     // and everyone else's
        int v0;
        const size_t bh = tile_bh(t, v0);

        float4 s[kMaxRowsPerThread];
#pragma unroll
        for (int r = 0; r < kMaxRowsPerThread; ++r) {
            const int i = rg + r * RG;
            if (i < DK) s[r] = *reinterpret_cast<const float4 *>(&sS[slot][i * BV + cg * 4]);
        }
        float kk = 0.f, kq = 0.f;
        if (tid < DK) {
            const float kt = to_f32(skq[slot][0][tid]), qt = to_f32(skq[slot][1][tid]);
            sa[tid] = kChannel ? sal[slot][tid] : 0.f;
            kk = kt * kt;
            kq = kt * qt;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            kk += __shfl_xor_sync(0xffffffffu, kk, off);
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
        }
        if (lane == 0) { snorm[0][warp] = kk; snorm[1][warp] = kq; }
        __syncthreads();
        float knorm2 = 0.f, kdotq = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) { knorm2 += snorm[0][w]; kdotq += snorm[1][w]; }
        const float beta = kla_beta(seta[slot][0], knorm2, p.eps, p.beta_raw);
        const float a_scalar = kChannel ? 1.f : sal[slot][0];

        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
        for (int r = 0; r < kMaxRowsPerThread; ++r) {
            const int i = rg + r * RG;
            if (i < DK) {
                const float a = kChannel ? sa[i] : a_scalar;
                const float ak = a * to_f32(skq[slot][0][i]), aq = a * to_f32(skq[slot][1][i]);
                pk.x = fmaf(ak, s[r].x, pk.x); pk.y = fmaf(ak, s[r].y, pk.y);
                pk.z = fmaf(ak, s[r].z, pk.z); pk.w = fmaf(ak, s[r].w, pk.w);
                pq.x = fmaf(aq, s[r].x, pq.x); pq.y = fmaf(aq, s[r].y, pq.y);
                pq.z = fmaf(aq, s[r].z, pq.z); pq.w = fmaf(aq, s[r].w, pq.w);
            }
        }
#pragma unroll
        for (int off = NCG; off < 32; off <<= 1) {
            pk.x += __shfl_xor_sync(0xffffffffu, pk.x, off); pk.y += __shfl_xor_sync(0xffffffffu, pk.y, off);
            pk.z += __shfl_xor_sync(0xffffffffu, pk.z, off); pk.w += __shfl_xor_sync(0xffffffffu, pk.w, off);
            pq.x += __shfl_xor_sync(0xffffffffu, pq.x, off); pq.y += __shfl_xor_sync(0xffffffffu, pq.y, off);
            pq.z += __shfl_xor_sync(0xffffffffu, pq.z, off); pq.w += __shfl_xor_sync(0xffffffffu, pq.w, off);
        }
        if (lane < NCG) {
            *reinterpret_cast<float4 *>(&sred[0][warp][lane * 4]) = pk;
            *reinterpret_cast<float4 *>(&sred[1][warp][lane * 4]) = pq;
        }
        __syncthreads();
        float4 pred = make_float4(0.f, 0.f, 0.f, 0.f), rd = pred;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const float4 x = *reinterpret_cast<const float4 *>(&sred[0][w][cg * 4]);
            const float4 y = *reinterpret_cast<const float4 *>(&sred[1][w][cg * 4]);
            pred.x += x.x; pred.y += x.y; pred.z += x.z; pred.w += x.w;
            rd.x += y.x; rd.y += y.y; rd.z += y.z; rd.w += y.w;
        }
        const TIn *vv = &sv[slot][cg * 4];
        float4 e;
        e.x = to_f32(vv[0]) - pred.x; e.y = to_f32(vv[1]) - pred.y;
        e.z = to_f32(vv[2]) - pred.z; e.w = to_f32(vv[3]) - pred.w;
        if (rg == 0) {   // o = s (S~^T q + beta e (k . q))
            TIn *o = static_cast<TIn *>(p.o) + bh * DV + v0 + cg * 4;
            const float bkq = beta * kdotq, sc = p.q_scale;
            o[0] = from_f32<TIn>(sc * fmaf(bkq, e.x, rd.x));
            o[1] = from_f32<TIn>(sc * fmaf(bkq, e.y, rd.y));
            o[2] = from_f32<TIn>(sc * fmaf(bkq, e.z, rd.z));
            o[3] = from_f32<TIn>(sc * fmaf(bkq, e.w, rd.w));
        }
        float *Sbh = p.S + bh * DK * DV;
#pragma unroll
        for (int r = 0; r < kMaxRowsPerThread; ++r) {   // S = S~ + beta k e^T
            const int i = rg + r * RG;
            if (i < DK) {
                const float a = kChannel ? sa[i] : a_scalar;
                const float bk = beta * to_f32(skq[slot][0][i]);
                float4 x;
                x.x = fmaf(a, s[r].x, bk * e.x); x.y = fmaf(a, s[r].y, bk * e.y);
                x.z = fmaf(a, s[r].z, bk * e.z); x.w = fmaf(a, s[r].w, bk * e.w);
                *reinterpret_cast<float4 *>(Sbh + static_cast<size_t>(i) * DV + v0 + cg * 4) = x;
            }
        }
        __syncthreads();   // slot, sa, sred and snorm are rewritten by the next tile
    }
}

template <typename TIn, bool kChannel>
int pipe_grid(int ntiles) {
    static int per_sm[64] = {};   // resident CTAs per SM, per device (looked up once)
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 0;
    if (per_sm[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_pipe_kernel<TIn, kChannel>, kThreads, 0) !=
                cudaSuccess || n <= 0)
            return 0;
        per_sm[dev] = n;
    }
    return std::min(ntiles, per_sm[dev] * sms);
}

bool pipe_ok(const DecodeArgs &a) {
    auto al = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
    return a.d_v % 32 == 0 && a.d_k % 8 == 0 && al(a.q) && al(a.k) && al(a.v) && al(a.S) &&
           (a.gate == KLA_GATE_SCALAR || al(a.alpha));
}

template <typename TIn, bool kChannel>
cudaError_t launch_t(const DecodeArgs &a) {
    const int BV = std::min(a.d_v, 32);
    DecodeParams p{a.q, a.k, a.v, a.alpha, a.eta, a.eps, a.S, a.o, a.B, a.H, a.d_k, a.d_v, BV, a.beta_raw, a.q_scale};
    if (pipe_ok(a)) {
        const int ntiles = (a.d_v / 32) * a.H * a.B;
        const int g = pipe_grid<TIn, kChannel>(ntiles);
        if (g > 0) {
            decode_pipe_kernel<TIn, kChannel><<<g, kThreads, 0, a.stream>>>(p, ntiles);
            return cudaGetLastError();
        }
    }
    dim3 grid(a.d_v / BV, a.H, a.B);
    if (BV == 32) decode_kernel<TIn, kChannel, 8><<<grid, kThreads, 0, a.stream>>>(p);
    else decode_kernel<TIn, kChannel, 4><<<grid, kThreads, 0, a.stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- several tokens per call
// Multi-token decode and speculative verification (T <= kShortSeqMaxT tokens per sequence in
// one call, kla_chunk_fwd): the persistent tile walk of decode_pipe_kernel with a token loop
// inside each tile. A tile (32 value columns of one head) of the state is copied in once, the
// T steps run on it in registers, in the single-token step's arithmetic and order (one block
// barrier per token, partial sums double-buffered by token parity), and it is written once as
// S_T; the tiles of the next head stream in meanwhile. The per-token ||k||^2 and k . q are
// formed up front, one warp per token. The step is issue-bound once the state streams, so the
// scalar gate scales the two reduced sums rather than every row, and d_k is fixed at 128.
struct TokParams {
    const void *q, *k, *v;
    const float *alpha, *eta;
    float eps;
    const float *S0;      // NULL: zeros
    float *S_T;           // NULL: not written; may alias S0 (each tile is read before it is written)
    void *o;
    int B, T, H, DK, DV;
    int beta_raw;
    float q_scale;
    int s_bytes;                                    // the state tile (one buffer)
    int stage_bytes, off_kq, off_v, off_a, off_e;   // the tokens' stage layout (two buffers)
};

// d_k = 128, two warps per tile: thread (rg, cg) holds key rows 16 rg .. 16 rg + 15
// (consecutive, so k_u and q_u of its rows arrive as 16-byte loads) and value columns
// 4 cg .. 4 cg + 3 of the tile; the cross-warp sum of a token's partials is over two warps.
constexpr int kTokThreads = 64;
template <typename TIn, bool kChannel>
__global__ void __launch_bounds__(kTokThreads, 8) tokens_pipe_kernel(const TokParams p, int ntiles) {
    constexpr int NCG = 8, BV = 32, DK = 128, RPT = 16;   // RPT rows per thread
    constexpr int kThreads = kTokThreads;
    static_assert(kThreads / NCG * RPT == DK, "rows per thread");
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ __align__(16) float sred[2][kThreads / 32][2 * NCG * 4];
    __shared__ float sbeta[kShortSeqMaxT], skqd[kShortSeqMaxT];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid % NCG, i0 = (tid / NCG) * RPT;
    const int DV = p.DV, T = p.T, ctiles = DV / BV;
    auto tile_bh = [&](int t, int &v0) {
        v0 = (t % ctiles) * BV;
        return static_cast<size_t>(t / ctiles);   // = b * H + h
    };
    auto row_of = [&](size_t bh, int u) {          // [B, T, H] row of token u of chain bh
        const int b = static_cast<int>(bh) / p.H, h = static_cast<int>(bh) - b * p.H;
        return (static_cast<size_t>(b) * T + u) * p.H + h;
    };
    // RPT consecutive values of a TIn row in shared memory, as fp32
    auto loadrow = [](const TIn *src, float (&x)[RPT]) {
#pragma unroll
        for (int h = 0; h < RPT / 8; ++h) {
            if constexpr (sizeof(TIn) == 2) {
                const uint4 w = *reinterpret_cast<const uint4 *>(src + 8 * h);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    x[8 * h + 2 * j] = __uint_as_float(ww[j] << 16);
                    x[8 * h + 2 * j + 1] = __uint_as_float(ww[j] & 0xffff0000u);
                }
            } else {
                const float4 a = *reinterpret_cast<const float4 *>(src + 8 * h);
                const float4 b = *reinterpret_cast<const float4 *>(src + 8 * h + 4);
                x[8 * h] = a.x; x[8 * h + 1] = a.y; x[8 * h + 2] = a.z; x[8 * h + 3] = a.w;
                x[8 * h + 4] = b.x; x[8 * h + 5] = b.y; x[8 * h + 6] = b.z; x[8 * h + 7] = b.w;
            }
        }
    };
    float *sS = reinterpret_cast<float *>(dsm);   // one state tile (refilled for the next tile early)
    auto stage = [&](int slot, int off) { return dsm + p.s_bytes + slot * p.stage_bytes + off; };
    auto prefetch_state = [&](int t) {
        int v0;
        const size_t bh = tile_bh(t, v0);
        if (p.S0) {
            const float *Sg = p.S0 + bh * DK * DV + v0;
            for (int c = tid; c < DK * (BV / 4); c += kThreads) {
                const int row = c >> 3, ch = c & 7;
                cp_async16(&sS[row * BV + ch * 4], Sg + static_cast<size_t>(row) * DV + ch * 4);
            }
        } else {
            for (int c = tid; c < DK * (BV / 4); c += kThreads)
                *reinterpret_cast<float4 *>(&sS[c * 4]) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto prefetch_tokens = [&](int t, int slot) {
        int v0;
        const size_t bh = tile_bh(t, v0);
        constexpr int per16 = 16 / sizeof(TIn);
        constexpr int nch = DK / per16;                // 16-byte chunks of one k or q row
        const size_t row0 = row_of(bh, 0);
        TIn *skq = reinterpret_cast<TIn *>(stage(slot, p.off_kq));
        for (int c = tid; c < T * 2 * nch; c += kThreads) {
            const int u = c / (2 * nch), rem = c - u * 2 * nch, which = rem / nch, ch = rem - which * nch;
            const TIn *src = static_cast<const TIn *>(which ? p.q : p.k) + (row0 + static_cast<size_t>(u) * p.H) * DK + ch * per16;
            cp_async16(skq + (2 * u + which) * DK + ch * per16, src);
        }
        TIn *sv = reinterpret_cast<TIn *>(stage(slot, p.off_v));
        constexpr int nvc = BV / per16;                // 16-byte chunks of a token's 32 values
        for (int c = tid; c < T * nvc; c += kThreads) {
            const int u = c / nvc, ch = c - u * nvc;
            cp_async16(sv + u * BV + ch * per16,
                       static_cast<const TIn *>(p.v) + (row0 + static_cast<size_t>(u) * p.H) * DV + v0 + ch * per16);
        }
        float *sa = reinterpret_cast<float *>(stage(slot, p.off_a));
        if (kChannel) {
            for (int c = tid; c < T * (DK / 4); c += kThreads) {
                const int u = c / (DK / 4), ch = c - u * (DK / 4);
                cp_async16(sa + u * DK + ch * 4, p.alpha + (row0 + static_cast<size_t>(u) * p.H) * DK + ch * 4);
            }
        } else if (tid < T) {
            cp_async4(sa + tid, p.alpha + row0 + static_cast<size_t>(tid) * p.H);
        }
        float *se = reinterpret_cast<float *>(stage(slot, p.off_e));
        if (tid >= 32 && tid < 32 + T) cp_async4(se + (tid - 32), p.eta + row0 + static_cast<size_t>(tid - 32) * p.H);
    };

    int it = 0;
    if (blockIdx.x < ntiles) {
        prefetch_state(blockIdx.x);
        prefetch_tokens(blockIdx.x, 0);
    }
    cp_async_commit();
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int slot = it & 1;
        asm volatile("cp.async.wait_group 0;" ::: "memory");   // tile t's state and tokens have landed
        __syncthreads();     // everyone's copies (and the zero fill of a NULL S0) are visible
        int v0;
        const size_t bh = tile_bh(t, v0);
        const TIn *skq = reinterpret_cast<const TIn *>(stage(slot, p.off_kq));
        const TIn *sv = reinterpret_cast<const TIn *>(stage(slot, p.off_v));
        const float *sa = reinterpret_cast<const float *>(stage(slot, p.off_a));
        const float *se = reinterpret_cast<const float *>(stage(slot, p.off_e));

        for (int u = warp; u < T; u += kThreads / 32) {   // beta_u and k_u . q_u, one warp per token
            float kk = 0.f, kq = 0.f;
#pragma unroll
            for (int j = 0; j < DK / 32; ++j) {
                const float kt = to_f32(skq[2 * u * DK + lane + 32 * j]), qt = to_f32(skq[(2 * u + 1) * DK + lane + 32 * j]);
                kk = fmaf(kt, kt, kk);
                kq = fmaf(kt, qt, kq);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                kk += __shfl_xor_sync(0xffffffffu, kk, off);
                kq += __shfl_xor_sync(0xffffffffu, kq, off);
            }
            if (lane == 0) {
                sbeta[u] = kla_beta(se[u], kk, p.eps, p.beta_raw);
                skqd[u] = kq;
            }
        }
        float2 s[RPT][2];   // this thread's rows, columns (4 cg, 4 cg + 1) and (4 cg + 2, 4 cg + 3)
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const float4 x = *reinterpret_cast<const float4 *>(&sS[(i0 + r) * BV + cg * 4]);
            s[r][0] = make_float2(x.x, x.y);
            s[r][1] = make_float2(x.z, x.w);
        }
        __syncthreads();   // beta and k . q of every token are visible; the state buffer is free
        if (t + static_cast<int>(gridDim.x) < ntiles) {   // the next tile streams in during this one's tokens
            prefetch_state(t + gridDim.x);
            prefetch_tokens(t + gridDim.x, slot ^ 1);
        }
        cp_async_commit();

        const size_t row0 = row_of(bh, 0);
        int par = 0;
        for (int u = 0; u < T; ++u, par ^= 1) {
            float kv[RPT], qv[RPT], av[RPT];
            loadrow(skq + 2 * u * DK + i0, kv);
            loadrow(skq + (2 * u + 1) * DK + i0, qv);
            if (kChannel) {
#pragma unroll
                for (int j = 0; j < RPT / 4; ++j) {
                    const float4 x = *reinterpret_cast<const float4 *>(sa + u * DK + i0 + 4 * j);
                    av[4 * j] = x.x; av[4 * j + 1] = x.y; av[4 * j + 2] = x.z; av[4 * j + 3] = x.w;
                }
            }
            // scalar gate: S~^T k = alpha (S^T k), applied after the reduction; paired fp32 FMAs
            float2 pk0 = make_float2(0.f, 0.f), pk1 = pk0, pq0 = pk0, pq1 = pk0;
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const float ak = kChannel ? av[r] * kv[r] : kv[r], aq = kChannel ? av[r] * qv[r] : qv[r];
                const float2 kk2 = make_float2(ak, ak), qq2 = make_float2(aq, aq);
                pk0 = __ffma2_rn(kk2, s[r][0], pk0); pk1 = __ffma2_rn(kk2, s[r][1], pk1);
                pq0 = __ffma2_rn(qq2, s[r][0], pq0); pq1 = __ffma2_rn(qq2, s[r][1], pq1);
            }
            float4 pk = make_float4(pk0.x, pk0.y, pk1.x, pk1.y), pq = make_float4(pq0.x, pq0.y, pq1.x, pq1.y);
#pragma unroll
            for (int off = NCG; off < 32; off <<= 1) {
                pk.x += __shfl_xor_sync(0xffffffffu, pk.x, off); pk.y += __shfl_xor_sync(0xffffffffu, pk.y, off);
                pk.z += __shfl_xor_sync(0xffffffffu, pk.z, off); pk.w += __shfl_xor_sync(0xffffffffu, pk.w, off);
                pq.x += __shfl_xor_sync(0xffffffffu, pq.x, off); pq.y += __shfl_xor_sync(0xffffffffu, pq.y, off);
                pq.z += __shfl_xor_sync(0xffffffffu, pq.z, off); pq.w += __shfl_xor_sync(0xffffffffu, pq.w, off);
            }
            if (lane < NCG) {
                *reinterpret_cast<float4 *>(&sred[par][warp][lane * 4]) = pk;
                *reinterpret_cast<float4 *>(&sred[par][warp][NCG * 4 + lane * 4]) = pq;
            }
            __syncthreads();   // the partial sums of token u (the other parity is token u +- 1's)
            float4 pred = make_float4(0.f, 0.f, 0.f, 0.f), rd = pred;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) {
                const float4 x = *reinterpret_cast<const float4 *>(&sred[par][w][cg * 4]);
                const float4 y = *reinterpret_cast<const float4 *>(&sred[par][w][NCG * 4 + cg * 4]);
                pred.x += x.x; pred.y += x.y; pred.z += x.z; pred.w += x.w;
                rd.x += y.x; rd.y += y.y; rd.z += y.z; rd.w += y.w;
            }
            const float a_scalar = kChannel ? 1.f : sa[u];
            if (!kChannel) {
                pred.x *= a_scalar; pred.y *= a_scalar; pred.z *= a_scalar; pred.w *= a_scalar;
                rd.x *= a_scalar; rd.y *= a_scalar; rd.z *= a_scalar; rd.w *= a_scalar;
            }
            const TIn *vv = sv + u * BV + cg * 4;
            float4 e;
            e.x = to_f32(vv[0]) - pred.x; e.y = to_f32(vv[1]) - pred.y;
            e.z = to_f32(vv[2]) - pred.z; e.w = to_f32(vv[3]) - pred.w;
            const float beta = sbeta[u];
            if (i0 == 0) {   // o = s (S~^T q + beta e (k . q))
                TIn *o = static_cast<TIn *>(p.o) + (row0 + static_cast<size_t>(u) * p.H) * DV + v0 + cg * 4;
                const float bkq = beta * skqd[u], sc = p.q_scale;
                o[0] = from_f32<TIn>(sc * fmaf(bkq, e.x, rd.x));
                o[1] = from_f32<TIn>(sc * fmaf(bkq, e.y, rd.y));
                o[2] = from_f32<TIn>(sc * fmaf(bkq, e.z, rd.z));
                o[3] = from_f32<TIn>(sc * fmaf(bkq, e.w, rd.w));
            }
            const float2 be01 = make_float2(beta * e.x, beta * e.y), be23 = make_float2(beta * e.z, beta * e.w);
#pragma unroll
            for (int r = 0; r < RPT; ++r) {   // S = S~ + k (beta e)^T
                const float a = kChannel ? av[r] : a_scalar;
                const float2 a2 = make_float2(a, a), k2 = make_float2(kv[r], kv[r]);
                s[r][0] = __ffma2_rn(a2, s[r][0], __fmul2_rn(k2, be01));
                s[r][1] = __ffma2_rn(a2, s[r][1], __fmul2_rn(k2, be23));
            }
        }
        if (p.S_T) {
            float *Sbh = p.S_T + bh * DK * DV;
#pragma unroll
            for (int r = 0; r < RPT; ++r)
                *reinterpret_cast<float4 *>(Sbh + static_cast<size_t>(i0 + r) * DV + v0 + cg * 4) =
                    make_float4(s[r][0].x, s[r][0].y, s[r][1].x, s[r][1].y);
        }
        // the next tile's first barrier orders this tile's reads of the token slot, beta and
        // k . q before they are rewritten
    }
}

// Several tokens per call, bf16 with a scalar gate, d_k = d_v = 128: the call's T tokens form one
// chunk of the chunk form of the recurrence (the prefill's algebra with C = T; GeekNews,
// "Revisando las variantes de atencion lineal de la familia DeltaNet", section "KDA por chunks").
// One CTA per head at a time (persistent over heads, two CTAs per SM), each warp on 16 value
// columns, contractions on warp-level tensor cores:
//   [K; Q] S            -> K S, Q S     bf16 MMAs, the state rounded to bf16 as an operand
//   Y = diag(beta) (V - diag(e^G) K S),  E = T Y,  T = (I + R)^{-1}      tf32 MMAs
//     (the page's order: provisional errors of all tokens, then the unit-lower solve)
//   O = s (diag(e^G) Q S + A E)                                          tf32 MMAs
//   S' = e^{G_end} S + K^T diag(e^{G_end - G}) E   bf16 MMAs into the fp32 state accumulators
// with G the in-call prefix of log alpha, R_im = beta_i e^{G_i - G_m} k_i . k_m (m < i) and
// A_im = e^{G_i - G_m} q_i . k_m (m <= i) from K K^T and Q K^T (bf16 MMAs); warp 0 forms R, A and
// T (substitution) while the other warps form Y, and hands them over on a named barrier. The
// state is read once from shared memory into the fp32 accumulators of the last contraction; each
// warp then writes its columns back as bf16 over the consumed fp32 words (8 consecutive keys of
// one 8-column tile land in distinct banks), so the buffer is released after the first
// contraction and the next head's state and tokens stream in while this head finishes (k, read by
// the last contraction, is double-buffered). Tokens are padded to 8 (T <= 8: one 16-row tile holds
// K in rows 0-7 and Q in rows 8-15) or 16.
namespace ttc {
constexpr int kThreads = 256;
constexpr int kPs = 136;   // fp32 state row pitch (words)
constexpr int kPb = 136;   // bf16 k / q / e_end . E row pitch (elements): conflict-free ldmatrix
constexpr int kPe = 136;   // fp32 Y / E row pitch: tf32 B fragments (rows q, columns g) hit banks 8q + g
constexpr int kMp = 17;    // 16 x 16 matrices
constexpr int kOffS = 0;                                  // state [128][kPs] f32
constexpr int kOffK = kOffS + 128 * kPs * 4;              // k [2][16][kPb] bf16 (double-buffered)
constexpr int kOffQ = kOffK + 2 * 16 * kPb * 2;           // q [16][kPb] bf16
constexpr int kOffV = kOffQ + 16 * kPb * 2;               // v [16][128] bf16
constexpr int kOffE = kOffV + 16 * 128 * 2;               // Y, then E [16][kPe] f32
constexpr int kOffEc = kOffE + 16 * kPe * 4;              // e_end . E [16][kPb] bf16
constexpr int kOffM = kOffEc + 16 * kPb * 2;              // R, A, T [3][16][kMp] f32
constexpr int kOffVec = kOffM + 3 * 16 * kMp * 4;         // alpha, eta [2][16] f32
constexpr int kBytes = kOffVec + 2 * 16 * 4;
static_assert(kOffK % 16 == 0 && kOffQ % 16 == 0 && kOffV % 16 == 0 && kOffE % 16 == 0 && kOffEc % 16 == 0 &&
                  kOffM % 16 == 0 && kOffVec % 16 == 0,
              "16-byte aligned regions");
// Byte offset, within row `key` of the state buffer, of the bf16 copy of 8-column tile nt of the
// warp's 16 columns (the warp's 64-byte segment starts at column nb): keys 4..7 of every 8 are
// shifted by 16 bytes so that eight consecutive keys fall in distinct groups of four banks.
__device__ __forceinline__ int bf16_slot(int key, int nb, int nt) {
    return key * kPs * 4 + nb * 4 + 16 * ((key >> 2) & 1) + 16 * nt;
}
}  // namespace ttc

template <int KT>   // 8-token steps over the padded tokens: 1 (T <= 8) or 2
__global__ void __launch_bounds__(ttc::kThreads, 2) tokens_tc_kernel(const TokParams p) {
    using namespace wmma16;
    typedef __nv_bfloat16 bf16;
    constexpr int DK = 128, DV = 128, MP = ttc::kMp;
    extern __shared__ __align__(16) unsigned char dsm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, q4 = lane & 3;
    const int T = p.T, nheads = p.B * p.H, nb = 16 * warp;
    float *sS = reinterpret_cast<float *>(dsm + ttc::kOffS);
    bf16 *sk0 = reinterpret_cast<bf16 *>(dsm + ttc::kOffK), *sq = reinterpret_cast<bf16 *>(dsm + ttc::kOffQ),
         *sv = reinterpret_cast<bf16 *>(dsm + ttc::kOffV), *sEc = reinterpret_cast<bf16 *>(dsm + ttc::kOffEc);
    float *sE = reinterpret_cast<float *>(dsm + ttc::kOffE);
    float *sR = reinterpret_cast<float *>(dsm + ttc::kOffM), *sAm = sR + 16 * MP, *sT = sAm + 16 * MP;
    float *sal = reinterpret_cast<float *>(dsm + ttc::kOffVec), *seta = sal + 16;
    const uint32_t sS_u32 = sptr(sS);
    const unsigned full = 0xffffffffu;

    auto row_of = [&](int head) {   // [B, T, H] row of the head's first token
        const int b = head / p.H, h = head - b * p.H;
        return static_cast<size_t>(b) * T * p.H + h;
    };
    auto prefetch = [&](int head, int kbuf) {   // the state; 16 rows of k, q, v (zero beyond T); alpha, eta
        if (p.S0) {
            const float *Sg = p.S0 + static_cast<size_t>(head) * DK * DV;
            for (int c = tid; c < DK * (DV / 4); c += ttc::kThreads) {
                const int row = c >> 5, ch = c & 31;
                cp_async16(sS + row * ttc::kPs + ch * 4, Sg + row * DV + ch * 4);
            }
        } else {
            for (int c = tid; c < DK * (DV / 4); c += ttc::kThreads) {
                const int row = c >> 5, ch = c & 31;
                *reinterpret_cast<float4 *>(sS + row * ttc::kPs + ch * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        const size_t row0 = row_of(head);
        const int u = tid >> 4, ch = tid & 15;
        bf16 *dk = sk0 + (kbuf * 16 + u) * ttc::kPb + ch * 8, *dq = sq + u * ttc::kPb + ch * 8,
             *dv = sv + u * DV + ch * 8;
        if (u < T) {
            const size_t r = row0 + static_cast<size_t>(u) * p.H;
            cp_async16(dk, static_cast<const bf16 *>(p.k) + r * DK + ch * 8);
            cp_async16(dq, static_cast<const bf16 *>(p.q) + r * DK + ch * 8);
            cp_async16(dv, static_cast<const bf16 *>(p.v) + r * DV + ch * 8);
        } else {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(dk) = z;
            *reinterpret_cast<uint4 *>(dq) = z;
            *reinterpret_cast<uint4 *>(dv) = z;
        }
        if (tid < 16) {
            if (tid < T) cp_async4(sal + tid, p.alpha + row0 + static_cast<size_t>(tid) * p.H);
            else sal[tid] = 1.f;
        } else if (tid < 32) {
            const int t = tid - 16;
            if (t < T) cp_async4(seta + t, p.eta + row0 + static_cast<size_t>(t) * p.H);
            else seta[t] = 0.f;
        }
    };

    // e_end . E rows T..15 stay zero for the whole launch (rows 8..15 are never written when T <= 8)
    for (int c = tid; c < 16 * ttc::kPb / 2; c += ttc::kThreads) reinterpret_cast<uint32_t *>(sEc)[c] = 0u;
    if (static_cast<int>(blockIdx.x) < nheads) prefetch(blockIdx.x, 0);
    cp_async_commit();
    int kbuf = 0;
    for (int head = blockIdx.x; head < nheads; head += gridDim.x, kbuf ^= 1) {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();   // (0) the head's state and tokens are visible
        const bf16 *sk = sk0 + kbuf * 16 * ttc::kPb;
        const size_t row0 = row_of(head);

        // (1) warp 1: K K^T into sR, warp 2: Q K^T into sAm; every warp: its state columns into the
        // fp32 accumulators of the last contraction, back as bf16, then [K; Q] S; then the gates,
        // step sizes and the thread's values of V into registers
        if (warp == 1 || warp == 2) {
            float acc[2][4] = {};
            const bf16 *sa = warp == 1 ? sk : sq;
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks) {
                uint32_t a[4], b[4];
                frag_a_rk(sptr(sa), ttc::kPb, 0, 16 * ks, lane, a);
                frag_b_rk(sptr(sk), ttc::kPb, 0, 16 * ks, lane, b);
                mma(acc[0], a, b[0], b[1]);
                mma(acc[1], a, b[2], b[3]);
            }
            float *dst = warp == 1 ? sR : sAm;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    dst[(g + 8 * hh) * MP + 8 * nt + 2 * q4] = acc[nt][2 * hh];
                    dst[(g + 8 * hh) * MP + 8 * nt + 2 * q4 + 1] = acc[nt][2 * hh + 1];
                }
        }
        float sacc[8][2][4];   // rows (keys) 16 mt + g (+ 8), columns nb + 8 nt + 2 q4 (+ 1)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float *r = sS + (16 * mt + g) * ttc::kPs + nb + 8 * nt + 2 * q4;
                const float2 x = *reinterpret_cast<const float2 *>(r), y = *reinterpret_cast<const float2 *>(r + 8 * ttc::kPs);
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
                    *reinterpret_cast<uint32_t *>(dsm + ttc::bf16_slot(key, nb, nt) + 4 * q4) =
                        pack2(sacc[mt][nt][2 * hh], sacc[mt][nt][2 * hh + 1]);
                }
        __syncwarp();
        float pacc[KT][2][4] = {};   // [K or Q tile][n tile]; for T <= 8 tile 0 holds K S (rows g) and Q S (rows g + 8)
        {
            const int m = lane >> 3, r = lane & 7;
            // B fragments (ldmatrix.trans): matrix m = (k half m & 1, n tile m >> 1), row r = key
            const uint32_t bbase = sS_u32 + ttc::bf16_slot(8 * (m & 1) + r, nb, m >> 1);
            // A fragments for T <= 8: matrices (K rows, k lo), (Q rows, k lo), (K, k hi), (Q, k hi)
            const uint32_t abase =
                sptr((m & 1) ? sq : sk) + 2 * (r * ttc::kPb + 8 * (m >> 1));
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks) {
                uint32_t b[4];
                ldsm4t(bbase + 16 * ks * ttc::kPs * 4, b);
                if constexpr (KT == 1) {
                    uint32_t a[4];
                    ldsm4(abase + 2 * 16 * ks, a);
                    mma(pacc[0][0], a, b[0], b[1]);
                    mma(pacc[0][1], a, b[2], b[3]);
                } else {
                    uint32_t ak[4], aq[4];
                    frag_a_rk(sptr(sk), ttc::kPb, 0, 16 * ks, lane, ak);
                    frag_a_rk(sptr(sq), ttc::kPb, 0, 16 * ks, lane, aq);
                    mma(pacc[0][0], ak, b[0], b[1]);
                    mma(pacc[0][1], ak, b[2], b[3]);
                    mma(pacc[KT - 1][0], aq, b[0], b[1]);
                    mma(pacc[KT - 1][1], aq, b[2], b[3]);
                }
            }
        }
        const float al = lane < 16 ? sal[lane] : 1.f, et = lane < 16 ? seta[lane] : 0.f;
        float2 vv[2][2];   // [row half hh][n tile]: V[g + 8 hh][nb + 8 nt + 2 q4 + (0, 1)]
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                vv[hh][nt] = __bfloat1622float2(
                    *reinterpret_cast<const __nv_bfloat162 *>(sv + (g + 8 * hh) * DV + nb + 8 * nt + 2 * q4));
        __syncthreads();   // (1) the state, q, v, alpha and eta buffers are free: the next head streams in
        if (head + static_cast<int>(gridDim.x) < nheads) prefetch(head + gridDim.x, kbuf ^ 1);
        cp_async_commit();

        // (2) every warp: G (prefix of log alpha over the tokens) and beta by lane
        float G = lane < T ? fmaxf(logf(al), kMinLogGateDecode) : 0.f;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            const float y = __shfl_up_sync(full, G, o);
            if (lane >= o) G += y;
        }
        const float n2 = lane < 16 ? sR[lane * MP + lane] : 0.f;
        const float beta = lane < T ? kla_beta(et, n2, p.eps, p.beta_raw) : 0.f;
        const float Gend = __shfl_sync(full, G, T - 1);
        const float G0 = __shfl_sync(full, G, g), G1 = __shfl_sync(full, G, g + 8);
        const float b0 = __shfl_sync(full, beta, g), b1 = __shfl_sync(full, beta, g + 8);
        const float eG0 = __expf(G0), eG1 = __expf(G1);
        if (warp == 0) {
            // R and A in place (8 entries per lane; the diagonal of K K^T stays), then column
            // j = lane < 16 of T = (I + R)^{-1} by forward substitution
            const int i = lane >> 1;
            const float Gi = __shfl_sync(full, G, i), bi = __shfl_sync(full, beta, i);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int m = 8 * (lane & 1) + j;
                const float Gm = __shfl_sync(full, G, m);
                const float d = __expf(fminf(Gi - Gm, 0.f));
                if (m < i) sR[i * MP + m] *= bi * d;
                sAm[i * MP + m] = m <= i ? d * sAm[i * MP + m] : 0.f;
            }
            __syncwarp();
            if (lane < 16) {
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
            asm volatile("bar.arrive 1, 256;" ::: "memory");   // T and A are ready
        }
        // (3) per warp on its 16 columns: Y = diag(beta) (V - diag(e^G) K S) into sE
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            if (hh == 0 || KT == 2) {
                const int u = g + 8 * hh;
                const float bu = hh ? b1 : b0, eu = hh ? eG1 : eG0;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    *reinterpret_cast<float2 *>(sE + u * ttc::kPe + nb + 8 * nt + 2 * q4) =
                        make_float2(bu * (vv[hh][nt].x - eu * pacc[0][nt][2 * hh]),
                                    bu * (vv[hh][nt].y - eu * pacc[0][nt][2 * hh + 1]));
            }
        }
        if (warp != 0) asm volatile("bar.sync 1, 256;" ::: "memory");
        __syncwarp();
        // (4) E = T Y (tf32 MMAs over the tokens); E in place of Y, e_end . E as bf16
        float eacc[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < KT; ++ks) {
            const int k0 = 8 * ks;
            const uint32_t a[4] = {tf32(sT[g * MP + k0 + q4]), tf32(sT[(g + 8) * MP + k0 + q4]),
                                   tf32(sT[g * MP + k0 + q4 + 4]), tf32(sT[(g + 8) * MP + k0 + q4 + 4])};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                mma_tf32(eacc[nt], a, tf32(sE[(k0 + q4) * ttc::kPe + nb + 8 * nt + g]),
                         tf32(sE[(k0 + q4 + 4) * ttc::kPe + nb + 8 * nt + g]));
        }
        __syncwarp();
        {
            const float ee0 = __expf(Gend - G0), ee1 = __expf(Gend - G1);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (hh == 0 || KT == 2) {
                    const int u = g + 8 * hh;
                    const float s = hh ? ee1 : ee0;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int col = nb + 8 * nt + 2 * q4;
                        *reinterpret_cast<float2 *>(sE + u * ttc::kPe + col) =
                            make_float2(eacc[nt][2 * hh], eacc[nt][2 * hh + 1]);
                        *reinterpret_cast<uint32_t *>(sEc + u * ttc::kPb + col) =
                            pack2(s * eacc[nt][2 * hh], s * eacc[nt][2 * hh + 1]);
                    }
                }
            }
        }
        __syncwarp();
        // (5) O = s (diag(e^G) Q S + A E)
        {
            float oacc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                if constexpr (KT == 1) {
                    oacc[nt][0] = eG0 * pacc[0][nt][2]; oacc[nt][1] = eG0 * pacc[0][nt][3];
                    oacc[nt][2] = 0.f; oacc[nt][3] = 0.f;
                } else {
                    oacc[nt][0] = eG0 * pacc[KT - 1][nt][0]; oacc[nt][1] = eG0 * pacc[KT - 1][nt][1];
                    oacc[nt][2] = eG1 * pacc[KT - 1][nt][2]; oacc[nt][3] = eG1 * pacc[KT - 1][nt][3];
                }
            }
#pragma unroll
            for (int ks = 0; ks < KT; ++ks) {
                const int k0 = 8 * ks;
                const uint32_t a[4] = {tf32(sAm[g * MP + k0 + q4]), tf32(sAm[(g + 8) * MP + k0 + q4]),
                                       tf32(sAm[g * MP + k0 + q4 + 4]), tf32(sAm[(g + 8) * MP + k0 + q4 + 4])};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    mma_tf32(oacc[nt], a, tf32(sE[(k0 + q4) * ttc::kPe + nb + 8 * nt + g]),
                             tf32(sE[(k0 + q4 + 4) * ttc::kPe + nb + 8 * nt + g]));
            }
            bf16 *og = static_cast<bf16 *>(p.o);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int u = g + 8 * hh;
                if (u < T) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        *reinterpret_cast<__nv_bfloat162 *>(og + (row0 + static_cast<size_t>(u) * p.H) * DV + nb + 8 * nt + 2 * q4) =
                            __floats2bfloat162_rn(p.q_scale * oacc[nt][2 * hh], p.q_scale * oacc[nt][2 * hh + 1]);
                }
            }
        }
        // (6) S' = e^{G_end} S + K^T (e_end . E): bf16 MMAs over 16 tokens (rows beyond T are zero)
        {
            const float Gam = __expf(Gend);
            const float2 g2 = make_float2(Gam, Gam);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float2 lo = __fmul2_rn(g2, make_float2(sacc[mt][nt][0], sacc[mt][nt][1]));
                    const float2 hi = __fmul2_rn(g2, make_float2(sacc[mt][nt][2], sacc[mt][nt][3]));
                    sacc[mt][nt][0] = lo.x; sacc[mt][nt][1] = lo.y; sacc[mt][nt][2] = hi.x; sacc[mt][nt][3] = hi.y;
                }
            uint32_t b[4];
            frag_b_kr(sptr(sEc), ttc::kPb, nb, 0, lane, b);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                uint32_t a[4];
                frag_a_kr(sptr(sk), ttc::kPb, 16 * mt, 0, lane, a);
                mma(sacc[mt][0], a, b[0], b[1]);
                mma(sacc[mt][1], a, b[2], b[3]);
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
        // the next head's first barrier orders this head's reads of k, E, e_end . E and the
        // matrices before they are rewritten
    }
}

TokParams tok_params(const ChunkArgs &a) {
    const int esz = a.dtype == KLA_DTYPE_BF16 ? 2 : 4;
    auto up16 = [](int x) { return (x + 15) & ~15; };
    TokParams p{a.q, a.k, a.v, a.alpha, a.eta, a.eps, a.S0, a.S_T, a.o, a.B, a.T, a.H, a.d_k, a.d_v,
                a.beta_raw, a.q_scale, 0, 0, 0, 0, 0, 0};
    p.s_bytes = a.d_k * 32 * 4;
    p.off_kq = 0;
    p.off_v = up16(a.T * 2 * a.d_k * esz);
    p.off_a = up16(p.off_v + a.T * 32 * esz);
    p.off_e = up16(p.off_a + a.T * (a.gate == KLA_GATE_CHANNEL ? a.d_k : 1) * 4);
    p.stage_bytes = up16(p.off_e + a.T * 4);
    return p;
}

template <typename TIn, bool kChannel>
cudaError_t launch_tokens_t(const ChunkArgs &a) {
    // Looked up once per device (and token count): the shared-memory limit (set for the largest
    // stage, T = kShortSeqMaxT and d_k = 128), the SM count and the resident CTAs per SM, so a
    // launch costs no more host time than the single-token step's.
    static bool attr_set[64] = {};
    static int sms_of[64] = {};
    static int per_sm[64][kShortSeqMaxT + 1] = {};
    const TokParams p = tok_params(a);
    const int smem = p.s_bytes + 2 * p.stage_bytes;
    auto kern = tokens_pipe_kernel<TIn, kChannel>;
    constexpr int kThreads = kTokThreads;
    int dev = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        ChunkArgs big = a;
        big.T = kShortSeqMaxT;
        big.d_k = 128;
        const TokParams pb = tok_params(big);
        const int max_smem = pb.s_bytes + 2 * pb.stage_bytes;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem)) != cudaSuccess)
            return e;
        attr_set[dev] = true;
    }
    if (sms_of[dev] == 0 &&
        (e = cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    int &n = per_sm[dev][a.T];
    if (n == 0) {
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem)) != cudaSuccess) return e;
        n = std::max(1, n);
    }
    const int ntiles = (a.d_v / 32) * a.H * a.B;
    const int grid = std::min(ntiles, n * sms_of[dev]);
    kern<<<grid, kThreads, smem, a.stream>>>(p, ntiles);
    return cudaGetLastError();
}

// The chunk-form kernel for bf16 / scalar gate / d_v = 128 from 5 tokens up (measured on GB300
// at 64 x 16 heads: 31.4 us for T <= 8 and 35.5 us for T <= 16, against 31.4, 47.7 and 80.5 us
// of the token loop at T = 4, 8 and 16). q, k, v and o are 16-byte aligned here.
bool tokens_tc_preferred(const ChunkArgs &a) {
    return a.dtype == KLA_DTYPE_BF16 && a.gate == KLA_GATE_SCALAR && a.d_k == 128 && a.d_v == 128 && a.T >= 5;
}

cudaError_t launch_tokens_tc(const ChunkArgs &a) {
    // Cached per device: the shared-memory limit, the SM count and the resident CTAs per SM.
    static bool attr_set[64] = {};
    static int sms_of[64] = {}, per_sm[64] = {};
    const TokParams p = tok_params(a);
    int dev = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        if ((e = cudaFuncSetAttribute(tokens_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, ttc::kBytes)) !=
                cudaSuccess ||
            (e = cudaFuncSetAttribute(tokens_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, ttc::kBytes)) !=
                cudaSuccess)
            return e;
        attr_set[dev] = true;
    }
    if (sms_of[dev] == 0 &&
        (e = cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if (per_sm[dev] == 0) {
        int n = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tokens_tc_kernel<2>, ttc::kThreads, ttc::kBytes)) !=
            cudaSuccess)
            return e;
        per_sm[dev] = std::max(1, n);
    }
    const int nheads = a.B * a.H;
    const int grid = std::min(nheads, per_sm[dev] * sms_of[dev]);
    if (a.T <= 8) tokens_tc_kernel<1><<<grid, ttc::kThreads, ttc::kBytes, a.stream>>>(p);
    else tokens_tc_kernel<2><<<grid, ttc::kThreads, ttc::kBytes, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool tokens_pipe_supports(const ChunkArgs &a) {
    auto al = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
    return a.T >= 1 && a.T <= kShortSeqMaxT && a.d_v % 32 == 0 && a.d_k == 128 &&
           al(a.q) && al(a.k) && al(a.v) && (!a.S0 || al(a.S0)) && (!a.S_T || al(a.S_T)) &&
           (a.gate == KLA_GATE_SCALAR || al(a.alpha));
}

cudaError_t launch_tokens_pipe(const ChunkArgs &a) {
    const bool ch = a.gate == KLA_GATE_CHANNEL;
    if (a.dtype == KLA_DTYPE_BF16)
        return ch ? (tokens_ch_supports(a) ? launch_tokens_ch(a) : launch_tokens_t<__nv_bfloat16, true>(a))
                  : tokens_tc_preferred(a) ? launch_tokens_tc(a) : launch_tokens_t<__nv_bfloat16, false>(a);
    return ch ? launch_tokens_t<float, true>(a) : launch_tokens_t<float, false>(a);
}

cudaError_t launch_decode(const DecodeArgs &a) {
    const bool ch = a.gate == KLA_GATE_CHANNEL;
    if (a.dtype == KLA_DTYPE_BF16)
        return ch ? launch_t<__nv_bfloat16, true>(a) : launch_t<__nv_bfloat16, false>(a);
    return ch ? launch_t<float, true>(a) : launch_t<float, false>(a);
}

}  // namespace kla
