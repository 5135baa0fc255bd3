// kla_short.cu -- short sequences (multi-token decode, speculative verification): T <= 16.
//
// For a handful of new tokens the chunk algebra does not pay: the state tile is read once into
// registers, the tokens are walked in order with the fused single-token step (GeekNews,
// "Revisando las variantes de atencion lineal de la familia DeltaNet", section "Kernel Triton
// recurrente fusionado para decodificacion"; step size from the KLA page, section "La Regola
// di Aggiornamento KLA"), and the tile is written once. Per token,
//   S~ = alpha (.) S;  e = v - S~^T k;  beta = eta / (||k||^2 + eps);  S = S~ + beta k e^T;
//   o = S~^T q + beta e (k . q)   (= S^T q, the read after the write).
// Grid: one CTA of 128 threads per (32-column value tile, head, sequence); every thread keeps
// up to 8 float4 of the d_k x 32 tile. All tokens' q, k, v, gates and step sizes are staged in
// shared memory once, together with the state loads, so the token loop waits on no global
// load. All arithmetic is fp32.
#include <algorithm>

#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr int kThreads = 128;

struct ShortParams {
    const void *q, *k, *v;
    const float *alpha, *eta;
    float eps;
    const float *S0;
    void *o;
    float *S_T;
    int B, T, H, DK, DV;
};

// CGW = float4 column groups per warp (2 for a 32-column tile, 1 for 16 columns). A warp owns
// CGW * 4 columns over ALL d_k rows, so the reductions over the rows stay inside the warp and
// the token loop runs without block barriers; lanes split as CGW column groups x (32 / CGW)
// row groups, each lane holding kRows consecutive rows (kRows = d_k / row groups, at least 1;
// lanes past d_k hold nothing when d_k is below the row-group count).
template <int kRows>
__device__ __forceinline__ void rows_from_smem(const float *src, float (&dst)[kRows]) {
    if constexpr (kRows % 4 == 0) {
#pragma unroll
        for (int r = 0; r < kRows; r += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(src + r);
            dst[r] = x.x; dst[r + 1] = x.y; dst[r + 2] = x.z; dst[r + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int r = 0; r < kRows; ++r) dst[r] = src[r];
    }
}

template <typename TIn, bool kChannel, int CGW, int kRows>
__global__ void __launch_bounds__(kThreads) short_seq_kernel(const ShortParams p) {
    constexpr int kWarps = kThreads / 32;
    constexpr int BV = kWarps * CGW * 4;          // columns per CTA
    __shared__ __align__(16) float sk[kShortSeqMaxT][128];
    __shared__ __align__(16) float sq[kShortSeqMaxT][128];
    __shared__ __align__(16) float sa[kChannel ? kShortSeqMaxT : 1][128];
    __shared__ __align__(16) float sv[kShortSeqMaxT][BV];
    __shared__ float sbeta[kShortSeqMaxT], skq[kShortSeqMaxT], sas[kShortSeqMaxT];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = lane % CGW, rg = lane / CGW;
    const int h = blockIdx.y, b = blockIdx.z;
    const int vt0 = blockIdx.x * BV;              // first column of the CTA's tile
    const int col = vt0 + warp * CGW * 4 + cg * 4;   // first of this lane's four columns
    const size_t bh = static_cast<size_t>(b) * p.H + h;
    const int DK = p.DK, T = p.T;
    const int r0 = rg * kRows;
    const bool live = r0 < DK;

    // 1. state rows of this lane (the long pole: issued first)
    float4 s[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        s[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && p.S0) s[r] = *reinterpret_cast<const float4 *>(p.S0 + (bh * DK + r0 + r) * p.DV + col);
    }

    // 2. every token's vectors into shared memory
    auto tok = [&](int t) { return (static_cast<size_t>(b) * T + t) * p.H + h; };
    const TIn *gk = static_cast<const TIn *>(p.k), *gq = static_cast<const TIn *>(p.q);
    for (int idx = tid; idx < T * DK; idx += kThreads) {
        const int t = idx / DK, c = idx - t * DK;
        const size_t g = tok(t) * DK + c;
        sk[t][c] = to_f32(gk[g]);
        sq[t][c] = to_f32(gq[g]);
        if (kChannel) sa[t][c] = p.alpha[g];
    }
    const TIn *gv = static_cast<const TIn *>(p.v);
    for (int idx = tid; idx < T * BV; idx += kThreads) {
        const int t = idx / BV, c = idx - t * BV;
        sv[t][c] = to_f32(gv[tok(t) * p.DV + vt0 + c]);
    }
    if (tid < T) {
        if (!kChannel) sas[tid] = p.alpha[tok(tid)];
        sbeta[tid] = p.eta[tok(tid)];   // eta for now; replaced by beta below
    }
    __syncthreads();
    // 3. ||k||^2, k.q and beta per token (one warp per token)
    for (int t = warp; t < T; t += kWarps) {
        float kk = 0.f, kq = 0.f;
        for (int c = lane; c < DK; c += 32) {
            kk = fmaf(sk[t][c], sk[t][c], kk);
            kq = fmaf(sk[t][c], sq[t][c], kq);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            kk += __shfl_xor_sync(0xffffffffu, kk, off);
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
        }
        if (lane == 0) {
            sbeta[t] = kla_beta(sbeta[t], kk, p.eps);
            skq[t] = kq;
        }
    }
    __syncthreads();

    // 4. the tokens, in order; no block barrier from here on
    for (int t = 0; t < T; ++t) {
        const float beta = sbeta[t], kdotq = skq[t];
        const float as = kChannel ? 1.f : sas[t];
        float kr[kRows], qr[kRows], ar[kRows];
        const int rr = live ? r0 : 0;   // lanes past d_k read row 0 and discard it
        rows_from_smem<kRows>(&sk[t][rr], kr);
        rows_from_smem<kRows>(&sq[t][rr], qr);
        if constexpr (kChannel) rows_from_smem<kRows>(&sa[t][rr], ar);
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            if (live) {
                const float a = kChannel ? ar[r] : as;
                const float ak = a * kr[r], aq = a * qr[r];
                pk.x = fmaf(ak, s[r].x, pk.x); pk.y = fmaf(ak, s[r].y, pk.y);
                pk.z = fmaf(ak, s[r].z, pk.z); pk.w = fmaf(ak, s[r].w, pk.w);
                pq.x = fmaf(aq, s[r].x, pq.x); pq.y = fmaf(aq, s[r].y, pq.y);
                pq.z = fmaf(aq, s[r].z, pq.z); pq.w = fmaf(aq, s[r].w, pq.w);
            }
        }
#pragma unroll
        for (int off = CGW; off < 32; off <<= 1) {
            pk.x += __shfl_xor_sync(0xffffffffu, pk.x, off); pk.y += __shfl_xor_sync(0xffffffffu, pk.y, off);
            pk.z += __shfl_xor_sync(0xffffffffu, pk.z, off); pk.w += __shfl_xor_sync(0xffffffffu, pk.w, off);
            pq.x += __shfl_xor_sync(0xffffffffu, pq.x, off); pq.y += __shfl_xor_sync(0xffffffffu, pq.y, off);
            pq.z += __shfl_xor_sync(0xffffffffu, pq.z, off); pq.w += __shfl_xor_sync(0xffffffffu, pq.w, off);
        }
        const float4 vt = *reinterpret_cast<const float4 *>(&sv[t][col - vt0]);
        float4 e;
        e.x = vt.x - pk.x; e.y = vt.y - pk.y; e.z = vt.z - pk.z; e.w = vt.w - pk.w;
        if (rg == 0) {   // o = S~^T q + beta e (k . q)
            TIn *o = static_cast<TIn *>(p.o) + tok(t) * p.DV + col;
            const float bkq = beta * kdotq;
            o[0] = from_f32<TIn>(fmaf(bkq, e.x, pq.x));
            o[1] = from_f32<TIn>(fmaf(bkq, e.y, pq.y));
            o[2] = from_f32<TIn>(fmaf(bkq, e.z, pq.z));
            o[3] = from_f32<TIn>(fmaf(bkq, e.w, pq.w));
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) {   // S = S~ + beta k e^T
            if (live) {
                const float a = kChannel ? ar[r] : as;
                const float bk = beta * kr[r];
                s[r].x = fmaf(a, s[r].x, bk * e.x); s[r].y = fmaf(a, s[r].y, bk * e.y);
                s[r].z = fmaf(a, s[r].z, bk * e.z); s[r].w = fmaf(a, s[r].w, bk * e.w);
            }
        }
    }
    if (p.S_T) {
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            if (live) *reinterpret_cast<float4 *>(p.S_T + (bh * DK + r0 + r) * p.DV + col) = s[r];
    }
}

template <typename TIn, bool kChannel, int CGW>
cudaError_t launch_rows(const ChunkArgs &a, const ShortParams &p, dim3 grid) {
    const int rows = std::max(1, a.d_k / (32 / CGW));
    switch (rows) {
        case 1: short_seq_kernel<TIn, kChannel, CGW, 1><<<grid, kThreads, 0, a.stream>>>(p); break;
        case 2: short_seq_kernel<TIn, kChannel, CGW, 2><<<grid, kThreads, 0, a.stream>>>(p); break;
        case 4: short_seq_kernel<TIn, kChannel, CGW, 4><<<grid, kThreads, 0, a.stream>>>(p); break;
        default: short_seq_kernel<TIn, kChannel, CGW, 8><<<grid, kThreads, 0, a.stream>>>(p); break;
    }
    return cudaGetLastError();
}

template <typename TIn, bool kChannel>
cudaError_t launch_t(const ChunkArgs &a) {
    const int BV = std::min(a.d_v, 32);   // d_v is 16, 32, 64 or 128
    ShortParams p{a.q, a.k, a.v, a.alpha, a.eta, a.eps, a.S0, a.o, a.S_T, a.B, a.T, a.H, a.d_k, a.d_v};
    dim3 grid(a.d_v / BV, a.H, a.B);
    return BV == 32 ? launch_rows<TIn, kChannel, 2>(a, p, grid) : launch_rows<TIn, kChannel, 1>(a, p, grid);
}

}  // namespace

bool short_seq_supports(const ChunkArgs &a) { return a.T >= 1 && a.T <= kShortSeqMaxT; }

cudaError_t launch_short_seq(const ChunkArgs &a) {
    const bool ch = a.gate == KLA_GATE_CHANNEL;
    if (a.dtype == KLA_DTYPE_BF16)
        return ch ? launch_t<__nv_bfloat16, true>(a) : launch_t<__nv_bfloat16, false>(a);
    return ch ? launch_t<float, true>(a) : launch_t<float, false>(a);
}

}  // namespace kla
