// kla_recurrent.cu -- the token-by-token recurrence with the state in registers: short sequences
// (multi-token decode, speculative verification) and every shape the tensor-core chunk path
// does not take (fp32 inputs, heads other than 128, chunk other than 64).
//
// The state tile is read once into registers, the tokens are walked in order with the fused
// single-token step (GeekNews, "Revisando las variantes de atencion lineal de la familia
// DeltaNet", section "Kernel Triton recurrente fusionado para decodificacion"; step size from the
// KLA page, section "La Regola di Aggiornamento KLA"), and the tile is written once. Per token,
//   S~ = alpha (.) S;  e = v - S~^T k;  beta = eta / (||k||^2 + eps);  S = S~ + beta k e^T;
//   o = S~^T q + beta e (k . q)   (= S^T q, the read after the write).
// Grid: one CTA of 128 threads per (32-column value tile, head, sequence); every thread keeps
// up to 8 float4 of the d_k x 32 tile. The q, k, v, gates and step sizes of 16 tokens at a time
// are staged in shared memory (the first block together with the state loads), so the token
// loop waits on no global load and has one block barrier per 16 tokens. All arithmetic is fp32,
// in the recurrence's own order: it is also the exact (fp32) path.
#include <algorithm>

#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr int kThreads = 128;

struct RecParams {
    const void *q, *k, *v;
    const float *alpha, *eta;
    float eps;
    const float *S0;
    void *o;
    float *S_T;
    int B, T, H, DK, DV;
    int beta_raw;
    float q_scale;
    const unsigned *only;   // when set, chains with only[b * H + h] == 0 return at once
};

// Lane layout. A warp owns CGW float4 column groups (CGW * 4 value columns) over ALL d_k rows,
// so the reductions over the rows stay inside the warp and the token loop runs without block
// barriers. Lane = cg + CGW * rg: CGW column groups x (32 / CGW) row groups, each row group
// holding kRows consecutive rows (kRows = d_k / row groups, at least 1; row groups past d_k
// hold nothing). CGW = 2 (32-column tiles) or 1 (16-column tiles, d_v = 16).
//
// The state tile passes through shared memory on its way in and out, so HBM sees whole 128-byte
// rows per warp access; its 16-byte units are XOR-swizzled by row group, which keeps the
// per-lane row reads free of bank conflicts.
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

__device__ __forceinline__ void prefetch_l2(const void *ptr) { asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr)); }

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Reduce 8 partial sums over the row-group lanes of one column group. The first three levels
// halve the values each lane carries (reduce-scatter), so 8 + the remaining levels shuffles
// replace 8 per level; afterwards the lane with (lane >> 2) & 7 == m holds the full sum m.
template <int CGW>
__device__ __forceinline__ float reduce_scatter8(const float (&x)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float y[4], z[2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // off 16: keep the half selected by lane bit 4
        const float send = b4 ? x[j] : x[j + 4];
        const float keep = b4 ? x[j + 4] : x[j];
        y[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {   // off 8
        const float send = b3 ? y[j] : y[j + 2];
        const float keep = b3 ? y[j + 2] : y[j];
        z[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float w;
    {                               // off 4
        const float send = b2 ? z[0] : z[1];
        const float keep = b2 ? z[1] : z[0];
        w = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int off = 2; off >= CGW; off >>= 1) w += __shfl_xor_sync(0xffffffffu, w, off);
    return w;
}

template <typename TIn, bool kChannel, int CGW, int kRows>
__global__ void __launch_bounds__(kThreads) recurrent_kernel(const RecParams p) {
    constexpr int kWarps = kThreads / 32;
    constexpr int BV = kWarps * CGW * 4;          // columns per CTA
    constexpr int U = BV / 4;                     // 16-byte units per tile row
    __shared__ __align__(16) float sk[kShortSeqMaxT][128];
    __shared__ __align__(16) float sq[kShortSeqMaxT][128];
    __shared__ __align__(16) float sa[kChannel ? kShortSeqMaxT : 1][128];
    __shared__ __align__(16) float sv[kShortSeqMaxT][BV];
    __shared__ __align__(16) float stile[128 * BV];
    __shared__ float sbeta[kShortSeqMaxT], skq[kShortSeqMaxT], sas[kShortSeqMaxT];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = lane % CGW, rg = lane / CGW;
    const int h = blockIdx.y, b = blockIdx.z;
    if (p.only && p.only[static_cast<size_t>(b) * p.H + h] == 0) return;
    const int vt0 = blockIdx.x * BV;              // first column of the CTA's tile
    const int ucol = warp * CGW + cg;             // this lane's 16-byte unit within a tile row
    const size_t bh = static_cast<size_t>(b) * p.H + h;
    const int DK = p.DK, T = p.T;
    const int r0 = rg * kRows;
    const bool live = r0 < DK;
    // swizzled float offset of unit u of tile row i
    auto tile_at = [&](int i, int u) { return i * BV + ((u ^ (((i / kRows) & 3) << 1)) & (U - 1)) * 4; };

    // 1. state tile -> shared memory, coalesced, asynchronous
    if (p.S0) {
        const float *src = p.S0 + bh * DK * p.DV + vt0;
        for (int idx = tid; idx < DK * U; idx += kThreads) {
            const int i = idx / U, u = idx - i * U;
            cp_async16(&stile[tile_at(i, u)], src + static_cast<size_t>(i) * p.DV + u * 4);
        }
    }

    // 2. the vectors of tokens [tb, tb + n) into shared memory (slots 0 .. n-1), then
    // 3. ||k||^2, k.q and beta per token (one warp per token)
    auto tok = [&](int t) { return (static_cast<size_t>(b) * T + t) * p.H + h; };
    const TIn *gk = static_cast<const TIn *>(p.k), *gq = static_cast<const TIn *>(p.q);
    const TIn *gv = static_cast<const TIn *>(p.v);
    auto stage = [&](int tb, int n) {
        for (int idx = tid; idx < n * DK; idx += kThreads) {
            const int t = idx / DK, c = idx - t * DK;
            const size_t g = tok(tb + t) * DK + c;
            sk[t][c] = to_f32(gk[g]);
            sq[t][c] = to_f32(gq[g]);
            if (kChannel) sa[t][c] = p.alpha[g];
        }
        for (int idx = tid; idx < n * BV; idx += kThreads) {
            const int t = idx / BV, c = idx - t * BV;
            sv[t][c] = to_f32(gv[tok(tb + t) * p.DV + vt0 + c]);
        }
        if (tid < n) {
            if (!kChannel) sas[tid] = p.alpha[tok(tb + tid)];
            sbeta[tid] = p.eta[tok(tb + tid)];   // eta for now; replaced by beta below
        }
        __syncthreads();
        for (int t = warp; t < n; t += kWarps) {
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
                sbeta[t] = kla_beta(sbeta[t], kk, p.eps, p.beta_raw);
                skq[t] = kq;
            }
        }
    };
    // the next block's k, q (and per-channel gates) and v, pulled into L2 while this block runs
    auto prefetch_block = [&](int tb, int n) {
        const int lines_k = (DK * static_cast<int>(sizeof(TIn)) + 127) / 128;
        const int lines_a = kChannel ? (DK * 4 + 127) / 128 : 0;
        const int per = 2 * lines_k + lines_a + 1;
        for (int idx = tid; idx < n * per; idx += kThreads) {
            const int t = idx / per, l = idx - t * per;
            const size_t tk = tok(tb + t);
            const char *ptr;
            if (l < lines_k) ptr = reinterpret_cast<const char *>(gk + tk * DK) + 128 * l;
            else if (l < 2 * lines_k) ptr = reinterpret_cast<const char *>(gq + tk * DK) + 128 * (l - lines_k);
            else if (l < 2 * lines_k + lines_a) ptr = reinterpret_cast<const char *>(p.alpha + tk * DK) + 128 * (l - 2 * lines_k);
            else ptr = reinterpret_cast<const char *>(gv + tk * p.DV + vt0);
            prefetch_l2(ptr);
        }
    };
    stage(0, min(T, kShortSeqMaxT));
    if (T > kShortSeqMaxT) prefetch_block(kShortSeqMaxT, min(kShortSeqMaxT, T - kShortSeqMaxT));
    cp_async_wait_all();
    __syncthreads();

    // 4. this lane's rows of the state, as float2 pairs (x, y) and (z, w) of its four columns
    float2 s[kRows][2];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && p.S0) x = *reinterpret_cast<const float4 *>(&stile[tile_at(r0 + r, ucol)]);
        s[r][0] = make_float2(x.x, x.y);
        s[r][1] = make_float2(x.z, x.w);
    }
    const int rr = live ? r0 : 0;   // lanes past d_k read row 0 and discard it

    // 5. the tokens, in order, kShortSeqMaxT at a time (one block barrier per block, none per token)
    for (int tb = 0; tb < T; tb += kShortSeqMaxT) {
        const int n = min(kShortSeqMaxT, T - tb);
        if (tb > 0) {
            __syncthreads();   // every lane is done with the previous block's vectors
            stage(tb, n);
            __syncthreads();
            if (tb + kShortSeqMaxT < T) prefetch_block(tb + kShortSeqMaxT, min(kShortSeqMaxT, T - tb - kShortSeqMaxT));
        }
        for (int t = 0; t < n; ++t) {
            const float beta = sbeta[t], kdotq = skq[t];
            const float as = kChannel ? 1.f : sas[t];
            float kr[kRows], qr[kRows], ar[kRows], kg[kRows];
            rows_from_smem<kRows>(&sk[t][rr], kr);
            rows_from_smem<kRows>(&sq[t][rr], qr);
#pragma unroll
            for (int r = 0; r < kRows; ++r) kg[r] = kr[r];
            if constexpr (kChannel) {
                rows_from_smem<kRows>(&sa[t][rr], ar);
#pragma unroll
                for (int r = 0; r < kRows; ++r) { kg[r] *= ar[r]; qr[r] *= ar[r]; }   // rows of alpha (.) k, q
            }
            // partial S~^T k and S~^T q over this lane's rows (for a scalar gate alpha is applied
            // after the reduction); packed fp32 FMAs over column pairs
            float2 pk0 = make_float2(0.f, 0.f), pk1 = pk0, pq0 = pk0, pq1 = pk0;
            if (live) {
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    const float2 kk2 = make_float2(kg[r], kg[r]), qq2 = make_float2(qr[r], qr[r]);
                    pk0 = __ffma2_rn(kk2, s[r][0], pk0); pk1 = __ffma2_rn(kk2, s[r][1], pk1);
                    pq0 = __ffma2_rn(qq2, s[r][0], pq0); pq1 = __ffma2_rn(qq2, s[r][1], pq1);
                }
            }
            const float part[8] = {pk0.x, pk0.y, pk1.x, pk1.y, pq0.x, pq0.y, pq1.x, pq1.y};
            const float red = reduce_scatter8<CGW>(part, lane) * as;   // full sum number (lane >> 2) & 7
            // every lane needs the four prediction sums of its column group
            const int src = lane & 3;
            float pred[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) pred[j] = __shfl_sync(0xffffffffu, red, (j << 2) | src);
            const float4 vt = *reinterpret_cast<const float4 *>(&sv[t][ucol * 4]);
            const float e[4] = {vt.x - pred[0], vt.y - pred[1], vt.z - pred[2], vt.w - pred[3]};
            const int m = (lane >> 2) & 7;
            if (m >= 4 && (lane & (3 & ~(CGW - 1))) == 0) {   // o = s (S~^T q + beta e (k . q))
                const int j = m - 4;
                const float ej = j == 0 ? e[0] : j == 1 ? e[1] : j == 2 ? e[2] : e[3];
                static_cast<TIn *>(p.o)[tok(tb + t) * p.DV + vt0 + ucol * 4 + j] =
                    from_f32<TIn>(p.q_scale * fmaf(beta * kdotq, ej, red));
            }
            // S = S~ + beta k e^T (lanes past d_k update rows they never store)
            const float2 e01 = make_float2(e[0], e[1]), e23 = make_float2(e[2], e[3]);
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const float a = kChannel ? ar[r] : as;
                const float bk = beta * kr[r];
                const float2 a2 = make_float2(a, a), bk2 = make_float2(bk, bk);
                s[r][0] = __ffma2_rn(a2, s[r][0], __fmul2_rn(bk2, e01));
                s[r][1] = __ffma2_rn(a2, s[r][1], __fmul2_rn(bk2, e23));
            }
        }
    }

    // 6. final state -> shared memory -> HBM, coalesced
    if (p.S_T) {
        __syncthreads();   // every lane's reads of the incoming tile are done
        if (live) {
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                *reinterpret_cast<float4 *>(&stile[tile_at(r0 + r, ucol)]) =
                    make_float4(s[r][0].x, s[r][0].y, s[r][1].x, s[r][1].y);
        }
        __syncthreads();
        float *dst = p.S_T + bh * DK * p.DV + vt0;
        for (int idx = tid; idx < DK * U; idx += kThreads) {
            const int i = idx / U, u = idx - i * U;
            *reinterpret_cast<float4 *>(dst + static_cast<size_t>(i) * p.DV + u * 4) =
                *reinterpret_cast<const float4 *>(&stile[tile_at(i, u)]);
        }
    }
}

template <typename TIn, bool kChannel, int CGW>
cudaError_t launch_rows(const ChunkArgs &a, const RecParams &p, dim3 grid) {
    const int rows = std::max(1, a.d_k / (32 / CGW));
    switch (rows) {
        case 1: recurrent_kernel<TIn, kChannel, CGW, 1><<<grid, kThreads, 0, a.stream>>>(p); break;
        case 2: recurrent_kernel<TIn, kChannel, CGW, 2><<<grid, kThreads, 0, a.stream>>>(p); break;
        case 4: recurrent_kernel<TIn, kChannel, CGW, 4><<<grid, kThreads, 0, a.stream>>>(p); break;
        default: recurrent_kernel<TIn, kChannel, CGW, 8><<<grid, kThreads, 0, a.stream>>>(p); break;
    }
    return cudaGetLastError();
}

template <typename TIn, bool kChannel>
cudaError_t launch_t(const ChunkArgs &a) {
    const int BV = std::min(a.d_v, 32);   // d_v is 16, 32, 64 or 128
    RecParams p{a.q, a.k, a.v, a.alpha, a.eta, a.eps, a.S0, a.o, a.S_T, a.B, a.T, a.H, a.d_k, a.d_v, a.beta_raw,
                  a.q_scale, a.only};
    dim3 grid(a.d_v / BV, a.H, a.B);
    return BV == 32 ? launch_rows<TIn, kChannel, 2>(a, p, grid) : launch_rows<TIn, kChannel, 1>(a, p, grid);
}

}  // namespace

bool recurrent_preferred(const ChunkArgs &a) {
    return a.T >= 1 && (a.T <= kShortSeqMaxT || !chunk_tc_supports(a));
}

cudaError_t launch_recurrent(const ChunkArgs &a) {
    const bool ch = a.gate == KLA_GATE_CHANNEL;
    if (a.dtype == KLA_DTYPE_BF16)
        return ch ? launch_t<__nv_bfloat16, true>(a) : launch_t<__nv_bfloat16, false>(a);
    return ch ? launch_t<float, true>(a) : launch_t<float, false>(a);
}

}  // namespace kla
