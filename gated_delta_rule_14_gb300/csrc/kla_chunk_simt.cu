// kla_chunk_simt.cu -- chunkwise KLA prefill on the CUDA cores, in fp32.
//
// The fp32 path: every storage type (fp32 or bf16 q/k/v), every supported head size and
// chunk length, scalar or per-key-channel gates. It is the path for fp32 inputs, where the
// tolerance leaves no room for bf16 tensor-core operands.
//
// Algebra (GeekNews, "Revisando las variantes de atencion lineal de la familia DeltaNet",
// section "KDA por chunks"), written in the d_k x d_v orientation of the KLA page. Per
// chunk with incoming state S and tokens i = 0..C-1:
//   G_i          in-chunk inclusive prefix of log-gates (per key channel for KDA)
//   beta_i       = eta_i / (||k_i||^2 + eps)                                   (KLA page)
//   R_ij (j<i)   = beta_i sum_c k_i[c] k_j[c] exp(G_i[c] - G_j[c])
//   A_ij (j<=i)  = sum_c q_i[c] k_j[c] exp(G_i[c] - G_j[c])
//   (I + R) W    = diag(beta) (exp(G) . K),   (I + R) U = diag(beta) V          (WY/UT form)
//   E            = U - W S                      (the corrected, beta-scaled errors)
//   O            = (exp(G) . Q) S + A E
//   S'           = exp(G_end) . S + K_end^T E,  K_end[j] = exp(G_end - G_j) . k_j
// Every exponent above is <= 0, so no factor overflows.
//
// Grid: one CTA per (value tile of <= 32 columns, head, sequence); the CTA walks the chunks
// of its sequence in order. Value columns of S evolve independently, so tiles need no
// communication; the d_k-side work (R, A, W) is recomputed per tile.
#include <algorithm>

#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr int kThreads = 256;
constexpr float kMinLogGate = -80.0f;   // a gate below e^-80 is indistinguishable from 0 in fp32

struct SimtParams {
    const void *q, *k, *v;
    const float *alpha, *eta;
    float eps;
    const float *S0;
    void *o;
    float *S_T;
    int B, T, H, DK, DV, C, BV;
    int beta_raw;
    float q_scale;
};

template <typename TIn, bool kChannel>
__global__ void __launch_bounds__(kThreads) chunk_simt_kernel(const SimtParams p) {
    extern __shared__ float4 smem_f4[];
    float *smem = reinterpret_cast<float *>(smem_f4);
    const int DK = p.DK, C = p.C, BV = p.BV;
    const int v0 = blockIdx.x * BV;
    const int h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;

    float *sK = smem;                    // [C][DK]
    float *sQ = sK + C * DK;             // [C][DK]
    float *sW = sQ + C * DK;             // [C][DK]  rhs, then W
    float *sG = sW + C * DK;             // [C][DK] (channel) or [C] (scalar)
    float *sU = sG + (kChannel ? C * DK : C);   // [C][BV] rhs, then U, then E
    float *sR = sU + C * BV;             // [C][C]
    float *sA = sR + C * C;              // [C][C]
    float *sS = sA + C * C;              // [DK][BV]
    float *sBeta = sS + DK * BV;         // [C]
    float *sEta = sBeta + C;             // [C]

    const TIn *q = static_cast<const TIn *>(p.q);
    const TIn *k = static_cast<const TIn *>(p.k);
    const TIn *v = static_cast<const TIn *>(p.v);
    TIn *o = static_cast<TIn *>(p.o);
    const size_t bh = static_cast<size_t>(b) * p.H + h;

    for (int idx = tid; idx < DK * BV; idx += kThreads) {
        const int ch = idx / BV, m = idx % BV;
        sS[idx] = p.S0 ? p.S0[(bh * DK + ch) * p.DV + v0 + m] : 0.0f;
    }

    const int nchunks = (p.T + C - 1) / C;
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * C;
        const int L = min(C, p.T - t0);
        __syncthreads();   // previous chunk fully consumed
        // ---- load the chunk (padded tokens are zero, gate 1, eta 0)
        for (int idx = tid; idx < C * DK; idx += kThreads) {
            const int i = idx / DK, ch = idx % DK;
            float kv = 0.f, qv = 0.f;
            if (i < L) {
                const size_t off = ((static_cast<size_t>(b) * p.T + t0 + i) * p.H + h) * DK + ch;
                kv = to_f32(k[off]);
                qv = to_f32(q[off]);
            }
            sK[idx] = kv;
            sQ[idx] = qv;
            if (kChannel) {
                float g = 0.f;
                if (i < L) g = fmaxf(logf(p.alpha[((static_cast<size_t>(b) * p.T + t0 + i) * p.H + h) * DK + ch]),
                                     kMinLogGate);
                sG[idx] = g;
            }
        }
        for (int idx = tid; idx < C * BV; idx += kThreads) {
            const int i = idx / BV, m = idx % BV;
            sU[idx] = (i < L) ? to_f32(v[((static_cast<size_t>(b) * p.T + t0 + i) * p.H + h) * p.DV + v0 + m]) : 0.f;
        }
        if (tid < C) {
            const size_t tok = (static_cast<size_t>(b) * p.T + t0 + tid) * p.H + h;
            sEta[tid] = (tid < L) ? p.eta[tok] : 0.f;
            if (!kChannel) sG[tid] = (tid < L) ? fmaxf(logf(p.alpha[tok]), kMinLogGate) : 0.f;
        }
        __syncthreads();
        // ---- prefix of log-gates, ||k||^2 and beta
        if (kChannel) {
            for (int ch = tid; ch < DK; ch += kThreads) {
                float acc = 0.f;
                for (int i = 0; i < C; ++i) { acc += sG[i * DK + ch]; sG[i * DK + ch] = acc; }
            }
        } else if (tid == 0) {
            float acc = 0.f;
            for (int i = 0; i < C; ++i) { acc += sG[i]; sG[i] = acc; }
        }
        if (tid >= 32 && tid < 32 + C) {
            const int i = tid - 32;
            float n2 = 0.f;
            for (int ch = 0; ch < DK; ++ch) n2 = fmaf(sK[i * DK + ch], sK[i * DK + ch], n2);
            sBeta[i] = kla_beta(sEta[i], n2, p.eps, p.beta_raw);
        }
        __syncthreads();
        // ---- R, A and the right-hand sides
        for (int idx = tid; idx < C * C; idx += kThreads) {
            const int i = idx / C, j = idx % C;
            float r = 0.f, a = 0.f;
            if (j <= i) {
                if (kChannel) {
                    for (int ch = 0; ch < DK; ++ch) {
                        const float dcy = expf(sG[i * DK + ch] - sG[j * DK + ch]);
                        const float kj = sK[j * DK + ch] * dcy;
                        r = fmaf(sK[i * DK + ch], kj, r);
                        a = fmaf(sQ[i * DK + ch], kj, a);
                    }
                } else {
                    for (int ch = 0; ch < DK; ++ch) {
                        r = fmaf(sK[i * DK + ch], sK[j * DK + ch], r);
                        a = fmaf(sQ[i * DK + ch], sK[j * DK + ch], a);
                    }
                    const float dcy = expf(sG[i] - sG[j]);
                    r *= dcy;
                    a *= dcy;
                }
                r = (j < i) ? r * sBeta[i] : 0.f;
            }
            sR[idx] = r;
            sA[idx] = a;
        }
        for (int idx = tid; idx < C * DK; idx += kThreads) {
            const int i = idx / DK;
            const float G = kChannel ? sG[idx] : sG[i];
            sW[idx] = sBeta[i] * expf(G) * sK[idx];
        }
        for (int idx = tid; idx < C * BV; idx += kThreads) sU[idx] *= sBeta[idx / BV];
        __syncthreads();
        // ---- unit-lower triangular solve (I + R) X = rhs, one thread per column of [W | U]
        for (int col = tid; col < DK + BV; col += kThreads) {
            float *X = col < DK ? sW + col : sU + (col - DK);
            const int ld = col < DK ? DK : BV;
            for (int i = 1; i < C; ++i) {
                float acc = X[i * ld];
                for (int j = 0; j < i; ++j) acc = fmaf(-sR[i * C + j], X[j * ld], acc);
                X[i * ld] = acc;
            }
        }
        __syncthreads();
        // ---- E = U - W S (in place in sU)
        for (int idx = tid; idx < C * BV; idx += kThreads) {
            const int i = idx / BV, m = idx % BV;
            float acc = sU[idx];
            for (int ch = 0; ch < DK; ++ch) acc = fmaf(-sW[i * DK + ch], sS[ch * BV + m], acc);
            sU[idx] = acc;
        }
        __syncthreads();
        // ---- O = s ((exp(G) . Q) S + A E)
        for (int idx = tid; idx < C * BV; idx += kThreads) {
            const int i = idx / BV, m = idx % BV;
            if (i >= L) continue;
            float acc = 0.f;
            for (int ch = 0; ch < DK; ++ch) {
                const float G = kChannel ? sG[i * DK + ch] : sG[i];
                acc = fmaf(expf(G) * sQ[i * DK + ch], sS[ch * BV + m], acc);
            }
            for (int j = 0; j <= i; ++j) acc = fmaf(sA[i * C + j], sU[j * BV + m], acc);
            o[((static_cast<size_t>(b) * p.T + t0 + i) * p.H + h) * p.DV + v0 + m] = from_f32<TIn>(p.q_scale * acc);
        }
        __syncthreads();
        // ---- S' = exp(G_end) . S + K_end^T E
        for (int idx = tid; idx < DK * BV; idx += kThreads) {
            const int ch = idx / BV, m = idx % BV;
            const float Gend = kChannel ? sG[(C - 1) * DK + ch] : sG[C - 1];
            float acc = expf(Gend) * sS[idx];
            for (int j = 0; j < L; ++j) {
                const float Gj = kChannel ? sG[j * DK + ch] : sG[j];
                acc = fmaf(expf(Gend - Gj) * sK[j * DK + ch], sU[j * BV + m], acc);
            }
            sS[idx] = acc;
        }
    }
    __syncthreads();
    if (p.S_T)
        for (int idx = tid; idx < DK * BV; idx += kThreads) {
            const int ch = idx / BV, m = idx % BV;
            p.S_T[(bh * DK + ch) * p.DV + v0 + m] = sS[idx];
        }
}

size_t simt_smem_bytes(int DK, int C, int BV, bool channel) {
    const size_t floats = 3ull * C * DK + (channel ? C * DK : C) + C * BV + 2ull * C * C + DK * BV + 2ull * C;
    return floats * sizeof(float);
}

template <typename TIn, bool kChannel>
cudaError_t launch_t(const ChunkArgs &a) {
    SimtParams p{a.q, a.k, a.v, a.alpha, a.eta, a.eps, a.S0, a.o, a.S_T,
                 a.B, a.T, a.H, a.d_k, a.d_v, a.chunk, std::min(a.d_v, 32), a.beta_raw, a.q_scale};
    const size_t smem = simt_smem_bytes(p.DK, p.C, p.BV, kChannel);
    cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel<TIn, kChannel>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(p.DV / p.BV, p.H, p.B);
    chunk_simt_kernel<TIn, kChannel><<<grid, kThreads, smem, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkArgs &a) {
    const bool ch = a.gate == KLA_GATE_CHANNEL;
    if (a.dtype == KLA_DTYPE_BF16)
        return ch ? launch_t<__nv_bfloat16, true>(a) : launch_t<__nv_bfloat16, false>(a);
    return ch ? launch_t<float, true>(a) : launch_t<float, false>(a);
}

}  // namespace kla
