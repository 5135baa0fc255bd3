// kla_bwd_carry_tc.cu -- the two chunk-state carries of the chunkwise backward on the tensor
// cores (tcgen05 with TMEM accumulators, operand tiles staged by TMA): the forward carry
// S_c -> S_{c+1} and the reverse carry dS_{c+1} -> dS_c of every (b, h) chain, one CTA per chain
// segment, chunks in order. They store the per-chunk records the gradient kernels read.
//
// The algebra is the chunk form of the forward and its reverse (GeekNews, "Revisando las
// variantes de atencion lineal de la familia DeltaNet", section "KDA por chunks"); with X the
// carried state (S forward, dS = dL/dS reverse), t a token, k a key and v a value channel,
// e_end = e^{G_end - G}, Gamma = e^{G_end}, s the query scale:
//   forward:  E  = U - W X,                       X' = Gamma X + (diag(e_end) K)^T E
//   reverse:  dE = diag(e_end) K X + s A^T dO,    X' = Gamma X + s (diag(e^G) Q)^T dO - W^T dE
// (per-key-channel gate: K and Q arrive as the prep's decayed records K_e and s Q_g, and Gamma is
// a diagonal e^{G_end} over the key channels of X's rows). Everything runs transposed so that the
// 128 value channels sit on the TMEM lanes (M = 128):
//   forward:  D1 = X^T W^T            (N = 64 tokens, K = 128)   -> E^T = U^T - D1
//             D2 = E^T K_e            (N = 128 keys,  K = 64)    -> X'^T = Gamma X^T + D2
//   reverse:  D1 = X^T K^T, D1b = dO^T A                          -> dE^T = e_end D1 + s D1b
//             D2 = dO^T Q_s, D2b = dE^T W                         -> X'^T = Gamma X^T + D2 - D2b
// X^T, E^T and dE^T enter as MN-major A operands from 128-byte-swizzled bf16 tiles whose layout
// is also that of the records ([k][v] and [t][v] row-major), so the same tiles leave by TMA
// store. K, W and A serve as K-major or MN-major B operands as they arrive. The carried state is
// fp32 in registers: thread (v, q) of the 16 warps holds X[k][v] for k in [32 q, 32 q + 32).
#include <cuda.h>

#include <mutex>

#include "kla_bwd_chunk.cuh"
#include "sm103_ptx.cuh"

namespace kla {
namespace bwdc {
namespace {

using namespace ptx;

constexpr int kThreads = 512;
constexpr uint32_t kTile = 16384;   // 64 rows x 128 bf16: two 64-column halves of 8 KB
constexpr uint32_t kHalf = 8192;
// One stage (chunk c, double-buffered): K | W | U (forward) or Q (reverse) | dO | A | gate vector.
constexpr uint32_t ST_K = 0, ST_W = kTile, ST_UQ = 2 * kTile, ST_DO = 3 * kTile, ST_A = 4 * kTile;
constexpr uint32_t ST_G = ST_A + kHalf;   // G of the chunk (64 fp32), or e^{G_end} per key channel (128 fp32)
constexpr uint32_t kStage = 73 * 1024;
constexpr uint32_t OFF_X = 2 * kStage;       // X^T, bf16 [v half][128 k][64 v]
constexpr uint32_t OFF_E = OFF_X + 2 * kTile;   // E^T or dE^T, bf16 [v half][64 t][64 v]
constexpr uint32_t OFF_KS = OFF_E + kTile;    // scalar gate: K_e (forward) or s diag(e^G) Q (reverse), [k half][64 t][64 k]
constexpr uint32_t OFF_BAR = OFF_KS + kTile;  // full[2], mma, TMEM base, abort flag
constexpr uint32_t kSmemBytes = OFF_BAR + 64 + 1024;   // + room to align the base to 1024 bytes
static_assert(ST_G + 4 * kD <= kStage && kSmemBytes <= 232448, "carry shared memory");
// TMEM columns: D1 | D1b | D2 | D2b
constexpr uint32_t TM_D1 = 0, TM_D1B = 64, TM_D2 = 128, TM_D2B = 256;

// Waits for phase `parity` of `bar` by polling (the waits of a step are short; this form also keeps
// the forward per-channel carry within its registers). Gives up after 2^31 clock cycles (about a
// second).
__device__ __forceinline__ bool wait_poll(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > (1ll << 31)) return false;
    return true;
}

template <bool kRev, bool kCh>
__global__ void __launch_bounds__(kThreads, 1)
carry_tc_kernel(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mW,
                const __grid_constant__ CUtensorMap mUQ, const __grid_constant__ CUtensorMap mDO,
                const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mXr,
                const __grid_constant__ CUtensorMap mEr, const ScanParams p) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int v = 32 * (warp & 3) + lane, q = warp >> 2;   // TMEM lane (value channel), key-channel quarter
    const int bh = blockIdx.x / p.seg_count, r = p.seg_begin + static_cast<int>(blockIdx.x) % p.seg_count;
    const int b = bh / p.H, h = bh % p.H;
    if (p.skip && p.skip[bh]) return;
    const int sidx = kRev ? p.nseg - 1 - r : r;   // segment index in time
    const int c_lo = sidx * p.seg_len, c_hi = min((sidx + 1) * p.seg_len, p.nc) - 1;
    const int steps = c_hi - c_lo + 1;
    if (steps <= 0) return;
    const bool rec = p.records == 1 || (p.records == 2 && r == 0);
    const bool drive = p.drive != 0;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + OFF_BAR, bar_mma = bar_full + 16;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + 24);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_BAR + 32);

    if (tid == 0) {
        mbar_init(bar_full, 1);
        mbar_init(bar_full + 8, 1);
        mbar_init(bar_mma, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&mK);
        prefetch_tmap(&mW);
        prefetch_tmap(&mUQ);
        if (kRev) {
            prefetch_tmap(&mDO);
            prefetch_tmap(&mA);
        }
        prefetch_tmap(&mXr);
        prefetch_tmap(&mEr);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), 512);
        tmem_relinquish();
    }

    // X^T in registers: X[j] = X[k][v], k = 32 q + j
    float X[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int k = 32 * q + j;
        float x = 0.f;
        if (p.x0_mode == kX0Identity) x = k == v ? 1.f : 0.f;
        else if (p.x0_mode == kX0Given) x = p.Xst[((static_cast<size_t>(bh) * p.nseg + r) * kD + k) * kD + v];
        else if (p.X0 && r == 0) x = p.X0[(static_cast<size_t>(bh) * kD + k) * kD + v];
        X[j] = x;
    }
    // bf16 X^T tile (MN-major A operand and the state record): element (k, v) of this thread's
    // 64-channel column block; the E^T / dE^T tile likewise, element (t, v)
    unsigned short *xcol = reinterpret_cast<unsigned short *>(smem + OFF_X + (v >> 6) * kTile);
    unsigned short *ecol = reinterpret_cast<unsigned short *>(smem + OFF_E + (v >> 6) * kHalf);
    const uint32_t vb = (v & 63) * 2;
    auto put_x = [&]() {
#pragma unroll
        for (int j = 0; j < 32; ++j) xcol[sw128_off(32 * q + j, vb) >> 1] = bf16_bits(X[j]);
        fence_proxy_async_smem();
    };
    put_x();

    // chunk c's tiles into stage s (warp 0, one lane)
    auto issue = [&](int c, int s) {
        const uint32_t st = sbase + s * kStage, bar = bar_full + 8 * s;
        const int n64 = (bh * p.nc + c) * kC, t0 = c * kC;
        uint32_t bytes = 2 * kTile + (kCh ? kD * 4 : kC * 4);
        if (drive) bytes += kRev ? 2 * kTile + kHalf : kTile;
        mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            if (kCh) tma_load_2d(st + ST_K + hh * kHalf, &mK, bar, 64 * hh, n64);
            else tma_load_4d(st + ST_K + hh * kHalf, &mK, bar, 64 * hh, h, t0, b);
            tma_load_2d(st + ST_W + hh * kHalf, &mW, bar, 64 * hh, n64);
            if (drive) {
                if (!kRev || kCh) tma_load_2d(st + ST_UQ + hh * kHalf, &mUQ, bar, 64 * hh, n64);
                else tma_load_4d(st + ST_UQ + hh * kHalf, &mUQ, bar, 64 * hh, h, t0, b);
                if (kRev) tma_load_4d(st + ST_DO + hh * kHalf, &mDO, bar, 64 * hh, h, t0, b);
            }
        }
        if (kRev && drive) tma_load_2d(st + ST_A, &mA, bar, 0, n64);
        const size_t n = static_cast<size_t>(bh) * p.nc + c;
        if (kCh) bulk_load(st + ST_G, p.ws.gend + n * kD, kD * 4, bar);
        else bulk_load(st + ST_G, p.ws.cg + n * kCgFloats, kC * 4, bar);
    };

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t tl = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t id_n64 = idesc_bf16(128, 64, 1, 0);    // MN-major A, K-major B, N = 64
    const uint32_t id_n64t = idesc_bf16(128, 64, 1, 1);   // MN-major A and B, N = 64
    const uint32_t id_n128 = idesc_bf16(128, 128, 1, 1);  // MN-major A and B, N = 128
    if (warp == 0) {
        if (elect_one()) issue(kRev ? c_hi : c_lo, 0);
        __syncwarp();
    }

    uint32_t mma_par = 0;
    bool ok = true;
    for (int it = 0; it < steps; ++it) {
        const int c = kRev ? c_hi - it : c_lo + it, s = it & 1;
        const int n = bh * p.nc + c;
        const uint32_t st = sbase + s * kStage;
        const float *gv = reinterpret_cast<const float *>(smem + s * kStage + ST_G);
        // the stage s ^ 1 held chunk it - 1: its products and readers finished in that step
        if (warp == 0) {
            if (it + 1 < steps && elect_one()) issue(kRev ? c - 1 : c + 1, s ^ 1);
            __syncwarp();
        }
        ok = wait_poll(bar_full + 8 * s, (it >> 1) & 1);
        if (!ok) *abort_flag = 1;
        // the state record (S_c, or dS_{c+1} in reverse; thread 32 owns every record store and
        // waits for them) and the first products (warp 0)
        if (tid == 32 && ok && rec) {
            tma_store_2d(&mXr, sbase + OFF_X, 0, n * kD);
            tma_store_2d(&mXr, sbase + OFF_X + kTile, 64, n * kD);
            tma_store_commit();
        }
        if (warp == 0) {
            const bool wok = __all_sync(0xffffffffu, ok);
            if (wok && elect_one()) {
                tc_fence_after();
                const uint64_t dx = sw128_desc(sbase + OFF_X, kTile, 1024);
                const uint64_t db = sw128_desc(st + (kRev ? ST_K : ST_W), 16, 1024);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tbase + TM_D1, desc_add(dx, ks * 2048), desc_add(db, (ks >> 2) * kHalf + (ks & 3) * 32),
                             id_n64, ks);
                if (kRev && drive) {
                    const uint64_t ddo = sw128_desc(st + ST_DO, kHalf, 1024), da = sw128_desc(st + ST_A, kHalf, 1024);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tbase + TM_D1B, desc_add(ddo, ks * 2048), desc_add(da, ks * 2048), id_n64t, ks);
                }
                mma_commit(bar_mma);
            }
            __syncwarp();
        }
        // scalar gate: the decayed copy the second products read (K_e forward, s e^G Q reverse);
        // both tiles share one swizzled layout, so 16-byte granules copy in place
        if (!kCh && (!kRev || drive)) {
            const uint8_t *src = smem + s * kStage + (kRev ? ST_UQ : ST_K);
            uint8_t *dst = smem + OFF_KS;
            const float Gend = gv[kC - 1];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = tid + kThreads * u;   // granule i: k half i >> 9, token (i >> 3) & 63, granule i & 7
                const int t = (i >> 3) & (kC - 1);
                const uint32_t off = (i >> 9) * kHalf + t * 128 + (i & 7) * 16;
                const float f = kRev ? p.q_scale * __expf(gv[t]) : __expf(Gend - gv[t]);
                const uint4 x = *reinterpret_cast<const uint4 *>(src + off);
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = pack_bf16(f * __uint_as_float(w[e] << 16), f * __uint_as_float(w[e] & 0xffff0000u));
                *reinterpret_cast<uint4 *>(dst + off) = make_uint4(o[0], o[1], o[2], o[3]);
            }
            fence_proxy_async_smem();
        }
        if (!wait_poll(bar_mma, mma_par)) *abort_flag = 1;
        mma_par ^= 1;
        tc_fence_after();
        // E^T (forward) or dE^T (reverse) for tokens [16 q, 16 q + 16) of this lane's value channel
        {
            uint32_t d[16], d2[16];
            tmem_ld16(tl + TM_D1 + 16 * q, d);
            if (kRev && drive) tmem_ld16(tl + TM_D1B + 16 * q, d2);
            tmem_ld_wait();
            const float Gend = kCh ? 0.f : gv[kC - 1];
            const unsigned short *ucol =
                reinterpret_cast<const unsigned short *>(smem + s * kStage + ST_UQ + (v >> 6) * kHalf);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int t = 16 * q + jj;
                float e;
                if (kRev) {
                    const float ee = kCh ? 1.f : __expf(Gend - gv[t]);
                    e = ee * __uint_as_float(d[jj]);
                    if (drive) e = fmaf(p.q_scale, __uint_as_float(d2[jj]), e);
                } else {
                    const float u = drive ? bf16_val(ucol[sw128_off(t, vb) >> 1]) : 0.f;
                    e = u - __uint_as_float(d[jj]);
                }
                ecol[sw128_off(t, vb) >> 1] = bf16_bits(e);
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        if (tid == 32) tma_store_wait_read_all();   // the state record has left the X^T tile
        __syncthreads();
        if (*abort_flag) break;
        tc_fence_after();
        if (tid == 32 && rec) {
            tma_store_2d(&mEr, sbase + OFF_E, 0, n * kC);
            tma_store_2d(&mEr, sbase + OFF_E + kHalf, 64, n * kC);
            tma_store_commit();
        }
        if (warp == 0) {
            if (elect_one()) {
                const uint64_t de = sw128_desc(sbase + OFF_E, kHalf, 1024);
                if (kRev) {
                    if (drive) {
                        const uint64_t ddo = sw128_desc(st + ST_DO, kHalf, 1024);
                        const uint64_t dq = sw128_desc(kCh ? st + ST_UQ : sbase + OFF_KS, kHalf, 1024);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16(tbase + TM_D2, desc_add(ddo, ks * 2048), desc_add(dq, ks * 2048), id_n128, ks);
                    }
                    const uint64_t dw = sw128_desc(st + ST_W, kHalf, 1024);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tbase + TM_D2B, desc_add(de, ks * 2048), desc_add(dw, ks * 2048), id_n128, ks);
                } else {
                    const uint64_t dk = sw128_desc(kCh ? st + ST_K : sbase + OFF_KS, kHalf, 1024);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tbase + TM_D2, desc_add(de, ks * 2048), desc_add(dk, ks * 2048), id_n128, ks);
                }
                mma_commit(bar_mma);
            }
            __syncwarp();
        }
        if (!wait_poll(bar_mma, mma_par)) *abort_flag = 1;
        mma_par ^= 1;
        tc_fence_after();
        // X'^T = Gamma X^T + D2 (- D2b): the decay, then the products in two passes of 16 key channels
        if (kCh) {   // e^{G_end} of this thread's 32 key channels
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 g4 = *reinterpret_cast<const float4 *>(gv + 32 * q + 4 * i);
                X[4 * i] *= g4.x;
                X[4 * i + 1] *= g4.y;
                X[4 * i + 2] *= g4.z;
                X[4 * i + 3] *= g4.w;
            }
        } else {
            const float Gam = __expf(gv[kC - 1]);
#pragma unroll
            for (int j = 0; j < 32; ++j) X[j] *= Gam;
        }
        // every load in flight before one wait (two rounds for the forward per-channel carry,
        // whose registers are fullest)
        constexpr int kRounds = (!kRev && kCh) ? 2 : 1, kCols = 32 / kRounds;
#pragma unroll
        for (int pc = 0; pc < kRounds; ++pc) {
            uint32_t a[kCols], bb[kRev ? kCols : 1];
            const bool has_a = !kRev || drive;
            if (has_a) {
                if constexpr (kCols == 32) tmem_ld32(tl + TM_D2 + 32 * q, a);
                else tmem_ld16(tl + TM_D2 + 32 * q + 16 * pc, a);
            }
            if constexpr (kRev) tmem_ld32(tl + TM_D2B + 32 * q, bb);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < kCols; ++jj) {
                const int j = kCols * pc + jj;
                float x = X[j];
                if (has_a) x += __uint_as_float(a[jj]);
                if constexpr (kRev) x -= __uint_as_float(bb[jj]);
                X[j] = x;
            }
        }
        put_x();
        tc_fence_before();
        if (tid == 32) tma_store_wait_read_all();   // the E / dE record has left its tile
        __syncthreads();
    }
    const bool aborted = *abort_flag != 0;
    // the end state of the segment; in reverse, the segment holding chunk 0 ends in dL/dS0
    auto put_end = [&](float *dst) {
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[(32 * q + j) * kD + v] = X[j];
    };
    if (!aborted) {
        if (p.Xseg) put_end(p.Xseg + (static_cast<size_t>(bh) * p.nseg + r) * kD * kD);
        if (kRev && p.X_end && c_lo == 0) put_end(p.X_end + static_cast<size_t>(bh) * kD * kD);
    }
    if (tid == 32) tma_store_wait_all();
    if (tid == 0 && aborted && p.err) atomicOr(p.err, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

}  // namespace

// ---------------------------------------------------------------------------- host side
namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

}  // namespace

bool map_record(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool map_tokens(CUtensorMap *m, const void *base, int B, int T, int H) {
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(H) * kD * 2,
                                   static_cast<cuuint64_t>(T) * H * kD * 2};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kC), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
template <bool kRev, bool kCh>
cudaError_t launch_t(const ScanParams &p, int grid, cudaStream_t stream) {
    const uint64_t N = static_cast<uint64_t>(p.B) * p.H * p.nc;
    CUtensorMap mK, mW, mUQ, mDO, mA, mX, mE;
    bool ok = kCh ? map_record(&mK, p.ws.Ke, kD, N * kC, kC) : map_tokens(&mK, p.k, p.B, p.T, p.H);
    ok = ok && map_record(&mW, p.ws.W, kD, N * kC, kC);
    if (kRev) {
        ok = ok && (kCh ? map_record(&mUQ, p.ws.Qg, kD, N * kC, kC) : map_tokens(&mUQ, p.q, p.B, p.T, p.H));
        ok = ok && map_tokens(&mDO, p.dO, p.B, p.T, p.H) && map_record(&mA, p.ws.A, kC, N * kC, kC);
    } else {
        ok = ok && map_record(&mUQ, p.ws.UdE, kD, N * kC, kC);
        mDO = mW;   // unused
        mA = mW;
    }
    ok = ok && map_record(&mX, kRev ? p.ws.dS : p.ws.S, kD, N * kD, kD) &&
         map_record(&mE, kRev ? p.ws.dE : p.ws.E, kD, N * kC, kC);
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(carry_tc_kernel<kRev, kCh>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    carry_tc_kernel<kRev, kCh><<<grid, kThreads, kSmemBytes, stream>>>(mK, mW, mUQ, mDO, mA, mX, mE, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_carry_tc(const ScanParams &p, bool rev, bool ch, int grid, cudaStream_t stream) {
    if (grid <= 0) return cudaSuccess;
    if (rev) return ch ? launch_t<true, true>(p, grid, stream) : launch_t<true, false>(p, grid, stream);
    return ch ? launch_t<false, true>(p, grid, stream) : launch_t<false, false>(p, grid, stream);
}

}  // namespace bwdc
}  // namespace kla
