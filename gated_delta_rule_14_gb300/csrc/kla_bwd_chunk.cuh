// kla_bwd_chunk.cuh -- pieces shared by the chunkwise backward kernels (kla_bwd_chunk.cu: gradients
// of the scalar gate and the launch sequence; kla_bwd_prep_tc.cu: the scalar gate's prep on the
// tensor cores; kla_bwd_chunk_ch.cu: prep and gradients of the per-key-channel gate;
// kla_bwd_carry_tc.cu: both chunk-state carries, on the tensor cores):
// the per-chunk workspace records, the carries' parameters, padded shared-memory tiles,
// warp-level bf16 MMAs on them, cp.async staging and the 64 x 64 unit-lower inverse.
#pragma once

#include <cuda.h>

#include "kla_internal.cuh"
#include "sm103_ptx.cuh"
#include "warp_mma.cuh"

namespace kla {
namespace bwdc {

using namespace wmma16;

constexpr int kC = 64;                  // chunk
constexpr int kD = 128;                 // d_k = d_v
constexpr int kP = kD + 8;              // pitch (bf16 elements) of a tile with 128 columns
constexpr int kPs = kC + 8;             // pitch of a tile with 64 columns
constexpr int kTileTok = kC * kP * 2;   // 64 x 128 bf16 tile: 17408 bytes
constexpr int kTileSt = kD * kP * 2;    // 128 x 128: 34816
constexpr int kTileSq = kC * kPs * 2;   // 64 x 64: 9216
constexpr float kMinLogGate = -80.0f;

typedef __nv_bfloat16 bf16;

// ---- bulk copies of the tensor-core kernels (addresses 16-byte aligned; box columns a multiple of 8)
// A 2-D box of a tensor map into shared memory, counted on `bar`; a box out of shared memory in
// the thread's bulk group; a contiguous run of bytes (a multiple of 16) into shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(dst),
        "l"(tmap), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_store_2d(const void *tmap, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// A bf16 value as its 16 bits (round to nearest even) and back.
__device__ __forceinline__ unsigned short bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
__device__ __forceinline__ float bf16_val(unsigned short bits) { return __uint_as_float(static_cast<uint32_t>(bits) << 16); }

// ---- per-chunk workspace records (structure of arrays over n = chain * nc + chunk)
constexpr size_t kCgFloats = 3 * kC;    // G (scalar gate only), beta, den = ||k||^2 + eps
struct Ws {
    float *cg;        // [N][3][64]
    bf16 *W;          // [N][64][128]
    bf16 *UdE;        // [N][64][128]: U (prep -> forward carry), then dE with the scalar gate
    bf16 *dE;         // [N][64][128]: dE (reverse carry -> gradients): UdE, or its own record with
                      // the per-channel gate (so that the two carries may run at the same time)
    bf16 *A;          // [N][64][64]  lower(ratio . QK^T), unscaled by s
    bf16 *Tm;         // [N][64][64]  T = (I + R)^{-1}
    bf16 *S;          // [N][128][128] state entering the chunk
    bf16 *E;          // [N][64][128]
    bf16 *dS;         // [N][128][128] dL/d(state leaving the chunk)
    // per-key-channel gate only (NULL otherwise): the decayed key and query tiles the two carries
    // read in place of k and q, and the chunk's end decay per key channel (dE above follows them)
    bf16 *Ke;         // [N][64][128] K e^{G_end - G}
    bf16 *Qg;         // [N][64][128] s Q e^{G}
    float *gend;      // [N][128]     e^{G_end}
    float *seg;       // long chains split into segments: Z | M | start states, each [chains][nseg][128][128]
};
inline size_t ws_bytes_per_chunk(bool ch) {
    return kCgFloats * 4 + 2 * (3 * kC * kD + 2 * kC * kC + 2 * kD * kD) + (ch ? 2 * (3 * kC * kD) + 4 * kD : 0);
}
inline Ws carve(void *base, size_t N, bool ch) {
    char *p = static_cast<char *>(base);
    Ws w;
    w.cg = reinterpret_cast<float *>(p);             p += N * kCgFloats * 4;
    w.W = reinterpret_cast<bf16 *>(p);               p += N * kC * kD * 2;
    w.UdE = reinterpret_cast<bf16 *>(p);             p += N * kC * kD * 2;
    w.E = reinterpret_cast<bf16 *>(p);               p += N * kC * kD * 2;
    w.A = reinterpret_cast<bf16 *>(p);               p += N * kC * kC * 2;
    w.Tm = reinterpret_cast<bf16 *>(p);              p += N * kC * kC * 2;
    w.S = reinterpret_cast<bf16 *>(p);               p += N * kD * kD * 2;
    w.dS = reinterpret_cast<bf16 *>(p);              p += N * kD * kD * 2;
    w.Ke = w.Qg = nullptr;
    w.gend = nullptr;
    w.dE = w.UdE;
    if (ch) {
        w.dE = reinterpret_cast<bf16 *>(p);          p += N * kC * kD * 2;
        w.Ke = reinterpret_cast<bf16 *>(p);          p += N * kC * kD * 2;
        w.Qg = reinterpret_cast<bf16 *>(p);          p += N * kC * kD * 2;
        w.gend = reinterpret_cast<float *>(p);       p += N * kD * 4;
    }
    w.seg = reinterpret_cast<float *>(p);
    return w;
}

// ---------------------------------------------------------------- warp-level MMA helpers

template <int NT>   // NT n8 tiles (even)
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
}
// acc[16 x (8 NT)] += A[r0.., k0..k0+16*KS) * B[.., n0..]: one warp, A and B layouts as template flags.
template <int NT, int KS, bool kAT, bool kBT>
__device__ __forceinline__ void gemm(float (&acc)[NT][4], uint32_t ta, int pa, int r0, int ka, uint32_t tb, int pb,
                                     int n0, int kb, int lane) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[4];
        if (kAT) frag_a_kr(ta, pa, r0, ka + 16 * ks, lane, a);
        else frag_a_rk(ta, pa, r0, ka + 16 * ks, lane, a);
#pragma unroll
        for (int j = 0; j < NT / 2; ++j) {
            uint32_t b[4];
            if (kBT) frag_b_kr(tb, pb, n0 + 16 * j, kb + 16 * ks, lane, b);
            else frag_b_rk(tb, pb, n0 + 16 * j, kb + 16 * ks, lane, b);
            mma(acc[2 * j], a, b[0], b[1]);
            mma(acc[2 * j + 1], a, b[2], b[3]);
        }
    }
}
__device__ __forceinline__ void st_pair(bf16 *tile, int pitch, int r, int c, float lo, float hi) {
    *reinterpret_cast<uint32_t *>(tile + r * pitch + c) = pack2(lo, hi);
}
__device__ __forceinline__ float2 ld_pair(const bf16 *tile, int pitch, int r, int c) {
    return unpack2(*reinterpret_cast<const uint32_t *>(tile + r * pitch + c));
}
__device__ __forceinline__ void cp16(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sptr(dst)), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {   // 16-byte aligned, multiple of 16
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 64 token rows x 128 columns of a [B,T,H,128] bf16 tensor into a padded tile (rows >= L zero).
__device__ __forceinline__ void load_tok(bf16 *tile, const bf16 *src, size_t row_stride, int L, int tid,
                                         int nthreads) {
    for (int i = tid; i < kC * 16; i += nthreads) {
        const int r = i >> 4, c = (i & 15) * 8;
        const bool ok = r < L;
        cp16(tile + r * kP + c, src + (ok ? r : 0) * row_stride + c, ok);
    }
}
// `rows` dense rows of `cols` bf16 (cols = 64 or 128) from the workspace into a padded tile.
template <int kCols>
__device__ __forceinline__ void load_dense(bf16 *tile, const bf16 *src, int rows, int tid, int nthreads) {
    constexpr int kPitch = kCols + 8, kChunks = kCols / 8;
    for (int i = tid; i < rows * kChunks; i += nthreads) {
        const int r = i / kChunks, c = (i % kChunks) * 8;
        cp16(tile + r * kPitch + c, src + r * kCols + c, true);
    }
}
template <int kCols>
__device__ __forceinline__ void store_dense(bf16 *dst, const bf16 *tile, int rows, int tid, int nthreads) {
    constexpr int kPitch = kCols + 8, kChunks = kCols / 8;
    for (int i = tid; i < rows * kChunks; i += nthreads) {
        const int r = i / kChunks, c = (i % kChunks) * 8;
        *reinterpret_cast<uint4 *>(dst + r * kCols + c) = *reinterpret_cast<const uint4 *>(tile + r * kPitch + c);
    }
}

// acc[MT m16 tiles][NT n8 tiles] += A * B for MT row tiles at r0, r0 + 16, ... (B fragments shared).
template <int MT, int NT, int KS, bool kAT, bool kBT>
__device__ __forceinline__ void gemm_m(float (&acc)[MT][NT][4], uint32_t ta, int pa, int r0, int ka, uint32_t tb,
                                       int pb, int n0, int kb, int lane) {
#pragma unroll
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

__device__ __forceinline__ void bar_named(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// T = (I + R)^{-1} in place over the fp32 64 x 64 strictly-lower R (pitch kPR), by 8 warps of one
// CTA (every thread calls it; it ends with a block barrier). sX: fp32 [32][kPX] scratch.
constexpr int kPR = 68;   // pitch of the fp32 64 x 64 tile (4 mod 32: no conflicts)
constexpr int kPX = 36;
__device__ __forceinline__ void unit_lower_inverse64(float (*sR)[kPR], float *sX, int warp, int lane) {
    // (1) the four 16 x 16 diagonal blocks by substitution:
    // warp 0 lanes 0-15 / 16-31 take blocks 0 / 1, warp 1 blocks 2 / 3; lane = column.
    if (warp < 2) {
        const int blk = 2 * warp + (lane >> 4), j = lane & 15, o = 16 * blk;
        float t[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) t[m] = m == j ? 1.f : 0.f;
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int m = 0; m < i; ++m) {
                if (m & 1) a1 = fmaf(sR[o + i][o + m], t[m], a1);
                else a0 = fmaf(sR[o + i][o + m], t[m], a0);
            }
            if (i > j) t[i] = -(a0 + a1);
        }
        __syncwarp();
#pragma unroll
        for (int m = 0; m < 16; ++m) sR[o + m][o + j] = t[m];
    }
    __syncthreads();
    // (2) merges: [T11 0; R21 T22]^{-1} has lower block -T22 R21 T11, on tf32 warp MMAs.
    // Size 16: two merges side by side (blocks at 0 and 32), warp w < 4 takes merge w >> 1 and
    // output columns 8 (w & 1); size 32: warp w takes output rows 16 (w >> 2), columns 8 (w & 3).
    const float *R0 = &sR[0][0];
    float *R0w = &sR[0][0];
    const int g = lane >> 2, q4 = lane & 3;
    auto put_tile = [&](float *M, int pitch, int r, int cc, const float (&acc)[4], float sign) {
        M[(r + g) * pitch + cc + 2 * q4] = sign * acc[0];
        M[(r + g) * pitch + cc + 2 * q4 + 1] = sign * acc[1];
        M[(r + g + 8) * pitch + cc + 2 * q4] = sign * acc[2];
        M[(r + g + 8) * pitch + cc + 2 * q4 + 1] = sign * acc[3];
    };
    if (warp < 4) {   // X = R21 T11
        const int o = 32 * (warp >> 1), nc8 = 8 * (warp & 1);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        tile_tf32<2>(acc, R0, kPR, o + 16, o, R0, kPR, o, o + nc8, lane);
        put_tile(sX, kPX, 16 * (warp >> 1), nc8, acc, 1.f);
    }
    __syncthreads();
    if (warp < 4) {   // T21 = -T22 X
        const int o = 32 * (warp >> 1), nc8 = 8 * (warp & 1);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        tile_tf32<2>(acc, R0, kPR, o + 16, o + 16, sX, kPX, 16 * (warp >> 1), nc8, lane);
        put_tile(R0w, kPR, o + 16, o + nc8, acc, -1.f);
    }
    __syncthreads();
    {   // X = R21 T11 at size 32
        const int mr = 16 * (warp >> 2), nc8 = 8 * (warp & 3);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        tile_tf32<4>(acc, R0, kPR, 32 + mr, 0, R0, kPR, 0, nc8, lane);
        put_tile(sX, kPX, mr, nc8, acc, 1.f);
    }
    __syncthreads();
    {   // T21 = -T22 X
        const int mr = 16 * (warp >> 2), nc8 = 8 * (warp & 3);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        tile_tf32<4>(acc, R0, kPR, 32 + mr, 32, sX, kPX, 0, nc8, lane);
        put_tile(R0w, kPR, 32 + mr, nc8, acc, -1.f);
    }
    __syncthreads();
}

// ---- the per-key-channel chunkwise backward (kla_bwd_chunk_ch.cu); the carries are the
// scalar path's chunk_scan_kernel reading the Ke, Qg and gend records
struct ChBwd {
    const bf16 *q, *k, *v, *dO;
    const float *alpha, *eta;
    float eps, q_scale;
    int beta_raw;
    int B, T, H, nc;
    Ws ws;
    const unsigned *skip;   // [B*H] chains left to the token-sequential path (their CTAs return at once)
    float *dq, *dk, *dv, *dalpha, *deta;
    unsigned *err;          // device error word (a bounded wait that gives up sets kErrTimeout)
};
// ---- the chunk-state carries (one CTA per chain segment, chunks in order)
struct ScanParams {
    const bf16 *q, *k, *dO;
    const float *X0;      // S0 (forward) or dL/dS_T (reverse): [B,H,128,128] fp32, NULL = zeros
    float *X_end;         // reverse: dL/dS0 (NULL = not wanted)
    float q_scale;
    int B, T, H, nc;
    Ws ws;
    // Segments (a long chain split for a sequence-parallel scan; one segment = the whole chain
    // otherwise). Segment r in processing order covers chunks [s L, min((s + 1) L, nc)) with
    // s = r (forward) or s = nseg - 1 - r (reverse). A launch runs segments seg_begin ..
    // seg_begin + seg_count - 1 of every chain, one CTA each.
    int seg_len, seg_begin, seg_count, nseg;
    int x0_mode;          // kX0Chain, kX0Identity or kX0Given
    int drive;            // 0: drop U (forward) or the dO terms (reverse): the linear part only
    int records;          // per-chunk records (S_c, E_c or dS_{c+1}, dE_c): 0 none, 1 all, 2 segment r = 0 only
    float *Xseg;          // NULL, or [chains][nseg][128][128]: X at the end of each segment
    const float *Xst;     // kX0Given: [chains][nseg][128][128] start states
    const unsigned *skip; // NULL, or [B*H]: chains left to the token-sequential path (their CTAs return)
    unsigned *err;        // device error word (a bounded wait that gives up sets kErrTimeout)
};
enum : int {
    kX0Chain = 0,      // X0 for the chain's first segment (r = 0), zeros for the others
    kX0Identity = 1,   // the identity (the segment's transition)
    kX0Given = 2,      // Xst[chain][r]
};
}  // namespace bwdc
// Device address of the library's error word on the current device.
cudaError_t device_error_word(unsigned **out);
namespace bwdc {
// Tensor maps (128-byte swizzle) of the tensor-core kernels: a [rows][cols] bf16 record in boxes
// of box_rows x 64 columns, and a [B, T, H, 128] bf16 input in boxes of 64 tokens x 64 channels
// of one (b, h), tokens past T reading 0. False when the driver's encoder is unavailable or
// rejects the map.
bool map_record(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows);
bool map_tokens(CUtensorMap *m, const void *base, int B, int T, int H);
// The scalar gate's per-chunk records (cg, A, T, W, U) on the tensor cores, one CTA per chunk.
cudaError_t launch_prep_tc(const bf16 *q, const bf16 *k, const bf16 *v, const float *alpha, const float *eta,
                           float eps, int beta_raw, int B, int T, int H, int nc, const Ws &ws, unsigned *err,
                           cudaStream_t stream);
// Runs `grid` CTAs of the forward (rev = false) or reverse carry on the tensor cores.
cudaError_t launch_carry_tc(const ScanParams &p, bool rev, bool ch, int grid, cudaStream_t stream);

cudaError_t launch_bwd_prep_ch(const ChBwd &p, cudaStream_t stream);
cudaError_t launch_bwd_grad_ch(const ChBwd &p, cudaStream_t stream);

}  // namespace bwdc
}  // namespace kla
