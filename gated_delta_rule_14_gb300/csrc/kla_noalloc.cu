// kla_noalloc.cu -- chunkwise prefill for callers that cannot allocate device memory.
//
// Some callers of this library cannot allocate: a serving runtime whose memory manager
// reserves all device memory up front and hands kernels only the buffers it owns, or code
// running on a stream whose allocations would have to be serialised against work already in
// flight. kla_chunk_fwd asks those callers for a workspace when it splits long sequences into
// segments; kla_chunk_fwd_noalloc instead uses a fixed scratch array that is part of this
// library's device image.
//
// The array below is allocated on every GPU that loads the library and stays there until the
// process exits. Every call on a device shares it and it keeps the last call's contents; the
// segmented prefill writes every scratch element it later reads within the same call (segment
// value runs, transition runs, then the combine pass), so nothing has to be cleared between
// calls. Calls whose kernels may overlap on the GPU (different streams, no ordering between
// them) race on the array: callers must order them. kla_chunk_fwd_host borrows the array for
// the last part of its batch (ordered among host calls by an event of its own).
#include <mutex>

#include "kla_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

}  // namespace

namespace kla {
cudaError_t noalloc_scratch(void **out);
}  // namespace kla

// Device address of the scratch array on the current device. In host code the array's name
// is only a host-side stand-in, so the address must come from the runtime; it is looked up
// on the first call per device (with that device current) and cached.
cudaError_t kla::noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

extern "C" kla_status kla_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *alpha,
                                            const float *eta, float eps, const float *S0, void *o, float *S_T,
                                            int B, int T, int H, int d_k, int d_v, int chunk, kla_dtype dtype,
                                            kla_gate gate, void *stream) {
    // the errors of kla_chunk_fwd come first; only a valid call is refused for its size
    const kla_status st = kla::check_chunk_fwd(q, k, v, alpha, eta, eps, S0, o, S_T, B, T, H, d_k, d_v, chunk, dtype,
                                               gate, KLA_BETA_KACZMARZ, 1.0f);
    if (st != KLA_OK) return st;
    const size_t need = kla_chunk_fwd_workspace_size(B, T, H, d_k, d_v, chunk, dtype, gate);
    if (need > static_cast<size_t>(KLA_NOALLOC_SCRATCH_BYTES)) return KLA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (need > 0 && kla::noalloc_scratch(&scratch) != cudaSuccess) return KLA_ERR_CUDA;
    return kla_chunk_fwd(q, k, v, alpha, eta, eps, S0, o, S_T, B, T, H, d_k, d_v, chunk, dtype, gate, scratch,
                         need > 0 ? static_cast<size_t>(KLA_NOALLOC_SCRATCH_BYTES) : 0, stream);
}
