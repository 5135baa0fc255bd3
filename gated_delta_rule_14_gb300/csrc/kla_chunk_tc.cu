// kla_chunk_tc.cu -- tensor-core (tcgen05) chunkwise KLA prefill for sm_103a.
#include "kla_internal.cuh"

namespace kla {

bool chunk_tc_supports(const ChunkArgs &a) {
    (void)a;
    return false;
}

cudaError_t launch_chunk_tc(const ChunkArgs &a) {
    (void)a;
    return cudaErrorNotSupported;
}

}  // namespace kla
