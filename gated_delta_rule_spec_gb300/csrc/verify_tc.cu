// verify_tc.cu -- TMA + tcgen05 verify kernel (sm_103a).  Placeholder until
// the kernel lands: reports no supported shape, so every layer takes the
// CUDA-core kernel.
#include "common.cuh"

namespace gdnspec {

bool verify_tc_supported(const LayerArgs &, bool, bool) { return false; }

cudaError_t launch_verify_tc(const LayerArgs &, const CursorArgs &, const int32_t *, int,
                             const void *, const void *, const void *, const void *,
                             const void *, const float *, const float *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace gdnspec
