// Prefill attention kernel (tcgen05) -- placeholder until the kernel lands.
#include "common.cuh"
#include "internal.h"

namespace sage {

cudaError_t launch_prefill(const PrefillParams &, cudaStream_t, LaunchLog &) {
    return cudaErrorNotSupported;
}

}  // namespace sage
