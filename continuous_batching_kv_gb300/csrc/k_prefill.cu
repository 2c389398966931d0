// K3b: GQA flash attention, prefill / mixed path on tcgen05 (in progress).
#include "dev_common.cuh"
#include "kernels.h"

namespace kvk {

cudaError_t launch_prefill(const CUtensorMap *, const CUtensorMap *, const PrefillArgs &, int32_t,
                           cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace kvk
