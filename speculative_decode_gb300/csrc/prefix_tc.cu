// prefix_tc.cu -- shared-prefix attention on the tcgen05 tensor cores.
#include "plan.h"

namespace sa {

cudaError_t launch_prefix_tc(const sa_dims &, const PlanDevice &, const uint16_t *,
                             const uint16_t *, const uint16_t *, float, float *, float *, int64_t,
                             int32_t *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace sa
