// mx_qmm.cu -- prefill GEMM (placeholder until the tcgen05 kernel lands).
#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {
cudaError_t launch_qmm(const DeviceState &, cudaStream_t, int, const uint8_t *, const uint8_t *,
                       const uint16_t *, uint16_t *, int, int, int)
{
    return cudaErrorNotSupported;
}
}  // namespace mx
