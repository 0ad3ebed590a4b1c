// Tensor-core W4A16 matmul (tcgen05 / TMEM).  Not built yet.
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {

cudaError_t launch_gemm_tc(const void*, int64_t, int64_t, int64_t, const void*, const void*, void*,
                           const DeviceInfo&, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace w4
