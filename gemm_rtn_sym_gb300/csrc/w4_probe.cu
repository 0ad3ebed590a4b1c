// Diagnostic kernel for the bounded waits: one CTA waits on an mbarrier that is
// completed only when `arrive` is set.  A wait that runs out records a timeout in
// the device status word and the kernel returns normally.
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

__global__ void wait_probe_kernel(uint64_t limit_ns, int arrive, unsigned* status) {
    __shared__ alignas(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) mbar_init(b, 1);
    __syncthreads();
    if (arrive && threadIdx.x == 0) mbar_arrive(b);
    if (!mbar_wait(b, 0, limit_ns)) {
        if (threadIdx.x == 0) record_status(status, kStatusTimeout);
    }
}

}  // namespace

cudaError_t launch_wait_probe(int64_t limit_ns, int arrive, const DeviceInfo& dev,
                              cudaStream_t stream) {
    wait_probe_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(limit_ns), arrive, dev.status);
    return cudaGetLastError();
}

}  // namespace w4
