// host.cu -- host-side helpers shared by the kernel launchers: device
// properties the launch configurations depend on.
#include <atomic>

#include <cuda_runtime.h>

#include "internal.h"

namespace dlrm {

int sm_count()
{
    // The SM count is a property of the hardware, so a per-device cache stays valid for the life of the
    // process (also across a context reset).  Concurrent first calls store the same value.
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

int kernel_registers(const void* kernel)
{
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return 0;
    return fa.numRegs;
}

}  // namespace dlrm
