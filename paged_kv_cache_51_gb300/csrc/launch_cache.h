// Host launch setup done once per (kernel, device) instead of on every call:
// the dynamic shared-memory attribute and the number of CTAs that fit on an SM.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

namespace pkv {

constexpr int kMaxDevices = 64;

// CTAs of kernel `Kern` (threads, dynamic smem bytes) resident per SM on the
// current device, or 0 on a CUDA error.  The first call per device sets the
// kernel's dynamic shared-memory limit.  One cache per kernel: the kernel is a
// template argument, not a runtime pointer (kernels sharing a signature would
// otherwise share the entry).
template <auto Kern>
int kernel_occupancy(int threads, int smem) {
    static std::atomic<int> cached[kMaxDevices];
    const auto kern = Kern;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, size_t(smem)) !=
            cudaSuccess ||
        v < 1)
        return 0;
    cached[dev].store(v, std::memory_order_relaxed);
    return v;
}

}  // namespace pkv
