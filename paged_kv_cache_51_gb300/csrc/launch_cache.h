// Host launch setup done once per (kernel, device) instead of on every call:
// the dynamic shared-memory attribute and the number of CTAs that fit on an SM.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <utility>

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

// Launch `kern` with programmatic dependent launch allowed: it may become
// resident while the kernel before it on the stream is still running (once that
// kernel triggers its dependents), so the launch latency hides behind that
// kernel's tail.  Every kernel launched this way waits for its prerequisites
// (griddepcontrol.wait) before it reads or writes anything the work ahead of it
// could touch, so stream order holds.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace pkv
