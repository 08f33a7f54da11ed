// Warp-level reductions shared by the CUDA-core decode split kernels.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

constexpr unsigned kFullWarp = 0xffffffffu;

// Reduce-scatter across the warp: every lane holds NV partial sums; afterwards
// lane l holds the full sum of value l (NV = 32) or of value l >> 1 (NV = 16).
template <int NV>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV], int lane) {
#pragma unroll
    for (int step = 0; (NV >> step) > 1; ++step) {
        const int n = NV >> step;
        const int off = 16 >> step;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(kFullWarp, send, off);
        }
    }
    float r = v[0];
    if (NV == 16) r += __shfl_xor_sync(kFullWarp, r, 1);
    return r;
}

// max / sum over the lanes that hold the same query head
template <int G, int TC>
__device__ __forceinline__ float group_max(float x) {
    if (G == 1) {
#pragma unroll
        for (int off = 2; off < 32; off <<= 1) x = fmaxf(x, __shfl_xor_sync(kFullWarp, x, off));
    } else {
#pragma unroll
        for (int off = 1; off < TC; off <<= 1) x = fmaxf(x, __shfl_xor_sync(kFullWarp, x, off));
    }
    return x;
}
template <int G, int TC>
__device__ __forceinline__ float group_sum(float x) {
    if (G == 1) {
#pragma unroll
        for (int off = 2; off < 32; off <<= 1) x += __shfl_xor_sync(kFullWarp, x, off);
    } else {
#pragma unroll
        for (int off = 1; off < TC; off <<= 1) x += __shfl_xor_sync(kFullWarp, x, off);
    }
    return x;
}

__device__ __forceinline__ void consumer_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

}  // namespace pkv
