// Order-preserving keys and warp helpers shared by the top-k kernels (topk.cu,
// topk_filter.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace vl {

// fp32 -> u32 with the same order (larger value, larger key); -0.0 ranks as +0.0.
__device__ __forceinline__ uint32_t f2key(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key2f(uint32_t k) {
    return (k & 0x80000000u) ? __uint_as_float(k & 0x7fffffffu) : __uint_as_float(~k);
}

// composite order on (key, id): larger key first, then lower id
__device__ __forceinline__ unsigned long long comp(uint32_t key, uint32_t id) {
    return ((unsigned long long)key << 32) | (unsigned long long)(0xffffffffu - id);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// This warp's a-th largest of its values of the first tile (kVecT float4s a lane, all
// present): a rounds of taking the warp's largest out.
template <int kVecT>
__device__ __forceinline__ float warp_kth(const float4 (&v)[kVecT], uint32_t a, int lane) {
    float e[4 * kVecT];
#pragma unroll
    for (int u = 0; u < kVecT; ++u) { e[4 * u] = v[u].x; e[4 * u + 1] = v[u].y; e[4 * u + 2] = v[u].z; e[4 * u + 3] = v[u].w; }
    float top = -INFINITY;
    for (uint32_t i = 0; i < a; ++i) {
        float m = e[0];
#pragma unroll
        for (int q = 1; q < 4 * kVecT; ++q) m = fmaxf(m, e[q]);
        top = m;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) top = fmaxf(top, __shfl_xor_sync(0xffffffffu, top, off));
        // the lowest lane holding it takes one copy out
        const uint32_t holders = __ballot_sync(0xffffffffu, m == top);
        if (lane == __ffs(holders) - 1) {
            bool done = false;
#pragma unroll
            for (int q = 0; q < 4 * kVecT; ++q)
                if (!done && e[q] == top) { e[q] = -INFINITY; done = true; }
        }
    }
    return top;
}

}  // namespace vl
