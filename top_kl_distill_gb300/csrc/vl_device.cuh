// Device-side building blocks shared by the libvloss kernels (sm_103a).
//
// Inline PTX for what the CUDA C++ front end does not expose directly:
// mbarriers with transaction counts, 1-D bulk copies global -> shared
// (cp.async.bulk, the TMA engine's untiled form), cluster ranks and
// distributed shared memory, named barriers with a popcount, and the
// bounded waits (a wait that has not completed after ~2 s is a bug: the kernel
// records it and unwinds instead of hanging the GPU).
#pragma once

#include <cstdint>
#include <cfloat>
#include <cuda_runtime.h>

namespace vl {


constexpr float kLog2e = 1.4426950408889634f;   // log2(e)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


// 2^x on the special-function unit (ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init_cluster() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Acquire at cluster scope: pairs with a remote release-arrive from a peer CTA.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// SM cycles after which a wait gives up (about two seconds at the GB300's clocks).
constexpr long long kWaitTimeoutCycles = 4000000000ll;

// Bounded wait for the phase of `bar` with the given parity to complete.
// Returns false if the wait gave up: either another thread of the CTA raised
// *abort, or this wait ran past kWaitTimeoutCycles (then it raises *abort and
// sets *flag).  Every wait in the library goes through here.  The fast path is
// one try_wait (which itself suspends the thread for a while); the clock and the
// abort flag are only read after many failed polls.
template <bool kCluster>
__device__ __forceinline__ bool wait_parity(uint64_t* bar, uint32_t parity, volatile int* abort,
                                            unsigned int* flag, long long limit = kWaitTimeoutCycles) {
    const uint32_t b = smem_u32(bar);
    long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (kCluster ? mbar_try_wait_cluster(b, parity) : mbar_try_wait(b, parity)) return true;
        if ((it & 255u) == 255u) {
            if (*abort) return false;
            const long long now = clock64();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > limit) {
                *abort = 1;
                atomicOr(flag, 1u);
                return false;
            }
        }
    }
}

// Same wait without the abort check, for draining copies already in flight.
__device__ __forceinline__ bool wait_parity_drain(uint64_t* bar, uint32_t parity,
                                                  long long limit = kWaitTimeoutCycles) {
    const uint32_t b = smem_u32(bar);
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

// ------------------------------------------------------------------ bulk copy

// 1-D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is signalled on `bar`
// as a transaction count.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Same copy with an L2 eviction-priority policy (from createpolicy) on the source lines.
__device__ __forceinline__ void bulk_g2s_hint(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

// L2 policies: lines touched under evict_last stay ahead of everything else; under
// evict_first they are the first to go.
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------ cluster

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t ncluster_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float a, float b) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" :: "r"(addr), "f"(a), "f"(b) : "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float a) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(addr), "f"(a) : "memory");
}

// Asynchronous store into a peer CTA's shared memory that completes `bytes` of the
// transaction count of the peer's mbarrier when the data has landed (no fence).
__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float a, float b, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
                 :: "r"(addr), "f"(a), "f"(b), "r"(bar) : "memory");
}

__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float4 v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 :: "r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar) : "memory");
}

__device__ __forceinline__ void st_async_f32(uint32_t addr, float a, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
                 :: "r"(addr), "f"(a), "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_remote_release(uint32_t bar_cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(bar_cluster_addr) : "memory");
}

// ------------------------------------------------------------------ CTA-level

// Named barrier `id` over `n` threads (a multiple of 32).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}

// Named barrier that also returns how many participating threads passed pred = true.
__device__ __forceinline__ uint32_t named_sync_popc(uint32_t id, uint32_t n, bool pred) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.u32 p, %3, 0;\n\t"
                 "bar.red.popc.u32 %0, %1, %2, p;\n\t}"
                 : "=r"(r) : "r"(id), "r"(n), "r"((uint32_t)pred) : "memory");
    return r;
}

// Programmatic dependent launch: let the next kernel on the stream start its
// prologue; it still waits for this grid's memory before reading it.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------ stores / loads

__device__ __forceinline__ void st_global_v4(float* p, float4 v) {
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}

// Global float4 load that skips L1 and marks the L2 line with `policy`.
__device__ __forceinline__ float4 ld_global_v4_hint(const float* p, uint64_t policy) {
    float4 v;
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p), "l"(policy) : "memory");
    return v;
}

__device__ __forceinline__ void st_global_v4_hint(float* p, float4 v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;"
                 :: "l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "l"(policy) : "memory");
}

__device__ __forceinline__ float4 ld_shared_v4(const float* p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(smem_u32(p)));
    return v;
}

// ------------------------------------------------------------------ online softmax statistics

// Running (max, sum of exp(x - max)) of a stream of values.
struct MaxSum {
    float m;
    float s;
};

__device__ __forceinline__ MaxSum ms_empty() { return MaxSum{-FLT_MAX, 0.0f}; }

__device__ __forceinline__ void ms_add(MaxSum& a, float x) {
    if (x > a.m) {
        a.s = a.s * ex2((a.m - x) * kLog2e);
        a.m = x;
    }
    a.s += ex2((x - a.m) * kLog2e);
}

__device__ __forceinline__ float warp_sum(float a) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    return a;
}

// The warp's (max, sum): the max over the lanes first, then each lane's sum rescaled to
// it once and summed (butterflies: every lane holds the same bits).
__device__ __forceinline__ MaxSum ms_warp_reduce(MaxSum a) {
    float M = a.m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    return MaxSum{M, warp_sum(a.s * ex2((a.m - M) * kLog2e))};
}

}  // namespace vl
