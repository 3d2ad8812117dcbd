// common.cuh -- device helpers shared by the libmoeroute kernels (sm_103a):
// inline-PTX wrappers for mbarriers and the bulk (non-tensor) asynchronous
// copies between global and shared memory, bounded waits, and the launch
// parameter block that carries the per-rank token table.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_route.h"

namespace moe {

// Histogram tile: a run of consecutive (token, slot) items of one source rank.
constexpr int kHistThreads = 256;
constexpr int kHistWarps = kHistThreads / 32;
constexpr int kItemsPerThread = 8;
constexpr int kTileItems = kHistThreads * kItemsPerThread;   // 2048
constexpr int kItemsPerWarp = kTileItems / kHistWarps;       // 256

// Decoupled-lookback scan: elements per block.
constexpr int kScanThreads = 1024;
constexpr int kScanPerThread = 8;
constexpr int kScanChunk = kScanThreads * kScanPerThread;   // 8192

// Workspace header (bytes): [0] error word, [4] scan ticket.
constexpr size_t kWsHeader = 256;

// Bounded device waits end after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// Per-call rank table, passed by value as a kernel parameter (<= 2.1 KB), so
// no host-to-device copy is needed and a call can be captured in a graph.
struct RankTable {
    int R;
    int ntiles;                                  // total histogram tiles
    int32_t rank_off[MOE_MAX_RANKS + 1];         // token prefix: rank s owns [rank_off[s], rank_off[s+1])
    int32_t tile_off[MOE_MAX_RANKS + 1];         // tile prefix:  rank s owns tiles [tile_off[s], tile_off[s+1])
};

// Index s with a[s] <= v < a[s+1] for a non-decreasing a[0..n] (v in [a[0], a[n])).
__device__ __forceinline__ int upper_bound_minus_one(const int32_t *a, int n, int32_t v) {
    int lo = 0, hi = n + 1;   // first index with a[idx] > v lies in [1, n]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (a[mid] <= v) lo = mid; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// ------------------------------------------------------ bulk async copies

// global -> shared (this CTA), completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// shared (this CTA) -> global, tracked by the bulk async-group mechanism.
__device__ __forceinline__ void bulk_store(void *gdst, const void *smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All but the newest N committed store groups have finished READING shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// All committed store groups have completed (their writes are performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ global memory

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void set_device_error(int32_t *err, int bits) { atomicOr(err, bits); }

// Acquire load / release store and add of a 32-bit word in global memory, at
// GPU scope (the split halves' signals).
__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t *p) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int32_t *p, int32_t v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add_gpu(int32_t *p, int32_t v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Order this thread's completed async-proxy (bulk copy) writes to global
// memory before its later generic-proxy operations.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Programmatic dependent launch: allow the next kernel in the stream (if it
// was launched with programmatic stream serialization) to start now; wait
// until the kernel this one depends on has finished and its writes are
// visible (a no-op when there is no programmatic dependency).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace moe
