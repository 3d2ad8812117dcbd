// dispatch_noalloc.cu -- moe_dispatch_noalloc: moe_dispatch for callers that
// cannot allocate device memory.
//
// Who needs it: code that runs where allocation is not allowed or not
// possible -- for example a plugin inside another inference engine whose
// memory is owned and budgeted by that engine, or a serving loop that must not
// allocate on its hot path (an allocation can block, fragment a caching
// allocator or fail under memory pressure).  Such a caller can still pass its
// inputs and outputs, but not moe_dispatch's workspace.
//
// This variant takes its workspace from a fixed array in device memory that
// the library owns: a file-scope static __device__ buffer of
// MOE_NOALLOC_SCRATCH_BYTES bytes.  Every GPU that loads the library holds that
// buffer until the process exits.  Host code cannot use the array's name as a
// device address (in host code it names a host-side stand-in), so the first
// call on each device looks its device address up with cudaGetSymbolAddress,
// with that device current, and keeps it.  All calls on a device share the one
// buffer: calls that overlap on the GPU (different streams, or concurrent host
// threads) race on it, so they must be ordered.  The parts of the buffer that
// must start at zero (the error word, the lookback ticket and flags) are
// cleared on the stream at the start of every call, exactly as moe_dispatch
// does for a caller's workspace; the rest is fully overwritten by each call.
//
// The pages this library follows have no counterpart to this entry point.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "launch.h"
#include "moe_route.h"

namespace {

static __device__ __align__(256) unsigned char g_dispatch_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

// Device address of g_dispatch_scratch on the current device (looked up once per device).
moe_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" MOE_API moe_status moe_dispatch_noalloc(const void *x, const int32_t *topk_idx, int R, const int32_t *B,
                                                   int E, int K, int H, moe_dtype recv_dtype, void *recv_x,
                                                   float *recv_scale, int32_t *counts, int32_t *offsets,
                                                   int32_t *expert_offsets, int32_t *tok2row, int32_t *row2src,
                                                   moe_stream_t stream) {
    // moe_dispatch's own argument checks come first, so a call it would reject
    // reports the same status here; only a call that is otherwise valid can be
    // refused for its size.
    moe::RankTable rt;
    long long T = 0;
    bool fp8 = false;
    const moe_status v = moe::check_dispatch_args(x, topk_idx, R, B, E, K, H, recv_dtype, recv_x, recv_scale, true,
                                                  counts, offsets, expert_offsets, tok2row, row2src, rt, T, fp8);
    if (v != MOE_OK) return v;
    if (T == 0)   // nothing to scatter: moe_dispatch zero-fills the layout without a workspace
        return moe_dispatch(x, topk_idx, R, B, E, K, H, recv_dtype, recv_x, recv_scale, counts, offsets,
                            expert_offsets, tok2row, row2src, nullptr, 0, stream);
    if (moe_dispatch_workspace_bytes(R, E, K, T) > (size_t)MOE_NOALLOC_SCRATCH_BYTES)
        return MOE_ERR_WORKSPACE;   // beyond the static maximum

    void *scratch = nullptr;
    const moe_status st = scratch_address(&scratch);
    if (st != MOE_OK) return st;
    return moe_dispatch(x, topk_idx, R, B, E, K, H, recv_dtype, recv_x, recv_scale, counts, offsets, expert_offsets,
                        tok2row, row2src, scratch, (size_t)MOE_NOALLOC_SCRATCH_BYTES, stream);
}
