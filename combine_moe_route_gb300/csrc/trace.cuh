// trace.cuh -- optional phase timestamps for the dispatch and combine kernels.
//
// A library built with -DMOE_TRACE records, per call, the earliest and the
// latest %globaltimer value at which the kernels' blocks (or warps) reach each
// phase boundary: one slot pair per phase, min in the even slot and max in the
// odd one.  Each translation unit that stamps keeps its own array and exports
// its own reader (moe_trace_dispatch, moe_trace_combine), so no relocatable
// device code is needed.  Without MOE_TRACE every stamp compiles to nothing
// and no reader is exported; the default library is unchanged.
#pragma once

#include "common.cuh"

namespace moe {

// Phase slots (the reader returns kTraceSlots 64-bit values; even = min, odd = max).
enum TraceSlot : int {
    kTrPrepStart = 0,         // one-kernel path: prep kernel starts
    kTrSmallStart = 2,        // one-kernel path: block starts
    kTrSmallCounted = 4,      // counting done
    kTrSmallLayout = 6,       // scan of the totals and ranking done
    kTrSmallFirstStore = 8,   // a warp issues its first row stores
    kTrSmallWarpEnd = 10,     // a warp's stores have completed
    kTrHistStart = 12,        // three-kernel path: histogram block starts
    kTrHistEnd = 14,          // histogram block has written its ranks
    kTrScanStart = 16,        // scan block starts (before its wait)
    kTrScanWaitDone = 18,     // scan block's programmatic wait returned
    kTrScanTicket = 20,       // scan block has its virtual id
    kTrScanLocal = 22,        // loads and block-local scan done
    kTrScanLookback = 24,     // lookback done
    kTrScanEnd = 26,          // scan block has written its outputs
    kTrScatterStart = 28,     // scatter block starts
    kTrScatterWaitDone = 30,  // scatter warp's programmatic wait returned
    kTrScatterFirstStore = 32,
    kTrScatterWarpEnd = 34,
    kTrSmallStaged = 36,      // one-kernel path: routing table staged
    kTrCombineStart = 0,      // combine (its own array): block starts
    kTrCombineEnd = 2,        // block done
};
constexpr int kTraceSlots = 48;

}  // namespace moe

#ifdef MOE_TRACE
#define MOE_TRACE_DEFINE() static __device__ unsigned long long g_trace[moe::kTraceSlots];
#define MOE_STAMP(slot)                                                   \
    do {                                                                  \
        const unsigned long long t_ = moe::global_timer_ns();             \
        atomicMin(&g_trace[(slot)], t_);                                  \
        atomicMax(&g_trace[(slot) + 1], t_);                              \
    } while (0)
// reset != 0: arm the slots (min slots to ~0, max slots to 0); else copy them to out.
#define MOE_TRACE_READER(name)                                                                   \
    extern "C" MOE_API int name(int reset, unsigned long long *out) {                           \
        unsigned long long h[moe::kTraceSlots];                                                  \
        if (reset) {                                                                             \
            for (int i = 0; i < moe::kTraceSlots; ++i) h[i] = (i % 2 == 0) ? ~0ull : 0ull;      \
            return (int)cudaMemcpyToSymbol(g_trace, h, sizeof(h));                               \
        }                                                                                        \
        if (!out) return (int)cudaErrorInvalidValue;                                             \
        const cudaError_t e = cudaMemcpyFromSymbol(h, g_trace, sizeof(h));                       \
        for (int i = 0; i < moe::kTraceSlots; ++i) out[i] = h[i];                                \
        return (int)e;                                                                           \
    }
#else
#define MOE_TRACE_DEFINE()
#define MOE_STAMP(slot) ((void)0)
#define MOE_TRACE_READER(name)
#endif
