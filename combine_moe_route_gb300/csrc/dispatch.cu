// dispatch.cu -- count, exclusive scan and scatter of tokens into the
// expert-contiguous receive buffer, with an optional fused FP8 quantise.
//
// Sources:
//  * lehuy.net, "Decoding high-performance EP kernels", "Optimising for
//    throughput: ask first, send later" > "Dispatch": the layout is not known
//    in advance; count what goes where, exchange the counts, and a prefix sum
//    over them fixes a conflict-free layout; then each token is copied to the
//    slot the prefix sum assigned.
//  * Perplexity, "Enabling trillion-parameter models on AWS EFA", "Dispatch
//    and combine": per-expert token counts by shared-memory atomics inside a
//    block, a cumulative sum for the offsets, rows packed contiguously and
//    reorganised into the grouped-GEMM input.
//  * Perplexity, "Lower latency and higher throughput with multi-node DeepSeek
//    deployment", "Quantization": activation scales over 128-element vectors,
//    computed on the fly.
//
// With all R ranks in one HBM the count exchange is a read of the histogram
// in global memory and the send+receive pair is a single hop: each source row
// is staged once in shared memory by a bulk copy and written by bulk copies
// straight into its K destination rows.
//
// Batches of more than MOE_SMALL_DISPATCH_ITEMS (token, slot) items run three
// kernels, stream-ordered (the second and third launched with programmatic
// stream serialization, so each starts while its predecessor finishes and
// waits only where it reads the predecessor's output); smaller ones run the
// one-kernel path of section 4 below, with the same layout:
//  1. tile histogram: the items (g, j) of one rank are cut into tiles of
//     kTileItems consecutive items.  Each warp counts its run of 256 items
//     into a warp-private shared histogram; lanes holding the same expert are
//     grouped by a ballot per bit of the expert id and their leader adds the
//     group size with one shared-memory atomic, whose return value plus the
//     lane's position in the group is the item's rank among equal experts so
//     far.  The warps' histograms are then combined in warp order, giving
//     every item a stable rank inside (expert, tile) and every tile its
//     per-expert total.
//  2. exclusive scan over the histogram laid out expert-major, tile-minor
//     (e * ntiles + tile), one pass with decoupled lookback.  Because tiles
//     are rank-major and ranks hold consecutive tokens, this order is exactly
//     (expert, source rank, token): the scanned value of (e, tile) is the
//     first receive row of expert e's items in that tile.
//  3. scatter, one warp per token: row(g, j) = scan[e * ntiles + tile(g, j)]
//     + rank-in-tile; copy (or quantise once and copy) x[g] into its K rows.
//
// The low-latency layout (lehuy.net, same article, "Optimising for latency:
// send without asking") skips the scan: its rows are a static formula over a
// fixed region per (expert, source rank), so it runs kernels 1 and 3 only.
// Its unordered form lets each copy take its slot in the region by an atomic
// increment, and runs a zeroing kernel and kernel 3 only.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <atomic>
#include <mutex>

#include "launch.h"
#include "trace.cuh"

// Scatter launch shape (tunable at build time; the defaults are the measured best):
// warps per block and bulk-copy ring stages per warp.
#ifndef MOE_SCATTER_WARPS
#define MOE_SCATTER_WARPS 1
#endif
#ifndef MOE_SCATTER_STAGES
#define MOE_SCATTER_STAGES 2
#endif
// SMs the persistent scatter may occupy (0: all of them); fewer leaves room
// for work running concurrently on another stream.
#ifndef MOE_SCATTER_MAX_SMS
#define MOE_SCATTER_MAX_SMS 0
#endif

namespace moe {

MOE_TRACE_DEFINE()

// --------------------------------------------------------------------------
// 1. tile histogram + stable in-tile ranks
// --------------------------------------------------------------------------
// local_rank (aliases the tok2row output): in-tile rank of each item, or -1
// (an expert id out of range; the scatter, which reads every id again,
// reports it).  Block 0 also clears the call's workspace header (error word,
// scan ticket, scatter token counter), the split halves' signals and the
// lookback status words: nothing reads or writes them before this grid has
// completed, so no memset has to run ahead of this kernel.
__global__ void __launch_bounds__(kHistThreads) tile_hist_kernel(const int32_t *__restrict__ topk_idx, int E, int K,
                                                                 const __grid_constant__ RankTable rt,
                                                                 int32_t *__restrict__ tile_hist,
                                                                 int32_t *__restrict__ local_rank,
                                                                 int32_t *__restrict__ header,
                                                                 int32_t *__restrict__ signal, int nsignal,
                                                                 unsigned long long *__restrict__ status,
                                                                 int nstatus) {
    extern __shared__ int32_t hist[];   // [kHistWarps][E]
    pdl_launch_dependents();            // the scan may launch; it waits for this grid's writes
    if (threadIdx.x == 0) MOE_STAMP(kTrHistStart);
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < (int)(kWsHeader / 4); i += blockDim.x) header[i] = 0;
        for (int i = threadIdx.x; i < nsignal; i += blockDim.x) signal[i] = 0;
        for (int i = threadIdx.x; i < nstatus; i += blockDim.x) status[i] = 0ull;
    }
    const int tile = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int s = upper_bound_minus_one(rt.tile_off, rt.R, tile);
    const long long rank_lo = (long long)rt.rank_off[s] * K;
    const long long rank_hi = (long long)rt.rank_off[s + 1] * K;
    const long long lo = rank_lo + (long long)(tile - rt.tile_off[s]) * kTileItems;
    const long long hi = min(lo + (long long)kTileItems, rank_hi);

    for (int i = threadIdx.x; i < kHistWarps * E; i += blockDim.x) hist[i] = 0;
    __syncthreads();

    int32_t *my_hist = hist + warp * E;
    const unsigned lanemask_lt = (1u << lane) - 1u;
    const int ebits = (E > 1) ? 32 - __clz(E - 1) : 0;   // bits of the largest expert id
    int e_reg[kItemsPerThread];
    int r_reg[kItemsPerThread];
    // all of this thread's item loads first, so they are in flight together
#pragma unroll
    for (int step = 0; step < kItemsPerThread; ++step) {
        const long long i = lo + warp * kItemsPerWarp + step * 32 + lane;
        e_reg[step] = (i < hi) ? __ldg(topk_idx + i) : -1;
    }
#pragma unroll
    for (int step = 0; step < kItemsPerThread; ++step) {
        int e = e_reg[step];
        if (e >= E) e = -1;   // out of range: no rank (the scatter reports it)
        // lanes holding the same expert: one ballot per bit of the expert id
        // (a multi-split; its cost does not grow with the number of distinct
        // experts in the warp, unlike a match instruction)
        unsigned peers = __ballot_sync(0xffffffffu, e >= 0);
        for (int b = 0; b < ebits; ++b) {
            const bool bit = (e >> b) & 1;
            const unsigned m = __ballot_sync(0xffffffffu, bit);
            peers &= bit ? m : ~m;
        }
        // the group's lowest lane adds the group size; every lane then reads
        // its own group leader's old count in one full-warp shuffle (a
        // shuffle masked by the group would run once per distinct expert)
        const int leader = (e >= 0) ? __ffs(peers) - 1 : lane;
        int base = 0;
        if (e >= 0 && lane == leader) base = atomicAdd(&my_hist[e], __popc(peers));
        base = __shfl_sync(0xffffffffu, base, leader);
        e_reg[step] = e;
        r_reg[step] = (e >= 0) ? base + __popc(peers & lanemask_lt) : -1;
        __syncwarp();
    }
    __syncthreads();

    // combine the warps' histograms in warp order: hist[w][e] becomes the
    // exclusive prefix over warps, the tile total goes to global memory
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kHistWarps; ++w) {
            const int c = hist[w * E + e];
            hist[w * E + e] = run;
            run += c;
        }
        tile_hist[(long long)e * rt.ntiles + tile] = run;
    }
    __syncthreads();

#pragma unroll
    for (int step = 0; step < kItemsPerThread; ++step) {
        const long long i = lo + warp * kItemsPerWarp + step * 32 + lane;
        if (i < hi) {
            const int e = e_reg[step];
            local_rank[i] = (e >= 0) ? my_hist[e] + r_reg[step] : -1;
        }
    }
    if (threadIdx.x == 0) MOE_STAMP(kTrHistEnd);
}

// --------------------------------------------------------------------------
// 2. exclusive scan with decoupled lookback
// --------------------------------------------------------------------------
// status[b]: 0 = not yet published; (1 << 62 | aggregate) = block aggregate;
// (2 << 62 | inclusive prefix) = everything up to and including block b.
constexpr unsigned long long kFlagAgg = 1ull << 62;
constexpr unsigned long long kFlagPrefix = 2ull << 62;
constexpr unsigned long long kFlagMask = 3ull << 62;

__device__ __forceinline__ int warp_inclusive_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    return v;
}

// out[0..n] = exclusive prefix of in[0..n-1]; out[n] = total.
__global__ void __launch_bounds__(kScanThreads) lookback_scan_kernel(const int32_t *__restrict__ in,
                                                                     int32_t *__restrict__ out, int n,
                                                                     unsigned long long *status, int32_t *ticket,
                                                                     int32_t *err) {
    __shared__ int s_vid;
    __shared__ int s_warp[kScanThreads / 32];
    __shared__ int s_excl;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    if (tid == 0) MOE_STAMP(kTrScanStart);
    // virtual block id in start order: every lower id has started, so the
    // lookback below only waits on blocks that are already running
    pdl_launch_dependents();   // the scatter may launch and stage its first rows
    pdl_wait();                                    // the tile histogram is complete and visible
    if (tid == 0) MOE_STAMP(kTrScanWaitDone);
    // ticket and flags were cleared by the histogram grid
    if (tid == 0) s_vid = atomicAdd(ticket, 1);
    __syncthreads();
    const int vid = s_vid;
    if (tid == 0) MOE_STAMP(kTrScanTicket);
    // warp w owns kScanPerThread consecutive 32-element slices of the block's
    // chunk; slice k is read and written by the 32 lanes together (coalesced)
    const long long wbase = (long long)vid * kScanChunk + (long long)warp * (32 * kScanPerThread);

    int v[kScanPerThread];
    int incl[kScanPerThread];   // inclusive scan inside slice k
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) {
        const long long i = wbase + k * 32 + lane;
        v[k] = (i < n) ? in[i] : 0;
    }
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) incl[k] = warp_inclusive_scan(v[k]);
    int slice_excl[kScanPerThread];   // sum of the warp's earlier slices
    int wsum = 0;
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) {
        slice_excl[k] = wsum;
        wsum += __shfl_sync(0xffffffffu, incl[k], 31);
    }
    if (lane == 0) s_warp[warp] = wsum;
    __syncthreads();
    if (tid == 0) MOE_STAMP(kTrScanLocal);
    if (warp == 0) {
        const int wv = (lane < kScanThreads / 32) ? s_warp[lane] : 0;
        const int wincl = warp_inclusive_scan(wv);
        if (lane < kScanThreads / 32) s_warp[lane] = wincl - wv;   // exclusive over warps
        if (lane == kScanThreads / 32 - 1) {
            const int aggregate = wincl;
            int excl = 0;
#ifdef MOE_TEST_WITHHOLD_SCAN_BLOCK
            // Test builds only: this block never publishes, so its successor's
            // bounded lookback runs out (exercises the timeout path).
            const bool publish = vid != MOE_TEST_WITHHOLD_SCAN_BLOCK;
#else
            const bool publish = true;
#endif
            // a status word carries its own value, so publishing needs no fence
            if (vid == 0) {
                if (publish) atomicExch(&status[0], kFlagPrefix | (unsigned long long)(unsigned)aggregate);
            } else {
                if (publish) atomicExch(&status[vid], kFlagAgg | (unsigned long long)(unsigned)aggregate);
                int p = vid - 1;
                const uint64_t t0 = global_timer_ns();
                bool timed_out = false;
                while (p >= 0) {
                    const unsigned long long st = ld_volatile_u64(&status[p]);
                    const unsigned long long flag = st & kFlagMask;
                    if (flag == 0ull) {
                        if (global_timer_ns() - t0 > kWaitLimitNs) {
                            timed_out = true;
                            break;
                        }
                        __nanosleep(32);
                        continue;
                    }
                    excl += (int)(unsigned)(st & 0xffffffffull);
                    if (flag == kFlagPrefix) break;
                    --p;
                }
                if (timed_out) set_device_error(err, MOE_DEVERR_SCAN_TIMEOUT);
                if (publish) atomicExch(&status[vid], kFlagPrefix | (unsigned long long)(unsigned)(excl + aggregate));
            }
            s_excl = excl;
            if ((long long)(vid + 1) * kScanChunk >= n) out[n] = excl + aggregate;   // last block: total
        }
    }
    __syncthreads();
    if (tid == 0) MOE_STAMP(kTrScanLookback);
    const int wexcl = s_excl + s_warp[warp];
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) {
        const long long i = wbase + k * 32 + lane;
        if (i < n) out[i] = wexcl + slice_excl[k] + incl[k] - v[k];
    }
    if (tid == 0) MOE_STAMP(kTrScanEnd);
}

// --------------------------------------------------------------------------
// 3. scatter (+ fused FP8 quantise)
// --------------------------------------------------------------------------
struct ScatterArgs {
    const __nv_bfloat16 *x;
    const int32_t *topk_idx;
    const int32_t *scan;       // [E * ntiles + 1]
    void *recv_x;
    float *recv_scale;
    int32_t *counts;
    int32_t *offsets;
    int32_t *expert_offsets;
    int32_t *tok2row;          // in: in-tile ranks; out: rows
    int32_t *row2src;
    int32_t *err;
    const int32_t *tile_hist;  // [E * ntiles] (low-latency layout)
    int32_t *next_token;       // token counter, zero at launch (workspace header)
    int32_t *arrive;           // send half: copies landed per destination rank (zero at launch), else null
    int T, E, K, H;
    int C;                     // low-latency layout: rows per (expert, source rank) region
};

// 16 lanes quantise one 128-channel block: lane owns 8 consecutive channels.
__device__ __forceinline__ void quantize_block16(const uint4 xin, uint2 &qout, float &scale_out) {
    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&xin);
    float f[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 t = __bfloat1622float2(h2[k]);
        f[2 * k] = t.x;
        f[2 * k + 1] = t.y;
    }
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[k]));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    // raised to 2^-119, the smallest power of two with 448/amax finite in fp32:
    // a zero or tiny block keeps finite scales, and its nonzero bf16 values
    // (down to 2^-133) still map to nonzero codes
    amax = fmaxf(amax, 0x1p-119f);
    scale_out = __fdiv_rn(amax, 448.0f);
    const float inv = __fdiv_rn(448.0f, amax);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float a = __fmul_rn(f[2 * k], inv);
        const float b = __fmul_rn(f[2 * k + 1], inv);
        // low byte = first element (little endian, same as consecutive bytes in memory)
        w[k] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    }
    qout.x = w[0] | (w[1] << 16);
    qout.y = w[2] | (w[3] << 16);
}

// Shared memory of one ring stage: a bf16 source row (H*2 bytes; for FP8 the
// e4m3 row is written in place over its first H bytes), then for FP8 the
// row's H/128 scales.
__host__ __device__ inline size_t scatter_stage_bytes(int H, bool fp8) {
    size_t b = (size_t)H * 2 + (fp8 ? (size_t)(H / 128) * 4 : 0);
    return (b + 127) & ~(size_t)127;
}

// Quantise one staged bf16 row to e4m3 in place (its H/128 fp32 scales after
// the row's 2H bytes): two 128-channel blocks per step (16 lanes per block),
// ascending, so every e4m3 byte lands on bf16 bytes that have already been read.
__device__ __forceinline__ void quantize_stage(unsigned char *buf, int H, int lane) {
    const int nblk = H / 128;
    float *sc = reinterpret_cast<float *>(buf + (size_t)H * 2);
    const uint4 *src = reinterpret_cast<const uint4 *>(buf);
    uint2 *q = reinterpret_cast<uint2 *>(buf);
    const int hl = lane & 15;
    for (int b0 = 0; b0 < nblk; b0 += 2) {
        const int b = b0 + (lane >> 4);
        const bool valid = b < nblk;
        const uint4 xin = valid ? src[b * 16 + hl] : make_uint4(0u, 0u, 0u, 0u);
        uint2 qo;
        float s;
        quantize_block16(xin, qo, s);
        // the second half-warp's codes land on bf16 bytes the first half-warp
        // read in this step: every lane's read comes before any lane's write
        __syncwarp();
        if (valid) {
            q[b * 16 + hl] = qo;
            if (hl == 0) sc[b] = s;
        }
    }
    fence_proxy_async_smem();
}

// Persistent, one warp per token.  Warp w starts with tokens w, w + W, ...,
// w + (S-1)W (W warps in the grid); after those, lane 0 claims each further
// token from a counter in the (zeroed) workspace header, so warps on faster
// SMs take more tokens and the grid ends together.  Each warp runs its own
// ring of S bulk-copy stages; its token sequence number it selects stage
// it % S.  Before waiting for the scan, a warp loads its first S tokens and
// (FP8) quantises the first one, none of which depends on the histogram.
// Per token:
//   1. lanes j < K compute the destination row of copy j (scan base of the
//      token's tile + its in-tile rank) and write tok2row / row2src;
//   2. wait for the staged source row (mbarrier, bounded);
//   3. FP8: quantise in place;
//   4. lane 0 issues K bulk stores of the row (and, when H % 512 == 0, K bulk
//      stores of the scale row; otherwise the lanes store the scales);
//   5. once the previous token's stores have read their stage, lane 0 refills
//      that stage with a newly claimed token (claimed one token in advance, so
//      the atomic's latency is hidden behind the current token).
//
// kLowLatency: the destination is a fixed rectangle with C rows per (expert,
// source rank) region; row = (e*R + s)*C + (tokens of rank s routed to e in
// the rank's earlier tiles) + in-tile rank.  No scan is needed.
// kLowLatencyUnordered: the same rectangle, but a copy takes its slot in the
// region by one atomic increment of the region's count (zeroed before the
// launch), so neither histogram nor scan runs; the order of a region's rows is
// whatever order the increments happened in.
//
// Send half of the split dispatch (a.arrive != null, ragged layout): the
// counts / offsets / expert_offsets are left to the receive half, and every
// warp tallies its copies per destination rank in shared memory; once its
// last bulk stores have completed it adds the tallies to the per-rank arrival
// counters with release semantics (the receive half waits for them).
enum ScatterMode : int { kRagged = 0, kLowLatency = 1, kLowLatencyUnordered = 2 };

template <bool kFp8, int kMode>
__global__ void __launch_bounds__(MOE_SCATTER_WARPS * 32) scatter_kernel(const ScatterArgs a,
                                                                         const __grid_constant__ RankTable rt) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[MOE_SCATTER_WARPS][MOE_SCATTER_STAGES];
    __shared__ int32_t s_rows[MOE_SCATTER_WARPS][MOE_MAX_TOPK];
    __shared__ int32_t s_tok[MOE_SCATTER_WARPS][MOE_SCATTER_STAGES];   // token held by each stage
    constexpr int S = MOE_SCATTER_STAGES;
    static_assert(S >= 2, "the refill schedule needs at least two stages per warp");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = a.H, K = a.K, E = a.E, T = a.T;
    const int nblk = H / 128;
    const size_t stage_bytes = scatter_stage_bytes(H, kFp8);
    const uint32_t in_bytes = (uint32_t)H * 2u;
    const uint32_t out_bytes = kFp8 ? (uint32_t)H : in_bytes;
    const size_t recv_pitch = kFp8 ? (size_t)H : (size_t)H * 2;
    const bool scale_bulk = kFp8 && (nblk * 4) % 16 == 0;

    unsigned char *wbase = smem + (size_t)warp * S * stage_bytes;
    auto stage = [&](int it) { return wbase + (size_t)(it % S) * stage_bytes; };
    // send half: this warp's copies per destination rank, after every warp's stages
    const bool send = kMode == kRagged && a.arrive != nullptr;
    const int L = E / rt.R;
    int32_t *s_arr = send ? reinterpret_cast<int32_t *>(smem + (size_t)MOE_SCATTER_WARPS * S * stage_bytes) +
                                (size_t)warp * rt.R
                          : nullptr;
    if (send) {
        for (int r = lane; r < rt.R; r += 32) s_arr[r] = 0;
        __syncwarp();
    }
    // the first S tokens of warp w are w, w + W, ..., w + (S-1)W (W warps in
    // the grid), which spreads a small batch over every warp; the tokens from
    // S*W on are handed out by the counter
    const long long W = (long long)gridDim.x * MOE_SCATTER_WARPS;
    const long long gw = (long long)blockIdx.x * MOE_SCATTER_WARPS + warp;
    const long long first_dynamic = (long long)S * W;

    if (threadIdx.x == 0) MOE_STAMP(kTrScatterStart);
    // prologue: the source rows do not depend on the histogram or the scan,
    // so the first S tokens are loaded before waiting for it
    int claimed = 0;      // tokens this warp has claimed and started loading
    long long next_g = T;   // lane 0: the token claimed in advance for the next refill
    if (lane == 0) {
        for (int st = 0; st < S; ++st) mbar_init(&bars[warp][st], 1);
        fence_proxy_async_smem();
        for (; claimed < S && gw + (long long)claimed * W < T; ++claimed) {
            const int g = (int)(gw + (long long)claimed * W);
            s_tok[warp][claimed] = g;
            mbar_arrive_expect_tx(&bars[warp][claimed], in_bytes);
#ifdef MOE_TEST_WITHHOLD_FIRST_LOAD
            // Test builds only: the warp holding token 0 arms its stage but never
            // issues the copy, so its bounded barrier wait runs out.
            if (g == 0) continue;
#endif
            bulk_load(stage(claimed), a.x + (long long)g * H, in_bytes, &bars[warp][claimed]);
        }
    }
    claimed = __shfl_sync(0xffffffffu, claimed, 0);
    __syncwarp();

    int failed_at = -1;
    bool first_quantised = false;
    if (kFp8 && claimed > 0) {
        if (__all_sync(0xffffffffu, mbar_wait_bounded(&bars[warp][0], 0u))) {
            quantize_stage(stage(0), H, lane);
            first_quantised = true;
        } else {
            failed_at = 0;
        }
    }
    // Nothing before this wait touches the workspace header: the unordered
    // low-latency mode zeroes it in the kernel this one waits for.
    pdl_wait();
    if (lane == 0) MOE_STAMP(kTrScatterWaitDone);
    if (lane == 0) {
        if (failed_at == 0) set_device_error(a.err, MOE_DEVERR_COPY_TIMEOUT);
        if (claimed == S) next_g = first_dynamic + atomicAdd(a.next_token, 1);
    }

    if (kMode == kLowLatency) {
        // counts[e*R + s]: the rank's tile totals for expert e
        const int n = E * rt.R;
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
            const int e = i / rt.R;
            const int s = i - e * rt.R;
            int c = 0;
            for (int tau = rt.tile_off[s]; tau < rt.tile_off[s + 1]; ++tau) c += a.tile_hist[(long long)e * rt.ntiles + tau];
            a.counts[i] = c;
        }
    } else if (kMode == kRagged && !send) {
        // counts / offsets / expert_offsets from the scanned histogram (the
        // split dispatch writes them in its receive half)
        const int n = E * rt.R;
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= n; i += gridDim.x * blockDim.x) {
            if (i < n) {
                const int e = i / rt.R;
                const int s = i - e * rt.R;
                const int o = a.scan[(long long)e * rt.ntiles + rt.tile_off[s]];
                const int o1 = a.scan[(long long)e * rt.ntiles + rt.tile_off[s + 1]];
                a.offsets[i] = o;
                a.counts[i] = o1 - o;
                if (s == 0) a.expert_offsets[e] = o;
            } else {
                const int total = a.scan[(long long)E * rt.ntiles];
                a.offsets[n] = total;
                a.expert_offsets[E] = total;
            }
        }
    }
    if (claimed == 0) return;

    for (int it = 0; failed_at < 0 && it < claimed; ++it) {
        const uint32_t parity = (uint32_t)((it / S) & 1);
        unsigned char *buf = stage(it);
        int my_dest = -1;   // send half: destination rank of this lane's copy (lane j = copy j)
        // 1. destination rows (lane j = copy j)
        {
            const long long g = s_tok[warp][it % S];
            const int sidx = upper_bound_minus_one(rt.rank_off, rt.R, (int32_t)g);
            const long long item0 = (long long)rt.rank_off[sidx] * K;
            int e = -1, row = -1;
            if (lane < K) {
                const long long i = g * K + lane;
                e = __ldg(a.topk_idx + i);
                if (kMode == kLowLatencyUnordered) {
                    if (e >= 0 && e < E) {
                        const int region = e * rt.R + sidx;
                        const int slot = atomicAdd(a.counts + region, 1);
                        // every B[s] <= C, so a region never overflows; the check keeps a
                        // write inside the rectangle whatever the input
                        row = (slot < a.C) ? region * a.C + slot : -1;
                    } else {
                        set_device_error(a.err, MOE_DEVERR_EXPERT_RANGE);
                    }
                    if (row >= 0) {
                        a.row2src[row] = (int32_t)i;
                    } else {
                        e = -1;
                    }
                } else {
                    const int lr = a.tok2row[i];
                    if (e < 0 || e >= E) set_device_error(a.err, MOE_DEVERR_EXPERT_RANGE);
                    if (e >= 0 && e < E && lr >= 0) {
                        const int tile = rt.tile_off[sidx] + (int)((i - item0) / kTileItems);
                        if (kMode == kLowLatency) {
                            int base = (e * rt.R + sidx) * a.C;
                            for (int tau = rt.tile_off[sidx]; tau < tile; ++tau)
                                base += a.tile_hist[(long long)e * rt.ntiles + tau];
                            row = base + lr;
                        } else {
                            row = a.scan[(long long)e * rt.ntiles + tile] + lr;
                        }
                        a.row2src[row] = (int32_t)i;
                    } else {
                        e = -1;
                    }
                }
                a.tok2row[i] = row;
                s_rows[warp][lane] = row;
                if (send && row >= 0) my_dest = e / L;
            }
            int dup = 0;
            for (int j = 0; j < K; ++j) {
                const int ej = __shfl_sync(0xffffffffu, e, j);
                if (lane < j && e >= 0 && e == ej) dup = 1;
            }
            if (__any_sync(0xffffffffu, dup) && lane == 0) set_device_error(a.err, MOE_DEVERR_DUPLICATE);
        }

        // 2. the staged source row
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[warp][it % S], parity));
        if (!ok) {
            if (lane == 0) set_device_error(a.err, MOE_DEVERR_COPY_TIMEOUT);
            failed_at = it;
            break;
        }
        if (my_dest >= 0) atomicAdd(&s_arr[my_dest], 1);   // stored below

        // 3. quantise in place
        float *sc = reinterpret_cast<float *>(buf + (size_t)H * 2);
        if (kFp8 && !(it == 0 && first_quantised)) quantize_stage(buf, H, lane);
        __syncwarp();

        // 4. K bulk stores from the stage
        if (lane == 0) MOE_STAMP(kTrScatterFirstStore);
        if (lane == 0) {
            for (int j = 0; j < K; ++j) {
                const int row = s_rows[warp][j];
                if (row < 0) continue;
                bulk_store(static_cast<unsigned char *>(a.recv_x) + (size_t)row * recv_pitch, buf, out_bytes);
                if (scale_bulk) bulk_store(a.recv_scale + (size_t)row * nblk, sc, (uint32_t)nblk * 4u);
            }
            bulk_commit();
        }
        if (kFp8 && !scale_bulk) {
            for (int t = lane; t < K * nblk; t += 32) {
                const int j = t / nblk;
                const int b = t - j * nblk;
                const int row = s_rows[warp][j];
                if (row >= 0) a.recv_scale[(size_t)row * nblk + b] = sc[b];
            }
        }

        // 5. refill the previous token's stage (sequence number it - 1 + S ==
        //    claimed, the ring being full) once its stores have read it
        if (lane == 0 && it >= 1 && next_g < T) {
            bulk_wait_read<1>();
            const int nxt = claimed;
            s_tok[warp][nxt % S] = (int32_t)next_g;
            mbar_arrive_expect_tx(&bars[warp][nxt % S], in_bytes);
            bulk_load(stage(nxt), a.x + (long long)next_g * H, in_bytes, &bars[warp][nxt % S]);
            ++claimed;
            next_g = first_dynamic + atomicAdd(a.next_token, 1);
        }
        __syncwarp();   // s_rows, s_tok and the stage are reused in later iterations
        claimed = __shfl_sync(0xffffffffu, claimed, 0);
    }

    if (lane == 0) {
        if (failed_at >= 0) {
            // let every load this warp issued land before the block's shared
            // memory goes away (each wait is bounded; one that never arrives
            // costs its limit and the rest are still waited for)
            for (int t = failed_at; t < claimed; ++t)
                (void)mbar_wait_bounded(&bars[warp][t % S], (uint32_t)((t / S) & 1));
        }
        bulk_wait_all();
        MOE_STAMP(kTrScatterWarpEnd);
        if (send) {
            // the bulk stores are complete; order them before the releases below
            fence_proxy_async_global();
            __threadfence();
        }
    }
    if (send) {
        __syncwarp();
        for (int r = lane; r < rt.R; r += 32) {
            const int c = s_arr[r];
#ifdef MOE_TEST_WITHHOLD_ARRIVAL_RANK
            // Test builds only: copies bound for this rank are never announced,
            // so the receive half's bounded wait runs out.
            if (r == MOE_TEST_WITHHOLD_ARRIVAL_RANK) continue;
#endif
            if (c > 0) red_release_add_gpu(a.arrive + r, c);
        }
    }
}

// --------------------------------------------------------------------------
// 4. small batches: count, scan and scatter in one kernel
// --------------------------------------------------------------------------
// Inside expert e's segment the rows follow the global (rank-major) token
// order, so copy j of token g lands in
//   row(g, j) = start(e) + #{tokens g' < g routed to e},  e = topk_idx[g, j],
// where start(e) is the number of copies routed to the experts below e.  When
// the batch has few items, every block can afford to count all of them and
// the histogram and scan kernels (and the two kernel boundaries they cost)
// drop out: block b takes the contiguous tokens [g0, g1), and
//   A. each warp stages its first two source rows by bulk copy (they do not
//      depend on the routing, so the loads overlap the counting);
//   B. the block counts every item per expert (tot), the items before g0
//      (pre), and, for the source rank s = b (then b + grid, ...), the items
//      of the ranks below s (bef) and of rank s (ins);
//   C. tot is scanned into start(e); the block writes rank s's layout --
//      counts[e*R+s] = ins(e), offsets[e*R+s] = start(e) + bef(e);
//   D. chunk by chunk (ctok tokens, at most kSmallChunkItems items), the
//      block ranks each item of the chunk among the earlier items of the same
//      expert (pre counts those before the chunk and grows after each one),
//      and its warps scatter the chunk's tokens (one warp per token, two
//      bulk-copy stages, in-place FP8) as the scatter kernel does.
// A block normally holds a handful of tokens and one chunk; the chunks keep
// shared memory and the ranking bounded when a capped SM budget gives each
// block many.
// The kernel runs behind a one-block kernel that clears the workspace header
// and signals (programmatic stream serialization); it waits for that kernel
// before it first touches either.  The send half of the split dispatch
// (layout != null) writes offsets into the workspace, where its receive half
// reads them, instead of the counts / offsets / expert_offsets outputs.
constexpr int kSmallMaxWarps = 8;
constexpr int kSmallStages = 2;
constexpr int kSmallChunkItems = 512;
#ifndef MOE_SMALL_DISPATCH_ITEMS
#define MOE_SMALL_DISPATCH_ITEMS 16384   // T*K up to which a dispatch takes the one-kernel path
#endif

struct SmallArgs {
    const __nv_bfloat16 *x;
    const int32_t *topk_idx;
    void *recv_x;
    float *recv_scale;
    int32_t *counts;           // null in the send half
    int32_t *offsets;
    int32_t *expert_offsets;
    int32_t *layout;           // send half: offsets [E*R + 1] for the receive half, else null
    int32_t *tok2row;
    int32_t *row2src;
    int32_t *err;
    int32_t *arrive;           // send half: copies landed per destination rank, else null
    int T, E, K, H;
    int tpb;                   // tokens per block
    int ctok;                  // tokens per chunk: a multiple of the warps per block
    int stages;                // bulk-copy stages per warp: 2, or 1 when no warp has a second token
    int stage_ids;             // 1: the whole topk_idx is staged in shared memory by one bulk copy
};

// Tokens per chunk for W warps and top-K: the most whole rounds of W tokens
// whose items fit kSmallChunkItems (one round at least; W * K <= 256).
__host__ __device__ inline int small_chunk_tokens(int W, int K) {
    const int rounds = kSmallChunkItems / K / W;
    return W * (rounds > 0 ? rounds : 1);
}

// Bytes of dynamic shared memory of the one-kernel dispatch for W warps.
__host__ __device__ inline size_t small_smem_bytes(int W, int stages, int H, bool fp8, int E, int R, int K,
                                                   bool send) {
    size_t b = (size_t)W * stages * scatter_stage_bytes(H, fp8);
    b += (size_t)4 * E * 4;                   // tot, pre, bef, ins
    b += (size_t)2 * small_chunk_tokens(W, K) * K * 4;   // a chunk's expert ids and rows
    if (send) b += (size_t)W * R * 4;         // per-warp arrival tallies
    return b;
}

// Offset and bytes of the staged routing table (after everything above, 16-byte aligned).
__host__ __device__ inline size_t small_ids_offset(int W, int stages, int H, bool fp8, int E, int R, int K,
                                                    bool send) {
    return (small_smem_bytes(W, stages, H, fp8, E, R, K, send) + 15) & ~(size_t)15;
}

__global__ void dispatch_prep_kernel(int32_t *__restrict__ header, int32_t *__restrict__ signal, int nsignal) {
    pdl_launch_dependents();
    if (threadIdx.x == 0) MOE_STAMP(kTrPrepStart);
    for (int i = threadIdx.x; i < (int)(kWsHeader / 4); i += blockDim.x) header[i] = 0;
    for (int i = threadIdx.x; i < nsignal; i += blockDim.x) signal[i] = 0;
}

template <bool kFp8>
__global__ void __launch_bounds__(kSmallMaxWarps * 32) dispatch_small_kernel(const SmallArgs a,
                                                                             const __grid_constant__ RankTable rt) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[kSmallMaxWarps][kSmallStages];
    __shared__ __align__(8) uint64_t bar_ids;
    __shared__ int s_total;
    const int S = a.stages;   // 1 or 2 (kSmallStages)
    const int W = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = a.T, E = a.E, K = a.K, H = a.H, R = rt.R, L = E / R;
    const int nblk = H / 128;
    const size_t stage_bytes = scatter_stage_bytes(H, kFp8);
    const uint32_t in_bytes = (uint32_t)H * 2u;
    const uint32_t out_bytes = kFp8 ? (uint32_t)H : in_bytes;
    const size_t recv_pitch = kFp8 ? (size_t)H : (size_t)H * 2;
    const bool scale_bulk = kFp8 && (nblk * 4) % 16 == 0;
    const bool send = a.arrive != nullptr;

    const long long g0 = (long long)blockIdx.x * a.tpb;
    if (threadIdx.x == 0) MOE_STAMP(kTrSmallStart);
    const long long g1 = min(g0 + (long long)a.tpb, (long long)T);
    const int ntok = (int)(g1 - g0);
    const int my_n = ntok > warp ? (ntok - warp + W - 1) / W : 0;   // tokens g0 + warp + it*W

    int32_t *tot = reinterpret_cast<int32_t *>(smem + (size_t)W * S * stage_bytes);
    int32_t *pre = tot + E;
    int32_t *bef = pre + E;
    int32_t *ins = bef + E;
    int32_t *s_idx = ins + E;                 // [ctok*K] expert ids of the chunk's items
    int32_t *s_row = s_idx + a.ctok * K;      // [ctok*K] their rows
    int32_t *s_arr = send ? s_row + a.ctok * K + warp * R : nullptr;
    auto stage = [&](int it) { return smem + ((size_t)warp * S + (it % S)) * stage_bytes; };

    // A. stage the routing table (when it fits) and the first rows
    const long long n_all = (long long)T * K;
    int32_t *s_items = reinterpret_cast<int32_t *>(smem + small_ids_offset(W, S, H, kFp8, E, R, K, send));
    const uint32_t ids_bulk = (uint32_t)((n_all * 4) & ~15ll);   // the bulk copy's whole 16-byte units
    if (threadIdx.x == 0 && a.stage_ids) {
        mbar_init(&bar_ids, 1);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bar_ids, ids_bulk);
#ifndef MOE_TEST_WITHHOLD_IDS_COPY
        bulk_load(s_items, a.topk_idx, ids_bulk, &bar_ids);
#endif
        // (test builds with MOE_TEST_WITHHOLD_IDS_COPY arm the barrier but never
        // issue the copy, so its bounded wait runs out and the ids come from
        // global memory)
    }
    if (lane == 0) {
        for (int st = 0; st < S; ++st) mbar_init(&bars[warp][st], 1);
        fence_proxy_async_smem();
        for (int it = 0; it < S && it < my_n; ++it) {
            const long long g = g0 + warp + (long long)it * W;
            mbar_arrive_expect_tx(&bars[warp][it], in_bytes);
#ifdef MOE_TEST_WITHHOLD_FIRST_LOAD
            // Test builds only: token 0's stage is armed but never filled, so its
            // bounded barrier wait runs out.
            if (g == 0) continue;
#endif
            bulk_load(stage(it), a.x + g * H, in_bytes, &bars[warp][it]);
        }
    }

    // B. counts; the first chunk's expert ids are fetched first, so that they
    // arrive while the block counts
    const int cn_first = min(a.ctok, ntok);
    for (int k = threadIdx.x; k < cn_first * K; k += blockDim.x) s_idx[k] = __ldg(a.topk_idx + g0 * K + k);
    for (int i = threadIdx.x; i < 4 * E; i += blockDim.x) tot[i] = 0;
    if (send)
        for (int r = lane; r < R; r += 32) s_arr[r] = 0;
    // the routing table from shared memory when its copy landed (the last
    // few ids beyond the copy's 16-byte units are read here), else from global
    bool staged = false;
    if (a.stage_ids) {
        __syncthreads();   // bar_ids is initialised
        staged = mbar_wait_bounded(&bar_ids, 0u);
        for (long long i = ids_bulk / 4 + threadIdx.x; i < n_all; i += blockDim.x) s_items[i] = __ldg(a.topk_idx + i);
    }
    staged = __syncthreads_and(staged) != 0;
    if (threadIdx.x == 0) MOE_STAMP(kTrSmallStaged);
    const int32_t *ids = staged ? s_items : a.topk_idx;
    const long long pb = g0 * K;
    // Each thread takes 16 consecutive items per round and issues all their
    // loads (four 16-byte loads when the ids are 16-byte aligned) before the
    // first shared-memory atomic, so a round costs one L2 round trip.
    const bool vec_ids = (reinterpret_cast<uintptr_t>(a.topk_idx) & 15) == 0;
    auto count_pass = [&](long long lim, long long mlo, long long mhi, bool all) {
        constexpr int kU = 16;
        for (long long base = (long long)threadIdx.x * kU; base < lim; base += (long long)blockDim.x * kU) {
            int ev[kU];
            if (vec_ids && base + kU <= lim) {
#pragma unroll
                for (int q = 0; q < kU / 4; ++q) {
                    const int4 v = staged ? reinterpret_cast<const int4 *>(ids + base)[q]
                                          : __ldg(reinterpret_cast<const int4 *>(a.topk_idx + base) + q);
                    ev[4 * q] = v.x;
                    ev[4 * q + 1] = v.y;
                    ev[4 * q + 2] = v.z;
                    ev[4 * q + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int u = 0; u < kU; ++u) ev[u] = (base + u < lim) ? ids[base + u] : -1;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int e = ev[u];
                const long long i = base + u;
                if ((unsigned)e >= (unsigned)E) continue;   // out of range (reported in D) or past lim
                if (all) {
                    atomicAdd(&tot[e], 1);
                    if (i < pb) atomicAdd(&pre[e], 1);
                }
                if (i < mlo)
                    atomicAdd(&bef[e], 1);
                else if (i < mhi)
                    atomicAdd(&ins[e], 1);
            }
        }
    };
    // The first pass needs four per-expert counts: all items (tot), those
    // before g0 (pre), before rank s (bef) and inside rank s (ins).  Sorting
    // the three boundaries g0*K, rank_off[s]*K, rank_off[s+1]*K cuts the items
    // into four contiguous segments; each item adds to its segment's histogram
    // (one shared-memory atomic instead of up to four), and the four counts
    // are sums of leading segments.
    int s_meta = blockIdx.x;
    {
        const long long mlo = s_meta < R ? (long long)rt.rank_off[s_meta] * K : 0;
        const long long mhi = s_meta < R ? (long long)rt.rank_off[s_meta + 1] * K : 0;
        long long c0 = pb, c1 = mlo, c2 = mhi;   // sorted into c0 <= c1 <= c2
        if (c0 > c1) { const long long t = c0; c0 = c1; c1 = t; }
        if (c1 > c2) { const long long t = c1; c1 = c2; c2 = t; }
        if (c0 > c1) { const long long t = c0; c0 = c1; c1 = t; }
        int32_t *seg = tot;   // [4][E]: tot, pre, bef, ins reused as the segment histograms
        constexpr int kU = 16;   // items per thread per round, all loads issued before the atomics
        for (long long base = (long long)threadIdx.x * kU; base < n_all; base += (long long)blockDim.x * kU) {
            int ev[kU];
            if (vec_ids && base + kU <= n_all) {
#pragma unroll
                for (int q = 0; q < kU / 4; ++q) {
                    const int4 v = staged ? reinterpret_cast<const int4 *>(ids + base)[q]
                                          : __ldg(reinterpret_cast<const int4 *>(a.topk_idx + base) + q);
                    ev[4 * q] = v.x;
                    ev[4 * q + 1] = v.y;
                    ev[4 * q + 2] = v.z;
                    ev[4 * q + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int u = 0; u < kU; ++u) ev[u] = (base + u < n_all) ? ids[base + u] : -1;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int e = ev[u];
                const long long i = base + u;
                if ((unsigned)e >= (unsigned)E) continue;   // out of range (reported in D) or past the end
                const int sg = (i >= c0) + (i >= c1) + (i >= c2);
                atomicAdd(&seg[sg * E + e], 1);
            }
        }
        __syncthreads();
        // segment k covers [c_{k-1}, c_k): the items below a boundary are the
        // segments up to the boundary's place among c0 <= c1 <= c2
        const int r_pre = pb == c0 ? 0 : (pb == c1 ? 1 : 2);
        const int r_lo = mlo == c0 ? 0 : (mlo == c1 ? 1 : 2);
        const int r_hi = mhi == c0 ? 0 : (mhi == c1 ? 1 : 2);
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const int run0 = seg[e];
            const int run1 = run0 + seg[E + e];
            const int run2 = run1 + seg[2 * E + e];
            const int run3 = run2 + seg[3 * E + e];
            auto below = [&](int r) { return r == 0 ? run0 : (r == 1 ? run1 : run2); };
            const int lo = below(r_lo);
            tot[e] = run3;
            pre[e] = below(r_pre);
            bef[e] = lo;
            ins[e] = below(r_hi) - lo;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) MOE_STAMP(kTrSmallCounted);

    // C. start(e): exclusive scan of tot, in place, by the whole block: thread t
    // takes the consecutive entries [t*q, t*q + q) (q = ceil(E / threads), at
    // most 5), then warp sums, then the warps' totals
    {
        __shared__ int s_wsum[kSmallMaxWarps];
        const int q = (E + blockDim.x - 1) / blockDim.x;
        const int e0 = threadIdx.x * q;
        int mine = 0;
        for (int k = 0; k < q; ++k)
            if (e0 + k < E) mine += tot[e0 + k];
        const int incl = warp_inclusive_scan(mine);
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        int before = 0, all = 0;
        for (int w = 0; w < W; ++w) {
            const int ws = s_wsum[w];
            if (w < warp) before += ws;
            all += ws;
        }
        int run = before + incl - mine;
        for (int k = 0; k < q; ++k)
            if (e0 + k < E) {
                const int c = tot[e0 + k];
                tot[e0 + k] = run;
                run += c;
            }
        if (threadIdx.x == 0) s_total = all;
    }
    __syncthreads();
    const int total = s_total;
    // D. chunks.  The header (error word) and signals are cleared by the kernel
    // ahead; this kernel waits for it (griddepcontrol.wait, a no-op once it has
    // completed) only right before it first writes either -- an error bit, or
    // the send half's announcements at the end -- so the stores never wait.
    if (threadIdx.x == 0) MOE_STAMP(kTrSmallLayout);
    auto report = [&](int bits) {
        pdl_wait();
        set_device_error(a.err, bits);
    };
    int failed_at = -1;
    int it = 0;   // this warp's position in its token sequence g0 + warp + it*W
    for (long long c0 = g0; c0 < g1; c0 += a.ctok) {
        const int cn = (int)min((long long)a.ctok, g1 - c0);
        const long long cb = c0 * K;
        __syncthreads();   // the previous chunk's rows are read, and pre counts every item before c0
        if (c0 != g0) {    // the first chunk's ids were fetched in B
            for (int k = threadIdx.x; k < cn * K; k += blockDim.x) s_idx[k] = __ldg(a.topk_idx + cb + k);
            __syncthreads();
        }
        // row = start + the earlier items of the same expert: before the chunk, then inside it
        for (int k = threadIdx.x; k < cn * K; k += blockDim.x) {
            const int e = s_idx[k];
            int row = -1;
            if ((unsigned)e < (unsigned)E) {
                int rr = 0;
                for (int k2 = 0; k2 < k; ++k2) rr += (s_idx[k2] == e) ? 1 : 0;
                row = tot[e] + pre[e] + rr;
            }
            s_row[k] = row;
        }
        __syncthreads();
        for (int k = threadIdx.x; k < cn * K; k += blockDim.x) {   // pre for the next chunk
            const int e = s_idx[k];
            if ((unsigned)e < (unsigned)E) atomicAdd(&pre[e], 1);
        }
        for (; failed_at < 0 && it < my_n; ++it) {
            const long long g = g0 + warp + (long long)it * W;
            if (g >= c0 + cn) break;   // the warp's next token is in the next chunk
            const uint32_t parity = (uint32_t)((it / S) & 1);
            unsigned char *buf = stage(it);
            const int k0 = (int)(g - c0) * K;
            int my_dest = -1;
            {
                int e = -1, row = -1;
                if (lane < K) {
                    const long long i = g * K + lane;
                    e = s_idx[k0 + lane];
                    row = s_row[k0 + lane];
                    if ((unsigned)e >= (unsigned)E) {
                        report(MOE_DEVERR_EXPERT_RANGE);
                        e = -1;
                        row = -1;
                    }
                    a.tok2row[i] = row;
                    if (row >= 0) {
                        a.row2src[row] = (int32_t)i;
                        if (send) my_dest = e / L;
                    }
                }
                int dup = 0;
                for (int j = 0; j < K; ++j) {
                    const int ej = __shfl_sync(0xffffffffu, e, j);
                    if (lane < j && e >= 0 && e == ej) dup = 1;
                }
                if (__any_sync(0xffffffffu, dup) && lane == 0) report(MOE_DEVERR_DUPLICATE);
            }
            const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[warp][it % S], parity));
            if (!ok) {
                if (lane == 0) report(MOE_DEVERR_COPY_TIMEOUT);
                failed_at = it;
                break;
            }
            if (my_dest >= 0) atomicAdd(&s_arr[my_dest], 1);   // stored below
            float *sc = reinterpret_cast<float *>(buf + (size_t)H * 2);
            if (kFp8) quantize_stage(buf, H, lane);
            __syncwarp();
            if (lane == 0) MOE_STAMP(kTrSmallFirstStore);
            if (lane == 0) {
                for (int j = 0; j < K; ++j) {
                    const int row = s_row[k0 + j];
                    if (row < 0 || (unsigned)s_idx[k0 + j] >= (unsigned)E) continue;
                    bulk_store(static_cast<unsigned char *>(a.recv_x) + (size_t)row * recv_pitch, buf, out_bytes);
                    if (scale_bulk) bulk_store(a.recv_scale + (size_t)row * nblk, sc, (uint32_t)nblk * 4u);
                }
                bulk_commit();
            }
            if (kFp8 && !scale_bulk) {
                for (int t = lane; t < K * nblk; t += 32) {
                    const int j = t / nblk;
                    const int b = t - j * nblk;
                    const int row = s_row[k0 + j];
                    if (row >= 0 && (unsigned)s_idx[k0 + j] < (unsigned)E) a.recv_scale[(size_t)row * nblk + b] = sc[b];
                }
            }
            // refill the previous token's stage with token it - 1 + S once its stores have read it
            if (lane == 0 && S >= 2 && it >= 1 && it - 1 + S < my_n) {
                bulk_wait_read<1>();
                const int nxt = it - 1 + S;
                const long long gn = g0 + warp + (long long)nxt * W;
                mbar_arrive_expect_tx(&bars[warp][nxt % S], in_bytes);
                bulk_load(stage(nxt), a.x + gn * H, in_bytes, &bars[warp][nxt % S]);
            }
            __syncwarp();
        }
    }   // chunks
    // the layout of source ranks blockIdx.x, blockIdx.x + grid, ... (written after the
    // scatter: nothing in this kernel reads it, and the stores start sooner)
    for (; s_meta < R; s_meta += gridDim.x) {
        if (s_meta != (int)blockIdx.x) {   // a further rank: count again
            __syncthreads();
            for (int i = threadIdx.x; i < 2 * E; i += blockDim.x) bef[i] = 0;   // bef and ins
            __syncthreads();
            count_pass((long long)rt.rank_off[s_meta + 1] * K, (long long)rt.rank_off[s_meta] * K,
                       (long long)rt.rank_off[s_meta + 1] * K, false);
            __syncthreads();
        }
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const int o = tot[e] + bef[e];
            if (a.layout) {
                a.layout[e * R + s_meta] = o;
            } else {
                a.offsets[e * R + s_meta] = o;
                a.counts[e * R + s_meta] = ins[e];
                if (s_meta == 0) a.expert_offsets[e] = tot[e];
            }
        }
        if (s_meta == R - 1 && threadIdx.x == 0) {
            if (a.layout) {
                a.layout[E * R] = total;
            } else {
                a.offsets[E * R] = total;
                a.expert_offsets[E] = total;
            }
        }
    }
    if (a.stage_ids && !staged && threadIdx.x == 0) {
        // the routing table's copy did not land in time (the ids were read from
        // global memory): report it, and let it land before shared memory goes away
        report(MOE_DEVERR_COPY_TIMEOUT);
        (void)mbar_wait_bounded(&bar_ids, 0u);
    }
    pdl_wait();   // this grid ends after the kernel ahead, whatever path it took
    if (lane == 0) {
        if (failed_at >= 0) {
            // let every load this warp issued land before the block's shared memory goes away
            // tokens whose loads were issued: the first S, then one per refill (iterations 1 .. failed_at-1)
            const int issued = min(my_n, max(S, failed_at + S - 1));
            for (int t = failed_at; t < issued; ++t)
                (void)mbar_wait_bounded(&bars[warp][t % S], (uint32_t)((t / S) & 1));
        }
        bulk_wait_all();
        MOE_STAMP(kTrSmallWarpEnd);
        if (send) {
            fence_proxy_async_global();
            __threadfence();
        }
    }
    if (send) {
        pdl_wait();   // the arrival counters were cleared by the kernel ahead
        __syncwarp();
        for (int r = lane; r < R; r += 32) {
            const int c = s_arr[r];
#ifdef MOE_TEST_WITHHOLD_ARRIVAL_RANK
            if (r == MOE_TEST_WITHHOLD_ARRIVAL_RANK) continue;
#endif
            if (c > 0) red_release_add_gpu(a.arrive + r, c);
        }
    }
}

// --------------------------------------------------------------------------
// launcher
// --------------------------------------------------------------------------
static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

size_t signal_workspace_bytes(int R) { return kWsHeader + align256((size_t)R * 2 * 4); }

// Workspace layout for a tile count (a worst case, or the call's own).
DispatchPlan plan_dispatch(int E, int R, int ntiles) {
    DispatchPlan p{};
    p.ntiles = ntiles;
    const long long n = (long long)E * ntiles;
    p.nscan_blocks = (int)((n + kScanChunk - 1) / kScanChunk);
    if (p.nscan_blocks < 1) p.nscan_blocks = 1;
    p.off_signal = kWsHeader;   // arrive[R], then ready[R]
    p.off_status = signal_workspace_bytes(R);
    p.off_hist = p.off_status + align256((size_t)p.nscan_blocks * 8);
    p.off_scan = p.off_hist + align256((size_t)n * 4);
    p.total = p.off_scan + align256((size_t)(n + 1) * 4);
    return p;
}

int max_tiles(int R, int K, long long T) { return (int)((T * K + kTileItems - 1) / kTileItems) + R; }

// SM count of the current device, asked once per device (host threads may
// race to fill an entry; they all store the same value).
static int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n < 1) n = 1;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int device_sm_count() { return sm_count(); }

// Blocks per SM of a scatter variant at a dynamic shared-memory size on the
// current device.  The kernel's shared-memory limit is only ever raised and the
// occupancy is asked once per (kernel, device, size): both are host calls that
// would otherwise sit on every launch's critical path.
static cudaError_t kernel_blocks_per_sm(const void *kfn, int threads, size_t smem, int *per_sm) {
    struct Limit { const void *fn; int dev; size_t smem; };
    struct Occ { const void *fn; int dev; int threads; size_t smem; int per_sm; };
    static std::mutex mu;
    static Limit limits[16];
    static int nlimits = 0;
    static Occ occs[64];
    static int noccs = 0;
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return ce;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < noccs; ++i)
        if (occs[i].fn == kfn && occs[i].dev == dev && occs[i].threads == threads && occs[i].smem == smem) {
            *per_sm = occs[i].per_sm;
            return cudaSuccess;
        }
    int li = -1;
    for (int i = 0; i < nlimits; ++i)
        if (limits[i].fn == kfn && limits[i].dev == dev) li = i;
    if (li < 0 || limits[li].smem < smem) {
        if ((ce = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return ce;
        if (li >= 0)
            limits[li].smem = smem;
        else if (nlimits < 16)
            limits[nlimits++] = Limit{kfn, dev, smem};
    }
    int n = 0;
    if ((ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kfn, threads, smem)) != cudaSuccess) return ce;
    if (noccs < 64) occs[noccs++] = Occ{kfn, dev, threads, smem, n};
    *per_sm = n;
    return cudaSuccess;
}

// Persistent launch of the scatter (one wave), with programmatic stream
// serialization so that it stages its first rows while the previous kernel ends.
template <int kMode>
static const void *scatter_fn(bool fp8) {
    return fp8 ? (const void *)scatter_kernel<true, kMode> : (const void *)scatter_kernel<false, kMode>;
}

// max_sms > 0 caps the SMs the persistent grid spans (work on other streams
// can then run on the rest); the build-time MOE_SCATTER_MAX_SMS caps it too.
static cudaError_t launch_scatter(ScatterArgs a, const RankTable &rt, bool fp8, int mode, cudaStream_t stream,
                                  int max_sms = 0) {
    const long long T = a.T;
    const int H = a.H;
    cudaError_t ce;
    const size_t arrive_smem = a.arrive ? (size_t)rt.R * 4 * MOE_SCATTER_WARPS : 0;   // send half's tallies
    const size_t smem = scatter_stage_bytes(H, fp8) * MOE_SCATTER_STAGES * MOE_SCATTER_WARPS + arrive_smem;
    const void *kfn = mode == kRagged       ? scatter_fn<kRagged>(fp8)
                      : mode == kLowLatency ? scatter_fn<kLowLatency>(fp8)
                                            : scatter_fn<kLowLatencyUnordered>(fp8);
    int per_sm = 0;
    if ((ce = kernel_blocks_per_sm(kfn, MOE_SCATTER_WARPS * 32, smem, &per_sm)) != cudaSuccess) return ce;
    if (per_sm < 1) per_sm = 1;
    int sms = sm_count();
    if (MOE_SCATTER_MAX_SMS > 0 && MOE_SCATTER_MAX_SMS < sms) sms = MOE_SCATTER_MAX_SMS;
    if (max_sms > 0 && max_sms < sms) sms = max_sms;
    long long grid = (long long)sms * per_sm;   // persistent: one wave
    const long long need = (T + MOE_SCATTER_WARPS - 1) / MOE_SCATTER_WARPS;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(MOE_SCATTER_WARPS * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *params[] = {&a, const_cast<RankTable *>(&rt)};
    ce = cudaLaunchKernelExC(&cfg, kfn, params);
    if (ce != cudaSuccess) return ce;
    return cudaGetLastError();
}

bool small_dispatch(long long T, int K) { return T > 0 && T * K <= (long long)MOE_SMALL_DISPATCH_ITEMS; }

// The workspace layout of a call: the one-kernel path keeps one scan entry
// per (expert, source rank) (the send half leaves the offsets there for the
// receive half), the three-kernel path one per (expert, tile).
DispatchPlan call_plan(const RankTable &rt, int E, int K) {
    return plan_dispatch(E, rt.R, small_dispatch(rt.rank_off[rt.R], K) ? rt.R : rt.ntiles);
}

// prep (clears the header and signals) + the one-kernel dispatch
static cudaError_t launch_dispatch_small(const void *x, const int32_t *topk_idx, const RankTable &rt, int E, int K,
                                         int H, bool fp8, void *recv_x, float *recv_scale, int32_t *counts,
                                         int32_t *offsets, int32_t *expert_offsets, int32_t *tok2row,
                                         int32_t *row2src, void *workspace, bool send, int max_sms,
                                         cudaStream_t stream) {
    const long long T = rt.rank_off[rt.R];
    const DispatchPlan p = call_plan(rt, E, K);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    int32_t *signal = reinterpret_cast<int32_t *>(ws + p.off_signal);
    int sms = sm_count();
    if (max_sms > 0 && max_sms < sms) sms = max_sms;
    // warps per block: as many (up to 8) as two stages of rows per warp leave room for
    const size_t smem_cap = 227 * 1024 - 1024;
    int W = 0, tpb = 0, stages = 0;
    long long grid = 0;
    size_t smem = 0;
    for (int w = kSmallMaxWarps; w >= 1 && W == 0; --w) {
        long long gr = (T + w - 1) / w;
        if (gr > sms) gr = sms;
        const int tp = (int)((T + gr - 1) / gr);
        gr = (T + tp - 1) / tp;   // every block has at least one token
        const int st = tp > w ? kSmallStages : 1;   // one stage when every warp has one token
        const size_t sm = small_smem_bytes(w, st, H, fp8, E, rt.R, K, send);
        if (sm <= smem_cap) {
            W = w;
            tpb = tp;
            stages = st;
            grid = gr;
            smem = sm;
        }
    }
    if (W == 0) return cudaErrorInvalidConfiguration;   // unreachable for H <= MOE_MAX_HIDDEN
    // the routing table staged in shared memory when it fits beside the stages
    const size_t ids_need = small_ids_offset(W, stages, H, fp8, E, rt.R, K, send) + (((size_t)T * K * 4 + 15) & ~(size_t)15);
    const int stage_ids = ((reinterpret_cast<uintptr_t>(topk_idx) & 15) == 0 && T * K >= 4 && ids_need <= smem_cap) ? 1 : 0;
    if (stage_ids) smem = ids_need;
    const void *kfn = fp8 ? (const void *)dispatch_small_kernel<true> : (const void *)dispatch_small_kernel<false>;
    int per_sm = 0;
    cudaError_t ce;
    if ((ce = kernel_blocks_per_sm(kfn, W * 32, smem, &per_sm)) != cudaSuccess) return ce;

    dispatch_prep_kernel<<<1, 256, 0, stream>>>(reinterpret_cast<int32_t *>(ws), signal, 2 * rt.R);
    if ((ce = cudaGetLastError()) != cudaSuccess) return ce;

    SmallArgs a{};
    a.x = static_cast<const __nv_bfloat16 *>(x);
    a.topk_idx = topk_idx;
    a.recv_x = recv_x;
    a.recv_scale = recv_scale;
    a.counts = counts;
    a.offsets = offsets;
    a.expert_offsets = expert_offsets;
    a.layout = send ? reinterpret_cast<int32_t *>(ws + p.off_scan) : nullptr;
    a.tok2row = tok2row;
    a.row2src = row2src;
    a.err = reinterpret_cast<int32_t *>(ws);
    a.arrive = send ? signal : nullptr;
    a.T = (int)T;
    a.E = E;
    a.K = K;
    a.H = H;
    a.tpb = tpb;
    a.ctok = small_chunk_tokens(W, K);
    a.stages = stages;
    a.stage_ids = stage_ids;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(W * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *params[] = {&a, const_cast<RankTable *>(&rt)};
    if ((ce = cudaLaunchKernelExC(&cfg, kfn, params)) != cudaSuccess) return ce;
    return cudaGetLastError();
}

// hist + scan + scatter; send: the split dispatch's send half (arrival
// counters instead of counts / offsets / expert_offsets).
static cudaError_t launch_dispatch_impl(const void *x, const int32_t *topk_idx, const RankTable &rt, int E, int K,
                                        int H, bool fp8, void *recv_x, float *recv_scale, int32_t *counts,
                                        int32_t *offsets, int32_t *expert_offsets, int32_t *tok2row,
                                        int32_t *row2src, void *workspace, bool send, int max_sms,
                                        cudaStream_t stream) {
    const long long T = rt.rank_off[rt.R];
    if (small_dispatch(T, K))
        return launch_dispatch_small(x, topk_idx, rt, E, K, H, fp8, recv_x, recv_scale, counts, offsets,
                                     expert_offsets, tok2row, row2src, workspace, send, max_sms, stream);
    const DispatchPlan p = plan_dispatch(E, rt.R, rt.ntiles);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    int32_t *err = reinterpret_cast<int32_t *>(ws);
    int32_t *ticket = reinterpret_cast<int32_t *>(ws + 4);   // scan block start order
    int32_t *signal = reinterpret_cast<int32_t *>(ws + p.off_signal);
    unsigned long long *status = reinterpret_cast<unsigned long long *>(ws + p.off_status);
    int32_t *tile_hist = reinterpret_cast<int32_t *>(ws + p.off_hist);
    int32_t *scan = reinterpret_cast<int32_t *>(ws + p.off_scan);

    cudaError_t ce;
    const size_t hist_smem = (size_t)kHistWarps * E * 4;
    tile_hist_kernel<<<rt.ntiles, kHistThreads, hist_smem, stream>>>(topk_idx, E, K, rt, tile_hist, tok2row, err,
                                                                     signal, 2 * rt.R, status, p.nscan_blocks);
    if ((ce = cudaGetLastError()) != cudaSuccess) return ce;

    const int n = E * rt.ntiles;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)p.nscan_blocks);
        cfg.blockDim = dim3(kScanThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((ce = cudaLaunchKernelEx(&cfg, lookback_scan_kernel, (const int32_t *)tile_hist, scan, n, status, ticket,
                                     err)) != cudaSuccess)
            return ce;
    }

    ScatterArgs a{};
    a.x = static_cast<const __nv_bfloat16 *>(x);
    a.topk_idx = topk_idx;
    a.scan = scan;
    a.recv_x = recv_x;
    a.recv_scale = recv_scale;
    a.counts = counts;
    a.offsets = offsets;
    a.expert_offsets = expert_offsets;
    a.tok2row = tok2row;
    a.row2src = row2src;
    a.err = err;
    a.next_token = reinterpret_cast<int32_t *>(ws + 8);   // scatter token counter
    a.arrive = send ? signal : nullptr;
    a.T = (int)T;
    a.E = E;
    a.K = K;
    a.H = H;
    return launch_scatter(a, rt, fp8, kRagged, stream, max_sms);
}

cudaError_t launch_dispatch(const void *x, const int32_t *topk_idx, const RankTable &rt, int E, int K, int H,
                            bool fp8, void *recv_x, float *recv_scale, int32_t *counts, int32_t *offsets,
                            int32_t *expert_offsets, int32_t *tok2row, int32_t *row2src, void *workspace,
                            cudaStream_t stream) {
    return launch_dispatch_impl(x, topk_idx, rt, E, K, H, fp8, recv_x, recv_scale, counts, offsets, expert_offsets,
                                tok2row, row2src, workspace, false, 0, stream);
}

cudaError_t launch_dispatch_send(const void *x, const int32_t *topk_idx, const RankTable &rt, int E, int K, int H,
                                 bool fp8, void *recv_x, float *recv_scale, int32_t *tok2row, int32_t *row2src,
                                 void *workspace, int max_sms, cudaStream_t stream) {
    return launch_dispatch_impl(x, topk_idx, rt, E, K, H, fp8, recv_x, recv_scale, nullptr, nullptr, nullptr,
                                tok2row, row2src, workspace, true, max_sms, stream);
}

// --------------------------------------------------------------------------
// receive half of the split dispatch
// --------------------------------------------------------------------------
// Perplexity, "Enabling trillion-parameter models on AWS EFA", "Dispatch and
// combine": the receiver blocks until every transfer to it has landed, then
// hands the rows to the grouped GEMM.  Block r is destination rank r: thread 0
// waits (bounded) until the copies announced for rank r equal the rows its
// experts own in the scanned layout, consumes the counter (so a second
// receive without a new send waits again), and the block writes the
// receiver-side layout of rank r's experts: counts, offsets, expert_offsets.
// A wait is skipped when the routing was already reported bad (the copies
// never placed are then not awaited).
__global__ void __launch_bounds__(256) dispatch_recv_kernel(const int32_t *__restrict__ scan,
                                                            const __grid_constant__ RankTable rt, int E,
                                                            int32_t *arrive, int32_t *err, int32_t *__restrict__ counts,
                                                            int32_t *__restrict__ offsets,
                                                            int32_t *__restrict__ expert_offsets) {
    const int r = blockIdx.x;
    const int R = rt.R;
    const int L = E / R;
    const long long nt = rt.ntiles;
    if (threadIdx.x == 0) {
        const int expected = scan[(long long)(r + 1) * L * nt] - scan[(long long)r * L * nt];
        if (ld_acquire_gpu(arrive + r) != expected) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_gpu(arrive + r) != expected) {
                if (ld_acquire_gpu(err) & (MOE_DEVERR_EXPERT_RANGE | MOE_DEVERR_DUPLICATE)) break;
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    set_device_error(err, MOE_DEVERR_RECV_TIMEOUT);
                    break;
                }
                __nanosleep(64);
            }
        }
        arrive[r] = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < L * R; i += blockDim.x) {
        const int e = r * L + i / R;
        const int s = i - (i / R) * R;
        const int o = scan[(long long)e * nt + rt.tile_off[s]];
        const int o1 = scan[(long long)e * nt + rt.tile_off[s + 1]];
        offsets[e * R + s] = o;
        counts[e * R + s] = o1 - o;
        if (s == 0) expert_offsets[e] = o;
    }
    if (r == R - 1 && threadIdx.x == 0) {
        const int total = scan[(long long)E * nt];
        offsets[E * R] = total;
        expert_offsets[E] = total;
    }
}

cudaError_t launch_dispatch_recv(const RankTable &rt_in, int E, int K, int32_t *counts, int32_t *offsets,
                                 int32_t *expert_offsets, void *workspace, cudaStream_t stream) {
    const DispatchPlan p = call_plan(rt_in, E, K);
    RankTable rt = rt_in;
    if (small_dispatch(rt.rank_off[rt.R], K)) {   // the send half left offsets[e*R + s]: one "tile" per rank
        rt.ntiles = rt.R;
        for (int s = 0; s <= rt.R; ++s) rt.tile_off[s] = s;
    }
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    dispatch_recv_kernel<<<rt.R, 256, 0, stream>>>(reinterpret_cast<const int32_t *>(ws + p.off_scan), rt, E,
                                                   reinterpret_cast<int32_t *>(ws + p.off_signal),
                                                   reinterpret_cast<int32_t *>(ws), counts, offsets, expert_offsets);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_ll(const void *x, const int32_t *topk_idx, const RankTable &rt, int E, int K, int H,
                               int C, bool fp8, void *recv_x, float *recv_scale, int32_t *counts, int32_t *tok2row,
                               int32_t *row2src, void *workspace, cudaStream_t stream) {
    const long long T = rt.rank_off[rt.R];
    const DispatchPlan p = plan_dispatch(E, rt.R, rt.ntiles);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    int32_t *err = reinterpret_cast<int32_t *>(ws);
    int32_t *tile_hist = reinterpret_cast<int32_t *>(ws + p.off_hist);

    cudaError_t ce;
    const size_t hist_smem = (size_t)kHistWarps * E * 4;
    tile_hist_kernel<<<rt.ntiles, kHistThreads, hist_smem, stream>>>(topk_idx, E, K, rt, tile_hist, tok2row, err,
                                                                     nullptr, 0, nullptr, 0);
    if ((ce = cudaGetLastError()) != cudaSuccess) return ce;

    ScatterArgs a{};
    a.x = static_cast<const __nv_bfloat16 *>(x);
    a.topk_idx = topk_idx;
    a.recv_x = recv_x;
    a.recv_scale = recv_scale;
    a.counts = counts;
    a.tok2row = tok2row;
    a.row2src = row2src;
    a.err = err;
    a.next_token = reinterpret_cast<int32_t *>(ws + 8);   // scatter token counter
    a.tile_hist = tile_hist;
    a.T = (int)T;
    a.E = E;
    a.K = K;
    a.H = H;
    a.C = C;
    return launch_scatter(a, rt, fp8, kLowLatency, stream);
}


// Zero the workspace header (error word, token counter) and the region counts
// of the unordered low-latency dispatch; the scatter (launched with
// programmatic stream serialization) stages its first rows meanwhile and
// waits for this grid before it touches either.
__global__ void zero_counts_kernel(int32_t *__restrict__ header, int32_t *__restrict__ counts, int n) {
    pdl_launch_dependents();
    const int tid = blockIdx.x * blockDim.x + threadIdx.x;
    if (tid < (int)(kWsHeader / 4)) header[tid] = 0;
    for (int i = tid; i < n; i += gridDim.x * blockDim.x) counts[i] = 0;
}

cudaError_t launch_dispatch_ll_unordered(const void *x, const int32_t *topk_idx, const RankTable &rt, int E, int K,
                                         int H, int C, bool fp8, void *recv_x, float *recv_scale, int32_t *counts,
                                         int32_t *tok2row, int32_t *row2src, void *workspace, cudaStream_t stream) {
    const long long T = rt.rank_off[rt.R];
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    int32_t *err = reinterpret_cast<int32_t *>(ws);

    cudaError_t ce;
    const int n = E * rt.R;
    const int zblocks = (n + 1023) / 1024 < 64 ? (n + 1023) / 1024 : 64;
    zero_counts_kernel<<<zblocks, 1024, 0, stream>>>(err, counts, n);
    if ((ce = cudaGetLastError()) != cudaSuccess) return ce;

    ScatterArgs a{};
    a.x = static_cast<const __nv_bfloat16 *>(x);
    a.topk_idx = topk_idx;
    a.recv_x = recv_x;
    a.recv_scale = recv_scale;
    a.counts = counts;
    a.tok2row = tok2row;
    a.row2src = row2src;
    a.err = err;
    a.next_token = reinterpret_cast<int32_t *>(ws + 8);   // scatter token counter
    a.T = (int)T;
    a.E = E;
    a.K = K;
    a.H = H;
    a.C = C;
    return launch_scatter(a, rt, fp8, kLowLatencyUnordered, stream);
}

MOE_TRACE_READER(moe_trace_dispatch)

}  // namespace moe
