// combine.cu -- gather each token's K expert outputs and take their
// routing-weighted sum.
//
// Sources:
//  * lehuy.net, "Decoding high-performance EP kernels", "Optimising for
//    throughput" > "Combine": undo the permutation dispatch applied, bring the
//    outputs back to their source slots and add up each token's
//    contributions; the routing dispatch produced is reused, so no
//    coordination pass is needed.
//  * Perplexity, "Enabling trillion-parameter models on AWS EFA", "Dispatch
//    and combine": the combine receiver accumulates the returned tokens into
//    the output tensors (accumulation on the receiving side).
//
// On one GPU the return trip is a gather: token g reads rows tok2row[g*K+j]
// of y directly.  Each thread owns 16-byte column chunks (8 bf16 channels) of
// the token's row; for a chunk it issues the K row loads (up to 8 at a time,
// all in flight together), then folds them into 8 fp32 accumulators with
// fused multiply-adds in the fixed order j = 0..K-1, and writes bf16 (round
// to nearest even) or fp32.  One block per token (the kernel also walks
// tokens grid-stride, should a caller launch fewer blocks); weights and rows
// of the token sit in shared memory.
#include <cuda_bf16.h>

#include "launch.h"
#include "trace.cuh"

namespace moe {

MOE_TRACE_DEFINE()

constexpr int kCombineThreads = 128;
constexpr int kCombineBatch = 8;   // row loads in flight per chunk
// blocks per token, each summing one contiguous part of the token's columns: two halve the
// work a block holds, which shortens the launch's tail (DeepSeek-V3 prefill: 612.4-612.7 us
// against 616.5-616.6 us with one block per token; three or four blocks were slower)
constexpr int kCombineSplit = 2;

// bf16 pair (low half = first element) -> two fp32, exactly (bf16 is the high
// half of an fp32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even
    return (uint32_t)__bfloat16_as_ushort(h.x) | ((uint32_t)__bfloat16_as_ushort(h.y) << 16);
}

// acc[0..7] += w * (8 bf16 channels of v), in channel order.
__device__ __forceinline__ void fma_row(float (&acc)[8], float w, const uint4 v) {
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        acc[2 * k] = __fmaf_rn(w, bf16_lo(q[k]), acc[2 * k]);
        acc[2 * k + 1] = __fmaf_rn(w, bf16_hi(q[k]), acc[2 * k + 1]);
    }
}

// tok2row == nullptr reads row g*K + j (the layout a push-style return leaves
// on the origin rank); rows = number of rows of y (indices outside are skipped).
// kAfterWait: launched with programmatic stream serialization behind the
// combine receive half's wait kernel; nothing is read before that grid is done.
template <bool kOutF32, bool kAfterWait = false>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __nv_bfloat16 *__restrict__ y,
                                                                  const int32_t *__restrict__ tok2row,
                                                                  const float *__restrict__ topk_w, int T, int K,
                                                                  int H, long long rows, void *__restrict__ out) {
    __shared__ int32_t s_row[MOE_MAX_TOPK];
    __shared__ float s_w[MOE_MAX_TOPK];
    const int nchunk = H / 8;
    if (kAfterWait) pdl_wait();
    if (threadIdx.x == 0) MOE_STAMP(kTrCombineStart);

    // block b takes token b / kCombineSplit and its part b % kCombineSplit of the 16-byte chunks
    const int part = (int)(blockIdx.x % kCombineSplit);
    const int c_lo = (int)((long long)nchunk * part / kCombineSplit);
    const int c_hi = (int)((long long)nchunk * (part + 1) / kCombineSplit);
    for (long long g = blockIdx.x / kCombineSplit; g < T; g += gridDim.x / kCombineSplit) {
        __syncthreads();   // previous token's readers are done with s_row / s_w
        if (threadIdx.x < K) {
            const long long r = tok2row ? (long long)__ldg(tok2row + g * K + threadIdx.x) : g * K + threadIdx.x;
            s_row[threadIdx.x] = (r >= 0 && r < rows) ? (int32_t)r : -1;
            s_w[threadIdx.x] = __ldg(topk_w + g * K + threadIdx.x);
        }
        __syncthreads();

        for (int c = c_lo + threadIdx.x; c < c_hi; c += blockDim.x) {
            float acc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
            for (int j0 = 0; j0 < K; j0 += kCombineBatch) {
                uint4 v[kCombineBatch];
#pragma unroll
                for (int jj = 0; jj < kCombineBatch; ++jj) {
                    const int j = j0 + jj;
                    const int r = (j < K) ? s_row[j] : -1;
                    v[jj] = (r >= 0) ? ld_stream_v4(y + (size_t)r * H + (size_t)c * 8) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int jj = 0; jj < kCombineBatch; ++jj) {
                    const int j = j0 + jj;
                    if (j < K && s_row[j] >= 0) fma_row(acc, s_w[j], v[jj]);
                }
            }
            if (kOutF32) {
                float *o = static_cast<float *>(out) + (size_t)g * H + (size_t)c * 8;
                st_v4(o, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                                    __float_as_uint(acc[3])));
                st_v4(o + 4, make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]), __float_as_uint(acc[6]),
                                        __float_as_uint(acc[7])));
            } else {
                st_v4(static_cast<__nv_bfloat16 *>(out) + (size_t)g * H + (size_t)c * 8,
                      make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                                 pack_bf16x2(acc[6], acc[7])));
            }
        }
    }
#ifdef MOE_TRACE
    __syncthreads();
    if (threadIdx.x == 0) MOE_STAMP(kTrCombineEnd);
#endif
}

cudaError_t launch_combine(const void *y, const int32_t *tok2row, const float *topk_w, int T, int K, int H,
                           bool out_f32, void *out, long long rows, cudaStream_t stream) {
    // kCombineSplit blocks per token: the hardware hands each SM new work as soon as one
    // of its blocks finishes, which balances the row gathers better than any
    // fixed grid-stride split (measured: 16 blocks per SM walking the tokens
    // was 2 % slower on the DeepSeek-V3 prefill layer)
    long long grid = T * (long long)kCombineSplit;
    if (grid < 1) grid = kCombineSplit;
    const __nv_bfloat16 *yb = static_cast<const __nv_bfloat16 *>(y);
    if (out_f32)
        combine_kernel<true><<<(unsigned)grid, kCombineThreads, 0, stream>>>(yb, tok2row, topk_w, T, K, H, rows, out);
    else
        combine_kernel<false><<<(unsigned)grid, kCombineThreads, 0, stream>>>(yb, tok2row, topk_w, T, K, H, rows, out);
    return cudaGetLastError();
}

// --------------------------------------------------------------------------
// split combine: send and receive halves
// --------------------------------------------------------------------------
// Perplexity, "Enabling trillion-parameter models on AWS EFA": combine, like
// dispatch, is split into a sender half and a receiver half so the GPU can run
// other work while transfers are pending ("MoE all-to-all over EFA"); the
// receiver waits for completion and then accumulates the returned tokens into
// the output ("Dispatch and combine"); within a node the buffers are mapped
// into the peers, which push or pull tokens directly ("Send and receive
// buffers").  Here every rank's expert outputs already sit in the one HBM, so
// the send half publishes them: one release store per expert rank, ready[r] = 1.
// The receive half waits (bounded) for every rank's flag, consumes it, and
// pulls each token's K rows for the same fixed-order weighted sum as
// moe_combine (the sum kernel is launched behind the wait with programmatic
// stream serialization, so its blocks are resident when the wait ends).
__global__ void combine_send_kernel(int32_t *ready, int R) {
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
#ifdef MOE_TEST_WITHHOLD_READY_RANK
        // Test builds only: this rank never publishes, so the receive half's
        // bounded wait runs out.
        if (r == MOE_TEST_WITHHOLD_READY_RANK) continue;
#endif
        st_release_gpu(ready + r, 1);
    }
}

__global__ void combine_wait_kernel(int32_t *ready, int R, int32_t *err) {
    pdl_launch_dependents();   // the sum kernel may launch; it waits for this grid to finish
    bool timed_out = false;
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        if (ld_acquire_gpu(ready + r) != 1) {
            const uint64_t t0 = global_timer_ns();
            while (!timed_out && ld_acquire_gpu(ready + r) != 1) {
                if (global_timer_ns() - t0 > kWaitLimitNs) timed_out = true;
                else __nanosleep(64);
            }
        }
        ready[r] = 0;   // consumed: a second receive without a new send waits again
    }
    if (timed_out) set_device_error(err, MOE_DEVERR_RECV_TIMEOUT);
}

cudaError_t launch_combine_send(int R, void *workspace, cudaStream_t stream) {
    int32_t *ready = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + kWsHeader) + R;
    combine_send_kernel<<<1, 256, 0, stream>>>(ready, R);
    return cudaGetLastError();
}

cudaError_t launch_combine_recv(const void *y, const int32_t *tok2row, const float *topk_w, int T, int K, int H,
                                bool out_f32, void *out, int R, void *workspace, cudaStream_t stream) {
    int32_t *err = static_cast<int32_t *>(workspace);
    int32_t *ready = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + kWsHeader) + R;
    combine_wait_kernel<<<1, 256, 0, stream>>>(ready, R, err);
    cudaError_t ce = cudaGetLastError();
    if (ce != cudaSuccess) return ce;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((T > 0 ? T : 1) * kCombineSplit));   // the blocks of moe_combine
    cfg.blockDim = dim3(kCombineThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const __nv_bfloat16 *yb = static_cast<const __nv_bfloat16 *>(y);
    const long long rows = (long long)T * K;
    if (out_f32)
        ce = cudaLaunchKernelEx(&cfg, combine_kernel<true, true>, yb, tok2row, topk_w, T, K, H, rows, out);
    else
        ce = cudaLaunchKernelEx(&cfg, combine_kernel<false, true>, yb, tok2row, topk_w, T, K, H, rows, out);
    return ce;
}

// --------------------------------------------------------------------------
// push-style return of the low-latency layout
// --------------------------------------------------------------------------
// lehuy.net, "Decoding high-performance EP kernels", "Optimising for latency":
// dispatch tagged each token with its origin, so the expert's host writes each
// output straight to a private slot on the origin rank indexed by the token's
// position there and by which of its K experts produced it.  Here: blocks walk
// the (expert, source rank) regions; a block reads the region's count once and
// its warps copy the filled rows, 16 bytes per lane, to ret[row2src[row]].
constexpr int kPushThreads = 128;

__global__ void __launch_bounds__(kPushThreads) combine_push_kernel(const __nv_bfloat16 *__restrict__ y,
                                                                    const int32_t *__restrict__ row2src,
                                                                    const int32_t *__restrict__ counts, int C, int H,
                                                                    long long regions, long long ret_rows,
                                                                    __nv_bfloat16 *__restrict__ ret) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    for (long long region = blockIdx.x; region < regions; region += gridDim.x) {
        const int n = min(__ldg(counts + region), C);
        for (int slot = warp; slot < n; slot += nwarps) {
            const long long r = region * C + slot;
            const long long dst = __ldg(row2src + r);
            if (dst < 0 || dst >= ret_rows) continue;
            const __nv_bfloat16 *src = y + r * H;
            __nv_bfloat16 *d = ret + dst * H;
            for (int c = lane; c < H / 8; c += 32) st_v4(d + (size_t)c * 8, ld_stream_v4(src + (size_t)c * 8));
        }
    }
}

cudaError_t launch_combine_push(const void *y, const int32_t *row2src, const int32_t *counts, int C, int H,
                                long long rect_rows, long long ret_rows, void *ret, cudaStream_t stream) {
    const long long regions = rect_rows / C;
    long long grid = regions;
    const long long cap = (long long)device_sm_count() * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    combine_push_kernel<<<(unsigned)grid, kPushThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(y), row2src,
                                                                     counts, C, H, regions, ret_rows,
                                                                     static_cast<__nv_bfloat16 *>(ret));
    return cudaGetLastError();
}

// --------------------------------------------------------------------------
// sender-side partial accumulation
// --------------------------------------------------------------------------
// Perplexity, "Enabling trillion-parameter models on AWS EFA", "Evaluation":
// DeepEP accumulates on the sending side of combine to reduce the bytes
// returned, which may affect precision (pplx accumulates on the receiving
// side, as moe_combine does).  Send: for each token g and each rank r hosting
// some of g's experts (e / (E/R) == r), the partial
//   p[g,r] = bf16(fp32 fma over those copies, ascending j, from +0)
// goes to slot g*K + j0 (j0 = the rank's first copy).  Receive: the origin adds
// its partials in ascending rank order in fp32 from +0.

// Token g's copies ordered by (rank, j) in shared memory (thread 0; K <= 32):
// ord[k] = copy index, first/last mark the ends of each rank's run, slot[k] is
// the run's first copy.
struct PartialPlan {
    int32_t ord[MOE_MAX_TOPK];
    int32_t slot[MOE_MAX_TOPK];
    unsigned char first[MOE_MAX_TOPK];
    unsigned char last[MOE_MAX_TOPK];
};

__device__ __forceinline__ void plan_partials(const int32_t *idx_g, int K, int L, PartialPlan &pp) {
    int rank[MOE_MAX_TOPK];
    for (int j = 0; j < K; ++j) {
        const int e = idx_g[j];
        rank[j] = e >= 0 ? e / L : -1;
        pp.ord[j] = j;
    }
    for (int a = 1; a < K; ++a) {   // insertion sort by (rank, j): stable, so j stays ascending
        const int v = pp.ord[a];
        int b2 = a - 1;
        while (b2 >= 0 && rank[pp.ord[b2]] > rank[v]) {
            pp.ord[b2 + 1] = pp.ord[b2];
            --b2;
        }
        pp.ord[b2 + 1] = v;
    }
    int j0 = -1;
    for (int k = 0; k < K; ++k) {
        const bool f = k == 0 || rank[pp.ord[k]] != rank[pp.ord[k - 1]];
        if (f) j0 = pp.ord[k];
        pp.first[k] = f;
        pp.last[k] = (k == K - 1) || rank[pp.ord[k + 1]] != rank[pp.ord[k]];
        pp.slot[k] = j0;
    }
}

__global__ void __launch_bounds__(kCombineThreads) combine_partial_send_kernel(
    const __nv_bfloat16 *__restrict__ y, const int32_t *__restrict__ tok2row, const int32_t *__restrict__ topk_idx,
    const float *__restrict__ topk_w, int T, int K, int H, int L, long long rows, __nv_bfloat16 *__restrict__ partial) {
    __shared__ PartialPlan pp;
    __shared__ int32_t s_row[MOE_MAX_TOPK];
    __shared__ float s_w[MOE_MAX_TOPK];
    const int nchunk = H / 8;
    for (long long g = blockIdx.x; g < T; g += gridDim.x) {
        __syncthreads();
        if (threadIdx.x < K) {
            const long long r = __ldg(tok2row + g * K + threadIdx.x);
            s_row[threadIdx.x] = (r >= 0 && r < rows) ? (int32_t)r : -1;
            s_w[threadIdx.x] = __ldg(topk_w + g * K + threadIdx.x);
        }
        if (threadIdx.x == 0) plan_partials(topk_idx + g * K, K, L, pp);
        __syncthreads();
        for (int c = threadIdx.x; c < nchunk; c += blockDim.x) {
            float acc[8];
            for (int k0 = 0; k0 < K; k0 += kCombineBatch) {
                uint4 v[kCombineBatch];
#pragma unroll
                for (int kk = 0; kk < kCombineBatch; ++kk) {
                    const int k = k0 + kk;
                    const int r = (k < K) ? s_row[pp.ord[k]] : -1;
                    v[kk] = (r >= 0) ? ld_stream_v4(y + (size_t)r * H + (size_t)c * 8) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int kk = 0; kk < kCombineBatch; ++kk) {
                    const int k = k0 + kk;
                    if (k >= K) break;
                    if (pp.first[k]) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
                    }
                    const int j = pp.ord[k];
                    if (s_row[j] >= 0) {
                        const float w = s_w[j];
                        const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&v[kk]);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = __bfloat1622float2(h2[q]);
                            acc[2 * q] = __fmaf_rn(w, f.x, acc[2 * q]);
                            acc[2 * q + 1] = __fmaf_rn(w, f.y, acc[2 * q + 1]);
                        }
                    }
                    if (pp.last[k]) {
                        uint4 pk;
                        __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                        for (int q = 0; q < 4; ++q) p2[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
                        st_v4(partial + ((size_t)g * K + pp.slot[k]) * H + (size_t)c * 8, pk);
                    }
                }
            }
        }
    }
}

template <bool kOutF32>
__global__ void __launch_bounds__(kCombineThreads) combine_partial_recv_kernel(
    const __nv_bfloat16 *__restrict__ partial, const int32_t *__restrict__ topk_idx, int T, int K, int H, int L,
    void *__restrict__ out) {
    __shared__ PartialPlan pp;
    __shared__ int32_t s_slots[MOE_MAX_TOPK];
    __shared__ int s_n;
    const int nchunk = H / 8;
    for (long long g = blockIdx.x; g < T; g += gridDim.x) {
        __syncthreads();
        if (threadIdx.x == 0) {
            plan_partials(topk_idx + g * K, K, L, pp);
            int n = 0;
            for (int k = 0; k < K; ++k)
                if (pp.first[k] && topk_idx[g * K + pp.ord[k]] >= 0) s_slots[n++] = pp.ord[k];   // ascending rank
            s_n = n;
        }
        __syncthreads();
        const int n = s_n;
        for (int c = threadIdx.x; c < nchunk; c += blockDim.x) {
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
            for (int i0 = 0; i0 < n; i0 += kCombineBatch) {
                uint4 v[kCombineBatch];
#pragma unroll
                for (int ii = 0; ii < kCombineBatch; ++ii) {
                    const int i = i0 + ii;
                    v[ii] = (i < n) ? ld_stream_v4(partial + ((size_t)g * K + s_slots[i]) * H + (size_t)c * 8)
                                    : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int ii = 0; ii < kCombineBatch; ++ii) {
                    if (i0 + ii >= n) break;
                    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&v[ii]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 f = __bfloat1622float2(h2[q]);
                        acc[2 * q] = __fadd_rn(acc[2 * q], f.x);
                        acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], f.y);
                    }
                }
            }
            if (kOutF32) {
                float *o = static_cast<float *>(out) + (size_t)g * H + (size_t)c * 8;
                st_v4(o, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                                    __float_as_uint(acc[3])));
                st_v4(o + 4, make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]), __float_as_uint(acc[6]),
                                        __float_as_uint(acc[7])));
            } else {
                uint4 pk;
                __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                for (int q = 0; q < 4; ++q) p2[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
                st_v4(static_cast<__nv_bfloat16 *>(out) + (size_t)g * H + (size_t)c * 8, pk);
            }
        }
    }
}

cudaError_t launch_combine_partial(const void *y, const int32_t *tok2row, const int32_t *topk_idx,
                                   const float *topk_w, int T, int K, int H, int E, int R, void *partial,
                                   cudaStream_t stream) {
    // one block per token: the hardware hands each SM a new token as soon as one
    // of its blocks finishes, which balances the row gathers better than any
    // fixed grid-stride split (measured: 16 blocks per SM walking the tokens
    // was 2 % slower on the DeepSeek-V3 prefill layer)
    long long grid = T;
    if (grid < 1) grid = 1;
    combine_partial_send_kernel<<<(unsigned)grid, kCombineThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(y), tok2row, topk_idx, topk_w, T, K, H, E / R, (long long)T * K,
        static_cast<__nv_bfloat16 *>(partial));
    return cudaGetLastError();
}

cudaError_t launch_combine_partial_recv(const void *partial, const int32_t *topk_idx, int T, int K, int H, int E,
                                        int R, bool out_f32, void *out, cudaStream_t stream) {
    // one block per token: the hardware hands each SM a new token as soon as one
    // of its blocks finishes, which balances the row gathers better than any
    // fixed grid-stride split (measured: 16 blocks per SM walking the tokens
    // was 2 % slower on the DeepSeek-V3 prefill layer)
    long long grid = T;
    if (grid < 1) grid = 1;
    const __nv_bfloat16 *pb = static_cast<const __nv_bfloat16 *>(partial);
    if (out_f32)
        combine_partial_recv_kernel<true><<<(unsigned)grid, kCombineThreads, 0, stream>>>(pb, topk_idx, T, K, H, E / R,
                                                                                          out);
    else
        combine_partial_recv_kernel<false><<<(unsigned)grid, kCombineThreads, 0, stream>>>(pb, topk_idx, T, K, H,
                                                                                           E / R, out);
    return cudaGetLastError();
}

MOE_TRACE_READER(moe_trace_combine)

}  // namespace moe
