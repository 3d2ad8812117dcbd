/*
 * moe_route.h -- C ABI of libmoeroute: MoE expert-parallel routing, dispatch
 * and combine for one GB300 (sm_103a), with R expert-parallel ranks emulated
 * inside that one GPU's HBM.
 *
 * Sources (web pages, cited by title and section):
 *   [DSD] Perplexity, "Lower latency and higher throughput with multi-node
 *         DeepSeek deployment": "Expert parallelism", "Quantization",
 *         "CUDA Graph", "MoE router".
 *   [EFA] Perplexity, "Enabling trillion-parameter models on AWS EFA":
 *         "Send and receive buffers", "Dispatch and combine".
 *   [EPK] lehuy.net, "Decoding high-performance EP kernels" ("Giai ma nhan
 *         EP hieu suat cao"): "Our task", "Optimising for throughput: ask
 *         first, send later" > "Dispatch" / "Combine".
 *
 * Problem statement ([EPK] "Our task"): R ranks; rank s holds B[s] tokens of
 * hidden size H; E routed experts, E/R of them on each rank (expert e lives on
 * rank e / (E/R)); every token is routed to K experts.  Tokens are numbered
 * globally in rank-major order, g = rank_off[s] + t with
 * rank_off[s] = B[0] + ... + B[s-1] and T = rank_off[R].
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device (global) memory on the current
 *     device; pointers marked "host" are ordinary host memory read during the
 *     call.  The caller allocates and owns every buffer; the library never
 *     allocates, frees or synchronises (except moe_get_device_error, which
 *     says so).  Work is enqueued on `stream` and runs asynchronously, and
 *     the calls take no host-device synchronisation.  A layer of
 *     moe_route_topk, moe_dispatch (or moe_dispatch_ll[_unordered]),
 *     moe_expert_scale and moe_combine (or moe_combine_ll) can therefore be
 *     captured in a CUDA graph and replayed ([DSD] "CUDA Graph").
 *   - Arrays are dense, row-major, with no padding between rows.
 *   - Arguments are validated on the host before anything is enqueued; a bad
 *     argument returns MOE_ERR_INVALID_ARG (or MOE_ERR_UNSUPPORTED for a
 *     pointer alignment the kernels cannot use) and enqueues nothing.  A CUDA
 *     launch failure returns MOE_ERR_CUDA.  Errors that only the device can
 *     see (an expert id out of range, a repeated expert within one token, a
 *     bounded device wait that ran out) are recorded in the workspace's error
 *     word and read with moe_get_device_error.  No call aborts, traps or
 *     throws across this boundary.
 *   - bf16 is IEEE binary32 truncated to its top 16 bits with round to
 *     nearest even; fp8 is OCP E4M3 (bias 7, largest finite 448, no inf).
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ROUTE_ABI_VERSION 1

/* Symbols of this header are the only ones the shared library exports. */
#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* Limits checked by the argument validation. */
#define MOE_MAX_RANKS 256      /* R */
#define MOE_MAX_EXPERTS 1024   /* E */
#define MOE_MAX_TOPK 32        /* K */
#define MOE_MAX_HIDDEN 16384   /* H */
#define MOE_MAX_GROUPS 32      /* expert groups of moe_route_topk_grouped */

/* A CUDA stream (the same type as cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* a NULL, a size out of range, an inconsistent shape */
    MOE_ERR_UNSUPPORTED = 2,   /* a pointer not aligned to 16 bytes */
    MOE_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    MOE_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required */
    MOE_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out (see moe_get_device_error) */
    MOE_ERR_BAD_ROUTING = 6    /* device: expert id out of range or repeated within a token */
} moe_status;

typedef enum {
    MOE_DTYPE_BF16 = 0,
    MOE_DTYPE_FP8_E4M3 = 1,
    MOE_DTYPE_FP32 = 2
} moe_dtype;

/* Device error word bits (moe_get_device_error's *host_code). */
#define MOE_DEVERR_EXPERT_RANGE 0x1   /* a topk_idx entry outside [0, E) */
#define MOE_DEVERR_DUPLICATE 0x2      /* the same expert twice in one token's top-K */
#define MOE_DEVERR_SCAN_TIMEOUT 0x4   /* the decoupled-lookback wait ran out */
#define MOE_DEVERR_COPY_TIMEOUT 0x8   /* a bulk-copy barrier wait ran out */
#define MOE_DEVERR_RECV_TIMEOUT 0x10  /* a receive half's wait for its send half ran out */

/* Returns MOE_ROUTE_ABI_VERSION of the loaded library. */
MOE_API int moe_abi_version(void);

/* A static, NUL-terminated English description of a moe_status value. */
MOE_API const char *moe_strerror(int status);

/*
 * moe_route_topk -- the router's top-K ([DSD] "MoE router": a sort that keeps
 * the indices of the selected scores; "Expert parallelism": each token goes to
 * K of the routed experts and their outputs are summed with weights).
 *
 *   logits   device, fp32 [T, E]     router scores.  NaN is not supported.
 *   T        number of tokens, >= 0 (T == 0 enqueues nothing).
 *   E        experts, 1..MOE_MAX_EXPERTS.
 *   K        experts per token, 1..min(E, MOE_MAX_TOPK).
 *   topk_idx device, int32 [T, K]    out: the K largest logits' expert ids, by
 *            descending logit; equal logits go to the smaller id (+0 and -0
 *            count as equal).
 *   topk_w   device, fp32 [T, K]     out: softmax over the K selected logits,
 *            w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0), in fp32 (CUDA expf,
 *            the K terms summed pairwise across the warp, one IEEE division).
 * Errors: MOE_ERR_INVALID_ARG for T < 0, E or K out of range, NULL pointers
 * with T > 0; MOE_ERR_CUDA if the launch fails.
 */
MOE_API moe_status moe_route_topk(const float *logits, int T, int E, int K,
                          int32_t *topk_idx, float *topk_w, moe_stream_t stream);

/*
 * moe_route_topk_grouped -- group-limited top-K ([DSD] "MoE router": DeepSeek's
 * routing takes a group top-K first; Mixtral's is the special case where the
 * group top-K is the group of all experts).  The page gives no formula; the
 * reading implemented is: the E experts form n_groups contiguous groups of
 * E/n_groups; a group's score is its largest logit; the topk_groups best
 * groups are kept (equal scores go to the smaller group id); then the K
 * largest logits among the kept groups' experts are chosen and weighted
 * exactly as by moe_route_topk.  With n_groups == 1, or topk_groups ==
 * n_groups, the result equals moe_route_topk's.  With groups aligned to ranks
 * (n_groups = R) every token reaches at most topk_groups ranks.
 *
 *   n_groups    1..MOE_MAX_GROUPS, dividing E.
 *   topk_groups 1..n_groups, with K <= topk_groups * (E / n_groups).
 *   other arguments, outputs and errors as moe_route_topk.
 */
MOE_API moe_status moe_route_topk_grouped(const float *logits, int T, int E, int K, int n_groups,
                                          int topk_groups, int32_t *topk_idx, float *topk_w,
                                          moe_stream_t stream);

/*
 * Bytes of device workspace moe_dispatch needs for these sizes (an upper bound
 * that depends only on R, E, K and T = sum B).  Returns 0 for sizes that
 * moe_dispatch would reject.
 */
MOE_API size_t moe_dispatch_workspace_bytes(int R, int E, int K, int64_t T);

/*
 * moe_dispatch -- count, exclusive scan and scatter ([EPK] "Optimising for
 * throughput" > "Dispatch": count the tokens per destination, exchange the
 * counts, let a prefix sum fix a conflict-free layout, copy each token to its
 * slot; [EFA] "Dispatch and combine": per-expert counts by shared-memory
 * atomics, a prefix sum for the offsets, rows packed into the input of the
 * grouped GEMM).  With every rank in one HBM the count exchange is a read of
 * the count matrix and the copy is one hop into the destination rank's rows.
 *
 *   x          device, bf16 [T, H], 16-byte aligned: the tokens of all ranks,
 *              rank-major.
 *   topk_idx   device, int32 [T, K]: the routing (e.g. from moe_route_topk).
 *   R          ranks, 1..MOE_MAX_RANKS; E % R == 0.
 *   B          HOST, int32 [R]: tokens per rank, each >= 0; T = sum B and
 *              T * K < 2^31.
 *   E, K       as for moe_route_topk (K <= MOE_MAX_TOPK).
 *   H          hidden size, 8..MOE_MAX_HIDDEN, a multiple of 8; a multiple of
 *              128 when recv_dtype is MOE_DTYPE_FP8_E4M3.
 *   recv_dtype MOE_DTYPE_BF16 (copy) or MOE_DTYPE_FP8_E4M3 (quantise once per
 *              token: per 128-channel block, amax = max |x| raised to at
 *              least 2^-119 (the smallest power of two with 448 / amax finite
 *              in fp32), scale = amax / 448 and inv = 448 / amax (IEEE fp32
 *              divisions, subnormal results kept),
 *              q = e4m3(x * inv) with round-to-nearest-even and saturation to
 *              +-448; [DSD] "Quantization").
 *   recv_x     device [T*K, H] of recv_dtype, 16-byte aligned: out.  Rows are
 *              grouped by expert (expert_offsets), within an expert by source
 *              rank (offsets), within a rank by ascending token; rank r's
 *              receive window is rows [expert_offsets[r*E/R],
 *              expert_offsets[(r+1)*E/R]).
 *   recv_scale device fp32 [T*K, H/128], 16-byte aligned: out, FP8 only
 *              (ignored and may be NULL for bf16).  Dequantised value =
 *              e4m3 value * recv_scale[row, h/128].
 *   counts     device int32 [E*R]: out, counts[e*R + s] = tokens of rank s
 *              routed to expert e.
 *   offsets    device int32 [E*R + 1]: out, exclusive prefix sum of counts in
 *              (e, s) order; offsets[E*R] = T*K.
 *   expert_offsets device int32 [E + 1]: out, offsets[e*R].
 *   tok2row    device int32 [T*K]: out, the row holding copy j of token g is
 *              tok2row[g*K + j] (combine's gather map).
 *   row2src    device int32 [T*K]: out, row2src[row] = g*K + j (the inverse).
 *   workspace  device, >= moe_dispatch_workspace_bytes(R, E, K, T) bytes,
 *              16-byte aligned; its first 4 bytes are the device error word.
 *              Calls that share a workspace must not overlap in time.
 * Errors: MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE as
 * above, MOE_ERR_CUDA on a launch failure.  T == 0 writes zeros to counts,
 * offsets and expert_offsets and launches no kernel.  Bad routing is reported
 * through the error word; the outputs are then unspecified, but no write
 * leaves the buffers above.
 */
MOE_API moe_status moe_dispatch(const void *x, const int32_t *topk_idx,
                        int R, const int32_t *B, int E, int K, int H,
                        moe_dtype recv_dtype, void *recv_x, float *recv_scale,
                        int32_t *counts, int32_t *offsets, int32_t *expert_offsets,
                        int32_t *tok2row, int32_t *row2src,
                        void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_dispatch_noalloc -- moe_dispatch without a caller-supplied workspace,
 * for callers that cannot allocate device memory: a plugin whose memory is
 * owned and budgeted by a host framework, or a serving loop that must not
 * allocate on its hot path (an allocation can block, or fail under memory
 * pressure).
 * The pages this library follows have no counterpart to it.
 *
 * Arguments and outputs are those of moe_dispatch, minus the workspace.  The
 * workspace is a device array of MOE_NOALLOC_SCRATCH_BYTES bytes that the
 * library holds on every GPU that loads it, for the life of the process.
 * Neither this call nor its set-up calls cudaMalloc, cudaFree or any other
 * allocating routine.
 *   - Set-up: the first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress, with the device current) and keeps it for the
 *     life of the process (a cudaDeviceReset invalidates it).  Make that first
 *     call on each device before any stream capture.
 *   - Size limit: a call for which moe_dispatch_workspace_bytes(R, E, K, T)
 *     exceeds MOE_NOALLOC_SCRATCH_BYTES returns MOE_ERR_WORKSPACE and enqueues
 *     nothing; it does so only once moe_dispatch's own argument checks have
 *     passed (a call those reject gets moe_dispatch's status).  The limit
 *     depends on R, E and K: with E = 256 experts it is
 *     T*K <= (511 - R) * 2048 routed copies (1 030 144 at R = 8, 784 384 at
 *     R = 128); with E = 384 and R = 32 it is T*K <= 632 832.
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     last call's contents; each call clears the parts that must start at
 *     zero.  Calls that overlap on the GPU (other streams, other threads)
 *     race on it and must be ordered by the caller.
 *   - Device-side routing errors are recorded in the array's error word, which
 *     the caller cannot read; check the routing with moe_dispatch and
 *     moe_get_device_error where that matters.
 * Other errors: as moe_dispatch.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)

MOE_API moe_status moe_dispatch_noalloc(const void *x, const int32_t *topk_idx,
                                        int R, const int32_t *B, int E, int K, int H,
                                        moe_dtype recv_dtype, void *recv_x, float *recv_scale,
                                        int32_t *counts, int32_t *offsets, int32_t *expert_offsets,
                                        int32_t *tok2row, int32_t *row2src, moe_stream_t stream);

/*
 * moe_expert_scale -- stand-in for the grouped expert GEMM (which is not part
 * of this library): y[row] = bf16(xhat * s_e) with s_e = 1 + e/256 for the
 * expert e whose rows [expert_offsets[e], expert_offsets[e+1]) hold `row`
 * (s_e = 1 when identity != 0); xhat is the bf16 value, or for an FP8 buffer
 * e4m3 value * recv_scale (one fp32 multiply).
 *
 *   recv_x, recv_scale, recv_dtype   as produced by moe_dispatch.
 *   expert_offsets device int32 [E + 1]; rows = expert_offsets[E] = T*K.
 *   y          device bf16 [rows, H], 16-byte aligned: out.
 * Errors: MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_CUDA.
 */
MOE_API moe_status moe_expert_scale(const void *recv_x, const float *recv_scale, moe_dtype recv_dtype,
                            const int32_t *expert_offsets, int E, int H, int rows,
                            int identity, void *y, moe_stream_t stream);

/*
 * moe_combine -- gather each token's K expert outputs and take their
 * routing-weighted sum ([EPK] "Optimising for throughput" > "Combine": undo
 * the dispatch permutation and add up each token's contributions with the
 * routing dispatch produced; [EFA] "Dispatch and combine": the receiver
 * accumulates the returned tokens into the output).
 *
 *   y          device bf16 [T*K, H], 16-byte aligned: expert outputs in the
 *              dispatch row order.
 *   tok2row    device int32 [T*K]: from moe_dispatch.  Entries outside
 *              [0, T*K) contribute nothing.  NULL means the identity map
 *              (row g*K + j), the layout moe_combine_ll_push leaves.
 *   topk_w     device fp32 [T, K]: routing weights.
 *   out_dtype  MOE_DTYPE_BF16 or MOE_DTYPE_FP32.
 *   out        device [T, H] of out_dtype, 16-byte aligned:
 *              out[g] = sum_{j=0..K-1} topk_w[g,j] * y[tok2row[g*K+j]],
 *              accumulated in fp32 by fused multiply-add in the fixed order
 *              j = 0, 1, ..., K-1 from +0, then rounded to bf16 (nearest even)
 *              or stored as fp32.
 * Errors: MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_CUDA.
 */
MOE_API moe_status moe_combine(const void *y, const int32_t *tok2row, const float *topk_w,
                       int T, int K, int H, moe_dtype out_dtype, void *out,
                       moe_stream_t stream);

/*
 * moe_dispatch_ll -- the low-latency dispatch ([EPK] "Optimising for latency:
 * send without asking"): instead of a packed buffer whose layout needs a
 * prefix sum over the real counts, every (source rank, expert) pair owns a
 * fixed region of C rows, sized for the worst case, so the destination of a
 * token is a static formula and the scan disappears from the path; C is the
 * cap on the tokens a rank dispatches per call.  Copy j of token g (rank s,
 * expert e) goes to row (e*R + s)*C + slot, slot = the number of rank s's
 * earlier tokens routed to e (the same order as moe_dispatch's).
 *
 *   x, topk_idx, R, B, E, K, H, recv_dtype, workspace: as moe_dispatch (the
 *              workspace size moe_dispatch_workspace_bytes(R, E, K, T) is
 *              enough); every B[s] <= C.
 *   C          rows per region, >= 1, with E*R*C < 2^31.
 *   recv_x     device [E*R*C, H] of recv_dtype: out.  Rows at or past
 *              counts[e*R + s] in a region are not written.
 *   recv_scale device fp32 [E*R*C, H/128]: out, FP8 only.
 *   counts     device int32 [E*R]: out, filled rows of region (e, s).
 *   tok2row    device int32 [T*K]: out, row of copy j of token g.
 *   row2src    device int32 [E*R*C]: out, g*K + j for each filled row; other
 *              rows are not written.
 * Errors: as moe_dispatch; MOE_ERR_INVALID_ARG also for C < 1, B[s] > C or
 * E*R*C >= 2^31.  T == 0 writes zeros to counts and launches no kernel.
 */
MOE_API moe_status moe_dispatch_ll(const void *x, const int32_t *topk_idx, int R, const int32_t *B,
                                   int E, int K, int H, int C, moe_dtype recv_dtype,
                                   void *recv_x, float *recv_scale, int32_t *counts,
                                   int32_t *tok2row, int32_t *row2src,
                                   void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_dispatch_ll_unordered -- the low-latency dispatch with sender-side
 * slots ([EPK] "Optimising for latency: send without asking": the sender
 * alone writes its (source rank, expert) region, so it can number its own
 * copies there without asking anyone).  A copy takes its slot by one atomic
 * increment of its region's count, so no histogram or scan runs before the
 * copies move; the call is two kernels (zero the counts, scatter).  Rows, counts
 * and maps are those of moe_dispatch_ll up to the order of the rows inside
 * each region, which is unspecified and may differ from call to call:
 *   - counts[e*R + s] is exact (the number of rank s's copies routed to e);
 *   - region (e, s) holds exactly those copies in rows (e*R + s)*C + [0, counts);
 *   - tok2row and row2src are inverse maps over the filled rows;
 *   - each filled row holds its token's bytes (and FP8 scales) exactly as
 *     moe_dispatch_ll writes them.
 * moe_combine_ll over these rows therefore gives bit-identical sums (it adds
 * in the fixed order j through tok2row).  The sources fix the region of a copy
 * but not its place inside the region; moe_dispatch_ll numbers the copies in
 * token order, which needs the per-rank histogram first, and this entry lets
 * the order fall out of the increments instead.
 *
 *   arguments  as moe_dispatch_ll, except that only the first 256 bytes of
 *              the workspace are used (workspace_bytes >= 256).
 * Errors: as moe_dispatch_ll.  T == 0 writes zeros to counts and launches no
 * kernel.
 */
MOE_API moe_status moe_dispatch_ll_unordered(const void *x, const int32_t *topk_idx, int R, const int32_t *B,
                                             int E, int K, int H, int C, moe_dtype recv_dtype,
                                             void *recv_x, float *recv_scale, int32_t *counts,
                                             int32_t *tok2row, int32_t *row2src,
                                             void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_combine_ll -- moe_combine over the low-latency rectangle: y is
 * [E*R*C, H] bf16 (expert outputs in moe_dispatch_ll's rows), tok2row is
 * moe_dispatch_ll's; indices outside [0, E*R*C) contribute nothing.  The sum,
 * its order and rounding, and the errors are those of moe_combine.
 */
MOE_API moe_status moe_combine_ll(const void *y, int E, int R, int C, const int32_t *tok2row,
                                  const float *topk_w, int T, int K, int H, moe_dtype out_dtype,
                                  void *out, moe_stream_t stream);

/*
 * moe_combine_ll_push -- the push-style return of the low-latency layout
 * ([EPK] "Optimising for latency": the expert's host writes each output
 * straight to a private slot on the token's origin rank, indexed by the
 * token's position there and by which of its K experts produced it).  For
 * every filled row of the rectangle (slot < counts[region]),
 * ret[row2src[row]] = y[row].  moe_combine with tok2row = NULL then forms
 * the weighted sums on the origin side.
 *
 *   y        device bf16 [E*R*C, H], 16-byte aligned.
 *   row2src, counts  from moe_dispatch_ll.
 *   ret      device bf16 [T*K, H], 16-byte aligned: out.
 * Errors: MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_CUDA.
 */
MOE_API moe_status moe_combine_ll_push(const void *y, const int32_t *row2src, const int32_t *counts,
                                       int R, int E, int C, int K, int H, int T, void *ret,
                                       moe_stream_t stream);

/*
 * moe_combine_partial_send / moe_combine_partial_recv -- combine with
 * sender-side partial accumulation ([EFA] "Evaluation": DeepEP accumulates on
 * the sending side to reduce the bytes returned, which may affect precision;
 * moe_combine accumulates on the receiving side).  Reading implemented (the
 * page gives no formula): rank r hosts experts e with e / (E/R) == r.
 *   send: for each token g and each rank r hosting some of g's experts,
 *         p[g,r] = bf16(fp32 fma over those copies in ascending j, from +0)
 *         is written to partial row g*K + j0, j0 = the first such copy; other
 *         rows of partial are not written.  Only one row per (token, rank)
 *         would travel back instead of one per copy.
 *   recv: out[g] = fp32 sum of g's partials in ascending rank order from +0,
 *         then bf16 (nearest even) or fp32.
 *
 *   y, tok2row, topk_w  as moe_combine;  topk_idx  device int32 [T, K], the
 *   routing dispatch used (every entry in [0, E));  E, R as moe_dispatch.
 *   partial  device bf16 [T*K, H], 16-byte aligned.
 *   out      device [T, H] of out_dtype (BF16 or FP32), 16-byte aligned.
 * Errors: MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_CUDA.
 */
MOE_API moe_status moe_combine_partial_send(const void *y, const int32_t *tok2row, const int32_t *topk_idx,
                                            const float *topk_w, int T, int K, int H, int E, int R,
                                            void *partial, moe_stream_t stream);
MOE_API moe_status moe_combine_partial_recv(const void *partial, const int32_t *topk_idx, int T, int K, int H,
                                            int E, int R, moe_dtype out_dtype, void *out,
                                            moe_stream_t stream);

/*
 * Split dispatch and combine: each is cut into a send half and a receive half
 * ([EFA] "MoE all-to-all over EFA": so that the GPU can run other work, such
 * as the shared expert, while transfers are pending; the receiver blocks until
 * every transfer to it has landed.  [DSD] "Computation and communication
 * overlap": the shared expert runs right after Dispatch Send, and Dispatch
 * Recv is awaited after it).  Results equal moe_dispatch's and moe_combine's
 * bit for bit.
 *
 * Ordering: enqueue each receive half after its send half -- on the same
 * stream, or on another stream behind an event recorded after the send half.
 * The receive half's wait then confirms, per destination rank, that every
 * transfer the send half announced has landed; it never waits on a kernel
 * that is still to run.  If an announcement never comes the wait gives up
 * after about 2 s, sets MOE_DEVERR_RECV_TIMEOUT in the workspace's error word
 * (moe_get_device_error then returns MOE_ERR_TIMEOUT) and the call completes.
 * The four calls of a layer share one workspace of at least
 * moe_dispatch_workspace_bytes(R, E, K, T) bytes, 16-byte aligned; calls that
 * share a workspace must not overlap in time apart from this pairing.
 *
 * moe_dispatch_send -- the copies ([EFA] "Dispatch and combine": per-expert
 * counts by shared-memory atomics, a prefix sum for the offsets, tokens packed
 * for their peers; within a node pushed straight into the peers' buffers).
 * Histogram, scan and scatter of moe_dispatch: recv_x, recv_scale, tok2row
 * and row2src are written exactly as moe_dispatch writes them; every copy is
 * announced to its destination rank once its bytes are stored.  counts,
 * offsets and expert_offsets are the receive half's.
 *   arguments  as moe_dispatch, without counts, offsets and expert_offsets;
 *   max_sms    0: the copy kernel may span every SM; n > 0: at most n SMs, so
 *              that work the caller runs on another stream meanwhile keeps
 *              the others.
 * Errors: as moe_dispatch; MOE_ERR_INVALID_ARG for max_sms < 0.  T == 0
 * launches nothing.
 *
 * moe_dispatch_recv -- the receiver's wait ([EFA] "Dispatch and combine":
 * block until all transfers have landed, then hand the rows to the grouped
 * GEMM): per destination rank r, waits until the copies announced for r equal
 * the rows its experts own, consumes the announcements (a second receive
 * without a new send waits again), and writes counts, offsets and
 * expert_offsets as moe_dispatch defines them.  R, B, E, K and workspace are
 * the send half's.  Errors: MOE_ERR_INVALID_ARG / MOE_ERR_WORKSPACE /
 * MOE_ERR_UNSUPPORTED / MOE_ERR_CUDA.  T == 0 writes zeros and launches no
 * kernel.
 *
 * moe_combine_send -- the expert ranks publish their outputs: one release
 * flag per expert rank, set after the work enqueued before this call on
 * `stream` (the expert GEMM that wrote y).  Every rank's buffer is in the one
 * HBM, so the receive half pulls the rows itself ([EFA] "Send and receive
 * buffers": within a node the buffers are mapped into the peers, which push
 * or pull tokens directly) and nothing is copied here.
 *   workspace  at least 256 + 8*R bytes rounded up to a multiple of 256 (the
 *              layer's dispatch workspace is larger).
 * Errors: MOE_ERR_INVALID_ARG for R out of range, MOE_ERR_WORKSPACE,
 * MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA.
 *
 * moe_combine_recv -- waits until every expert rank's flag is set, consumes
 * the flags, then forms out[g] exactly as moe_combine does ([EFA] "Dispatch
 * and combine": the receiver accumulates the returned tokens into the output).
 * Arguments as moe_combine, plus R and the workspace of moe_combine_send.
 * Errors: as moe_combine; MOE_ERR_WORKSPACE.  T == 0 launches nothing.
 */
MOE_API moe_status moe_dispatch_send(const void *x, const int32_t *topk_idx, int R, const int32_t *B, int E, int K,
                                     int H, moe_dtype recv_dtype, void *recv_x, float *recv_scale, int32_t *tok2row,
                                     int32_t *row2src, int max_sms, void *workspace, size_t workspace_bytes,
                                     moe_stream_t stream);
MOE_API moe_status moe_dispatch_recv(int R, const int32_t *B, int E, int K, int32_t *counts, int32_t *offsets,
                                     int32_t *expert_offsets, void *workspace, size_t workspace_bytes,
                                     moe_stream_t stream);
MOE_API moe_status moe_combine_send(int R, void *workspace, size_t workspace_bytes, moe_stream_t stream);
MOE_API moe_status moe_combine_recv(const void *y, const int32_t *tok2row, const float *topk_w, int T, int K, int H,
                                    moe_dtype out_dtype, void *out, int R, void *workspace, size_t workspace_bytes,
                                    moe_stream_t stream);

/*
 * moe_get_device_error -- SYNCHRONOUS: waits for `stream`, then copies the
 * dispatch workspace's error word (an OR of MOE_DEVERR_* bits, 0 if none) to
 * *host_code.  Returns MOE_ERR_TIMEOUT if a timeout bit is set, else
 * MOE_ERR_BAD_ROUTING if a routing bit is set, else MOE_OK (MOE_ERR_CUDA if
 * the copy fails, MOE_ERR_INVALID_ARG for NULL pointers).  The word is reset
 * by the next moe_dispatch on that workspace.
 */
MOE_API moe_status moe_get_device_error(const void *workspace, int32_t *host_code, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H */
