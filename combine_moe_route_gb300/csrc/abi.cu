// abi.cu -- the extern "C" entry points of libmoeroute (declared and
// documented in include/moe_route.h): host-side argument validation, the
// per-call rank table, and the kernel launches.  Nothing here allocates,
// frees or synchronises, except moe_get_device_error, which is documented as
// synchronous.  Validation runs before the first CUDA call, so a rejected call
// touches no device state.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "launch.h"
#include "moe_route.h"


namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool topk_shape_ok(int E, int K) { return E >= 1 && E <= MOE_MAX_EXPERTS && K >= 1 && K <= E && K <= MOE_MAX_TOPK; }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Fill the rank table from host B; false if any B is negative or T*K overflows int32.
bool build_rank_table(int R, const int32_t *B, int K, moe::RankTable &rt, long long &T) {
    memset(&rt, 0, sizeof(rt));
    rt.R = R;
    long long acc = 0, tiles = 0;
    rt.rank_off[0] = 0;
    rt.tile_off[0] = 0;
    for (int s = 0; s < R; ++s) {
        if (B[s] < 0) return false;
        acc += B[s];
        if (acc * K >= (1ll << 31)) return false;
        tiles += ((long long)B[s] * K + moe::kTileItems - 1) / moe::kTileItems;
        rt.rank_off[s + 1] = (int32_t)acc;
        rt.tile_off[s + 1] = (int32_t)tiles;
    }
    rt.ntiles = (int)tiles;
    T = acc;
    return true;
}

}  // namespace

namespace moe {

// The checks moe_dispatch makes before it looks at the workspace, in its
// order.  On MOE_OK, rt, T and fp8 are filled; when T == 0 nothing is to be
// scattered, and x, topk_idx and the payload and map pointers are not checked.
// with_layout: the call writes counts / offsets / expert_offsets (moe_dispatch),
// or leaves them to a receive half (moe_dispatch_send).
moe_status check_dispatch_args(const void *x, const int32_t *topk_idx, int R, const int32_t *B, int E, int K, int H,
                               moe_dtype recv_dtype, const void *recv_x, const float *recv_scale, bool with_layout,
                               const int32_t *counts, const int32_t *offsets, const int32_t *expert_offsets,
                               const int32_t *tok2row, const int32_t *row2src, RankTable &rt, long long &T,
                               bool &fp8) {
    if (R < 1 || R > MOE_MAX_RANKS || !B || !topk_shape_ok(E, K) || E % R != 0) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > MOE_MAX_HIDDEN || H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (recv_dtype != MOE_DTYPE_BF16 && recv_dtype != MOE_DTYPE_FP8_E4M3) return MOE_ERR_INVALID_ARG;
    fp8 = recv_dtype == MOE_DTYPE_FP8_E4M3;
    if (fp8 && H % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (!build_rank_table(R, B, K, rt, T)) return MOE_ERR_INVALID_ARG;
    if (with_layout && (!counts || !offsets || !expert_offsets)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !topk_idx || !recv_x || !tok2row || !row2src || (fp8 && !recv_scale)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(recv_x) || (fp8 && !aligned16(recv_scale))) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace moe

extern "C" {

int moe_abi_version(void) { return MOE_ROUTE_ABI_VERSION; }

const char *moe_strerror(int status) {
    switch (status) {
        case MOE_OK: return "success";
        case MOE_ERR_INVALID_ARG: return "invalid argument (NULL pointer, size out of range or inconsistent shape)";
        case MOE_ERR_UNSUPPORTED: return "unsupported argument (pointer not 16-byte aligned)";
        case MOE_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
        case MOE_ERR_WORKSPACE: return "workspace missing or smaller than moe_dispatch_workspace_bytes()";
        case MOE_ERR_TIMEOUT: return "a bounded device wait ran out";
        case MOE_ERR_BAD_ROUTING: return "routing has an expert id out of range or repeated within a token";
        default: return "unknown moe_status";
    }
}

moe_status moe_route_topk(const float *logits, int T, int E, int K, int32_t *topk_idx, float *topk_w,
                          moe_stream_t stream) {
    if (T < 0 || !topk_shape_ok(E, K)) return MOE_ERR_INVALID_ARG;
    if ((long long)T * E >= (1ll << 40)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_route_topk(logits, T, E, K, 1, 1, topk_idx, topk_w, (cudaStream_t)stream));
}

moe_status moe_route_topk_grouped(const float *logits, int T, int E, int K, int n_groups, int topk_groups,
                                  int32_t *topk_idx, float *topk_w, moe_stream_t stream) {
    if (T < 0 || !topk_shape_ok(E, K)) return MOE_ERR_INVALID_ARG;
    if (n_groups < 1 || n_groups > MOE_MAX_GROUPS || E % n_groups != 0) return MOE_ERR_INVALID_ARG;
    if (topk_groups < 1 || topk_groups > n_groups || K > topk_groups * (E / n_groups)) return MOE_ERR_INVALID_ARG;
    if ((long long)T * E >= (1ll << 40)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_route_topk(logits, T, E, K, n_groups, topk_groups, topk_idx, topk_w,
                                              (cudaStream_t)stream));
}

size_t moe_dispatch_workspace_bytes(int R, int E, int K, int64_t T) {
    if (R < 1 || R > MOE_MAX_RANKS || !topk_shape_ok(E, K) || E % R != 0) return 0;
    if (T < 0 || T * K >= (1ll << 31)) return 0;
    const int ntiles = moe::max_tiles(R, K, T);
    return moe::plan_dispatch(E, R, ntiles).total;
}

moe_status moe_dispatch(const void *x, const int32_t *topk_idx, int R, const int32_t *B, int E, int K, int H,
                        moe_dtype recv_dtype, void *recv_x, float *recv_scale, int32_t *counts, int32_t *offsets,
                        int32_t *expert_offsets, int32_t *tok2row, int32_t *row2src, void *workspace,
                        size_t workspace_bytes, moe_stream_t stream) {
    moe::RankTable rt;
    long long T = 0;
    bool fp8 = false;
    const moe_status v = moe::check_dispatch_args(x, topk_idx, R, B, E, K, H, recv_dtype, recv_x, recv_scale, true,
                                                  counts, offsets, expert_offsets, tok2row, row2src, rt, T, fp8);
    if (v != MOE_OK) return v;
    cudaStream_t st = (cudaStream_t)stream;
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)E * R, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * ((size_t)E * R + 1), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * ((size_t)E + 1), st);
        return cuda_status(e);
    }
    if (!workspace) return MOE_ERR_WORKSPACE;
    if (workspace_bytes < moe::call_plan(rt, E, K).total) return MOE_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_dispatch(x, topk_idx, rt, E, K, H, fp8, recv_x, fp8 ? recv_scale : nullptr, counts,
                                            offsets, expert_offsets, tok2row, row2src, workspace, st));
}

moe_status moe_dispatch_send(const void *x, const int32_t *topk_idx, int R, const int32_t *B, int E, int K, int H,
                             moe_dtype recv_dtype, void *recv_x, float *recv_scale, int32_t *tok2row,
                             int32_t *row2src, int max_sms, void *workspace, size_t workspace_bytes,
                             moe_stream_t stream) {
    moe::RankTable rt;
    long long T = 0;
    bool fp8 = false;
    const moe_status v = moe::check_dispatch_args(x, topk_idx, R, B, E, K, H, recv_dtype, recv_x, recv_scale, false,
                                                  nullptr, nullptr, nullptr, tok2row, row2src, rt, T, fp8);
    if (v != MOE_OK) return v;
    if (max_sms < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;   // nothing to send; the receive half writes the empty layout
    if (!workspace) return MOE_ERR_WORKSPACE;
    if (workspace_bytes < moe::call_plan(rt, E, K).total) return MOE_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_dispatch_send(x, topk_idx, rt, E, K, H, fp8, recv_x, fp8 ? recv_scale : nullptr,
                                                 tok2row, row2src, workspace, max_sms, (cudaStream_t)stream));
}

moe_status moe_dispatch_recv(int R, const int32_t *B, int E, int K, int32_t *counts, int32_t *offsets,
                             int32_t *expert_offsets, void *workspace, size_t workspace_bytes, moe_stream_t stream) {
    if (R < 1 || R > MOE_MAX_RANKS || !B || !topk_shape_ok(E, K) || E % R != 0) return MOE_ERR_INVALID_ARG;
    moe::RankTable rt;
    long long T = 0;
    if (!build_rank_table(R, B, K, rt, T)) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || !expert_offsets) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)E * R, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * ((size_t)E * R + 1), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * ((size_t)E + 1), st);
        return cuda_status(e);
    }
    if (!workspace) return MOE_ERR_WORKSPACE;
    if (workspace_bytes < moe::call_plan(rt, E, K).total) return MOE_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_dispatch_recv(rt, E, K, counts, offsets, expert_offsets, workspace, st));
}

moe_status moe_combine_send(int R, void *workspace, size_t workspace_bytes, moe_stream_t stream) {
    if (R < 1 || R > MOE_MAX_RANKS) return MOE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < moe::signal_workspace_bytes(R)) return MOE_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_combine_send(R, workspace, (cudaStream_t)stream));
}

moe_status moe_combine_recv(const void *y, const int32_t *tok2row, const float *topk_w, int T, int K, int H,
                            moe_dtype out_dtype, void *out, int R, void *workspace, size_t workspace_bytes,
                            moe_stream_t stream) {
    if (T < 0 || K < 1 || K > MOE_MAX_TOPK || R < 1 || R > MOE_MAX_RANKS) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > MOE_MAX_HIDDEN || H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if ((long long)T * K >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
    if (out_dtype != MOE_DTYPE_BF16 && out_dtype != MOE_DTYPE_FP32) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y || !tok2row || !topk_w || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(out)) return MOE_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < moe::signal_workspace_bytes(R)) return MOE_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_combine_recv(y, tok2row, topk_w, T, K, H, out_dtype == MOE_DTYPE_FP32, out, R,
                                                workspace, (cudaStream_t)stream));
}

moe_status moe_expert_scale(const void *recv_x, const float *recv_scale, moe_dtype recv_dtype,
                            const int32_t *expert_offsets, int E, int H, int rows, int identity, void *y,
                            moe_stream_t stream) {
    if (E < 1 || E > MOE_MAX_EXPERTS || rows < 0) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > MOE_MAX_HIDDEN || H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (recv_dtype != MOE_DTYPE_BF16 && recv_dtype != MOE_DTYPE_FP8_E4M3) return MOE_ERR_INVALID_ARG;
    const bool fp8 = recv_dtype == MOE_DTYPE_FP8_E4M3;
    if (fp8 && H % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!recv_x || !expert_offsets || !y || (fp8 && !recv_scale)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(recv_x) || !aligned16(y)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_expert_scale(recv_x, recv_scale, fp8, expert_offsets, E, H, rows, identity, y,
                                                (cudaStream_t)stream));
}

moe_status moe_combine(const void *y, const int32_t *tok2row, const float *topk_w, int T, int K, int H,
                       moe_dtype out_dtype, void *out, moe_stream_t stream) {
    if (T < 0 || K < 1 || K > MOE_MAX_TOPK) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > MOE_MAX_HIDDEN || H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if ((long long)T * K >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
    if (out_dtype != MOE_DTYPE_BF16 && out_dtype != MOE_DTYPE_FP32) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y || !topk_w || !out) return MOE_ERR_INVALID_ARG;   // tok2row NULL: the identity map
    if (!aligned16(y) || !aligned16(out)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_combine(y, tok2row, topk_w, T, K, H, out_dtype == MOE_DTYPE_FP32, out,
                                           (long long)T * K, (cudaStream_t)stream));
}

// Checks shared by the two low-latency dispatch entries.  On MOE_OK with
// launch = true the call may go ahead with rt and fp8 filled; otherwise the
// returned status is the call's result (T == 0 has zeroed counts and returns
// MOE_OK with launch = false).  The ordered form needs the full dispatch
// workspace (histogram tiles), the unordered one only the header.
static moe_status check_dispatch_ll(bool ordered, const void *x, const int32_t *topk_idx, int R, const int32_t *B,
                                    int E, int K, int H, int C, moe_dtype recv_dtype, void *recv_x,
                                    float *recv_scale, int32_t *counts, int32_t *tok2row, int32_t *row2src,
                                    void *workspace, size_t workspace_bytes, cudaStream_t st, moe::RankTable &rt,
                                    bool &fp8, bool &launch) {
    launch = false;
    if (R < 1 || R > MOE_MAX_RANKS || !B || !topk_shape_ok(E, K) || E % R != 0) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > MOE_MAX_HIDDEN || H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (recv_dtype != MOE_DTYPE_BF16 && recv_dtype != MOE_DTYPE_FP8_E4M3) return MOE_ERR_INVALID_ARG;
    fp8 = recv_dtype == MOE_DTYPE_FP8_E4M3;
    if (fp8 && H % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (C < 1 || (long long)E * R * C >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
    long long T = 0;
    if (!build_rank_table(R, B, K, rt, T)) return MOE_ERR_INVALID_ARG;
    for (int s = 0; s < R; ++s)
        if (B[s] > C) return MOE_ERR_INVALID_ARG;   // the chunk cap bounds every region
    if (!counts) return MOE_ERR_INVALID_ARG;
    if (T == 0) return cuda_status(cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)E * R, st));
    if (!x || !topk_idx || !recv_x || !tok2row || !row2src || (fp8 && !recv_scale)) return MOE_ERR_INVALID_ARG;
    if (!workspace) return MOE_ERR_WORKSPACE;
    const size_t need = ordered ? moe::plan_dispatch(E, R, rt.ntiles).total : moe::kWsHeader;
    if (workspace_bytes < need) return MOE_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(recv_x) || !aligned16(workspace) || (fp8 && !aligned16(recv_scale)))
        return MOE_ERR_UNSUPPORTED;
    launch = true;
    return MOE_OK;
}

moe_status moe_dispatch_ll(const void *x, const int32_t *topk_idx, int R, const int32_t *B, int E, int K, int H, int C,
                           moe_dtype recv_dtype, void *recv_x, float *recv_scale, int32_t *counts, int32_t *tok2row,
                           int32_t *row2src, void *workspace, size_t workspace_bytes, moe_stream_t stream) {
    const cudaStream_t st = (cudaStream_t)stream;
    moe::RankTable rt;
    bool fp8 = false, launch = false;
    const moe_status v = check_dispatch_ll(true, x, topk_idx, R, B, E, K, H, C, recv_dtype, recv_x, recv_scale, counts,
                                           tok2row, row2src, workspace, workspace_bytes, st, rt, fp8, launch);
    if (v != MOE_OK || !launch) return v;
    return cuda_status(moe::launch_dispatch_ll(x, topk_idx, rt, E, K, H, C, fp8, recv_x, fp8 ? recv_scale : nullptr,
                                               counts, tok2row, row2src, workspace, st));
}

moe_status moe_dispatch_ll_unordered(const void *x, const int32_t *topk_idx, int R, const int32_t *B, int E, int K,
                                     int H, int C, moe_dtype recv_dtype, void *recv_x, float *recv_scale,
                                     int32_t *counts, int32_t *tok2row, int32_t *row2src, void *workspace,
                                     size_t workspace_bytes, moe_stream_t stream) {
    const cudaStream_t st = (cudaStream_t)stream;
    moe::RankTable rt;
    bool fp8 = false, launch = false;
    const moe_status v = check_dispatch_ll(false, x, topk_idx, R, B, E, K, H, C, recv_dtype, recv_x, recv_scale,
                                           counts, tok2row, row2src, workspace, workspace_bytes, st, rt, fp8, launch);
    if (v != MOE_OK || !launch) return v;
    return cuda_status(moe::launch_dispatch_ll_unordered(x, topk_idx, rt, E, K, H, C, fp8, recv_x,
                                                         fp8 ? recv_scale : nullptr, counts, tok2row, row2src,
                                                         workspace, st));
}

moe_status moe_combine_ll(const void *y, int E, int R, int C, const int32_t *tok2row, const float *topk_w, int T,
                          int K, int H, moe_dtype out_dtype, void *out, moe_stream_t stream) {
    if (T < 0 || K < 1 || K > MOE_MAX_TOPK || E < 1 || R < 1 || C < 1) return MOE_ERR_INVALID_ARG;
    if ((long long)E * R * C >= (1ll << 31) || (long long)T * K >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > MOE_MAX_HIDDEN || H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (out_dtype != MOE_DTYPE_BF16 && out_dtype != MOE_DTYPE_FP32) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y || !tok2row || !topk_w || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(out)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_combine(y, tok2row, topk_w, T, K, H, out_dtype == MOE_DTYPE_FP32, out,
                                           (long long)E * R * C, (cudaStream_t)stream));
}

moe_status moe_combine_ll_push(const void *y, const int32_t *row2src, const int32_t *counts, int R, int E, int C,
                               int K, int H, int T, void *ret, moe_stream_t stream) {
    if (T < 0 || K < 1 || K > MOE_MAX_TOPK || E < 1 || R < 1 || C < 1) return MOE_ERR_INVALID_ARG;
    if ((long long)E * R * C >= (1ll << 31) || (long long)T * K >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > MOE_MAX_HIDDEN || H % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y || !row2src || !counts || !ret) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(ret)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_combine_push(y, row2src, counts, C, H, (long long)E * R * C, (long long)T * K, ret,
                                                (cudaStream_t)stream));
}

moe_status moe_combine_partial_send(const void *y, const int32_t *tok2row, const int32_t *topk_idx,
                                    const float *topk_w, int T, int K, int H, int E, int R, void *partial,
                                    moe_stream_t stream) {
    if (T < 0 || R < 1 || R > MOE_MAX_RANKS || !topk_shape_ok(E, K) || E % R != 0) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > MOE_MAX_HIDDEN || H % 8 != 0 || (long long)T * K >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y || !tok2row || !topk_idx || !topk_w || !partial) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(partial)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(
        moe::launch_combine_partial(y, tok2row, topk_idx, topk_w, T, K, H, E, R, partial, (cudaStream_t)stream));
}

moe_status moe_combine_partial_recv(const void *partial, const int32_t *topk_idx, int T, int K, int H, int E, int R,
                                    moe_dtype out_dtype, void *out, moe_stream_t stream) {
    if (T < 0 || R < 1 || R > MOE_MAX_RANKS || !topk_shape_ok(E, K) || E % R != 0) return MOE_ERR_INVALID_ARG;
    if (H < 8 || H > MOE_MAX_HIDDEN || H % 8 != 0 || (long long)T * K >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
    if (out_dtype != MOE_DTYPE_BF16 && out_dtype != MOE_DTYPE_FP32) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!partial || !topk_idx || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(partial) || !aligned16(out)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_combine_partial_recv(partial, topk_idx, T, K, H, E, R, out_dtype == MOE_DTYPE_FP32,
                                                        out, (cudaStream_t)stream));
}

moe_status moe_get_device_error(const void *workspace, int32_t *host_code, moe_stream_t stream) {
    if (!workspace || !host_code) return MOE_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    *host_code = v;
    if (v & (MOE_DEVERR_SCAN_TIMEOUT | MOE_DEVERR_COPY_TIMEOUT | MOE_DEVERR_RECV_TIMEOUT)) return MOE_ERR_TIMEOUT;
    if (v & (MOE_DEVERR_EXPERT_RANGE | MOE_DEVERR_DUPLICATE)) return MOE_ERR_BAD_ROUTING;
    return MOE_OK;
}

}  // extern "C"
