// launch.h -- internal declarations shared by the libmoeroute translation
// units (host-side launchers and the dispatch workspace plan).  Not part of
// the public ABI, which is include/moe_route.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// Byte offsets inside the dispatch workspace: the header (error word, scan
// ticket, scatter token counter), the split halves' signals (per destination
// rank: copies landed, then expert outputs ready), the lookback status words,
// the tile histogram and its scan.
struct DispatchPlan {
    int ntiles;
    int nscan_blocks;
    size_t off_signal, off_status, off_hist, off_scan, total;
};

DispatchPlan plan_dispatch(int E, int R, int ntiles);
// Whether a dispatch of T tokens with top-K takes the one-kernel path, and the
// workspace layout the call uses.
bool small_dispatch(long long T, int K);
DispatchPlan call_plan(const RankTable &rt, int E, int K);
moe_status check_dispatch_args(const void *x, const int32_t *topk_idx, int R, const int32_t *B, int E, int K, int H,
                               moe_dtype recv_dtype, const void *recv_x, const float *recv_scale, bool with_layout,
                               const int32_t *counts, const int32_t *offsets, const int32_t *expert_offsets,
                               const int32_t *tok2row, const int32_t *row2src, RankTable &rt, long long &T,
                               bool &fp8);
// Bytes of workspace the combine halves need (header and signals only).
size_t signal_workspace_bytes(int R);
int max_tiles(int R, int K, long long T);
int device_sm_count();

cudaError_t launch_route_topk(const float *logits, int T, int E, int K, int G, int M, int32_t *topk_idx,
                              float *topk_w, cudaStream_t stream);
cudaError_t launch_dispatch(const void *x, const int32_t *topk_idx, const RankTable &rt, int E, int K, int H,
                            bool fp8, void *recv_x, float *recv_scale, int32_t *counts, int32_t *offsets,
                            int32_t *expert_offsets, int32_t *tok2row, int32_t *row2src, void *workspace,
                            cudaStream_t stream);
cudaError_t launch_dispatch_send(const void *x, const int32_t *topk_idx, const RankTable &rt, int E, int K, int H,
                                 bool fp8, void *recv_x, float *recv_scale, int32_t *tok2row, int32_t *row2src,
                                 void *workspace, int max_sms, cudaStream_t stream);
cudaError_t launch_dispatch_recv(const RankTable &rt, int E, int K, int32_t *counts, int32_t *offsets,
                                 int32_t *expert_offsets, void *workspace, cudaStream_t stream);
cudaError_t launch_combine_send(int R, void *workspace, cudaStream_t stream);
cudaError_t launch_combine_recv(const void *y, const int32_t *tok2row, const float *topk_w, int T, int K, int H,
                                bool out_f32, void *out, int R, void *workspace, cudaStream_t stream);
cudaError_t launch_dispatch_ll(const void *x, const int32_t *topk_idx, const RankTable &rt, int E, int K, int H,
                               int C, bool fp8, void *recv_x, float *recv_scale, int32_t *counts, int32_t *tok2row,
                               int32_t *row2src, void *workspace, cudaStream_t stream);
cudaError_t launch_dispatch_ll_unordered(const void *x, const int32_t *topk_idx, const RankTable &rt, int E, int K,
                                         int H, int C, bool fp8, void *recv_x, float *recv_scale, int32_t *counts,
                                         int32_t *tok2row, int32_t *row2src, void *workspace, cudaStream_t stream);
cudaError_t launch_combine(const void *y, const int32_t *tok2row, const float *topk_w, int T, int K, int H,
                           bool out_f32, void *out, long long rows, cudaStream_t stream);
cudaError_t launch_combine_push(const void *y, const int32_t *row2src, const int32_t *counts, int C, int H,
                                long long rect_rows, long long ret_rows, void *ret, cudaStream_t stream);
cudaError_t launch_combine_partial(const void *y, const int32_t *tok2row, const int32_t *topk_idx,
                                   const float *topk_w, int T, int K, int H, int E, int R, void *partial,
                                   cudaStream_t stream);
cudaError_t launch_combine_partial_recv(const void *partial, const int32_t *topk_idx, int T, int K, int H, int E,
                                        int R, bool out_f32, void *out, cudaStream_t stream);
cudaError_t launch_expert_scale(const void *recv, const float *recv_scale, bool fp8, const int32_t *expert_offsets,
                                int E, int H, int rows, int identity, void *y, cudaStream_t stream);

}  // namespace moe
