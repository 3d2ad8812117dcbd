// expert.cu -- stand-in for the grouped expert GEMM between dispatch and
// combine: y[row] = bf16(xhat * s_e) with s_e = 1 + e/256 for the expert e
// that owns the row (s_e = 1 in identity mode); xhat is the received bf16
// value, or the e4m3 value times its per-128-channel scale.
//
// The grouped GEMM itself is not part of this library (the sources run it
// with DeepGEMM; Perplexity, "Lower latency and higher throughput with
// multi-node DeepSeek deployment", section "GroupGEMM").  This kernel only
// gives combine deterministic, expert-dependent inputs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "launch.h"

namespace moe {

// One thread per 8 channels of a row; the row's expert comes from a binary
// search over expert_offsets held in shared memory.
template <bool kFp8>
__global__ void __launch_bounds__(256) expert_scale_kernel(const void *__restrict__ recv,
                                                           const float *__restrict__ recv_scale,
                                                           const int32_t *__restrict__ expert_offsets, int E, int H,
                                                           int rows, int identity, __nv_bfloat16 *__restrict__ y) {
    extern __shared__ int32_t s_eo[];   // [E + 1]
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_eo[i] = expert_offsets[i];
    __syncthreads();
    const int nchunk = H / 8;
    const long long total = (long long)rows * nchunk;
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < total;
         v += (long long)gridDim.x * blockDim.x) {
        const int row = (int)(v / nchunk);
        const int c = (int)(v - (long long)row * nchunk);
        // expert of the row: s_eo[e] <= row < s_eo[e+1]
        int lo = 0, hi = E;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_eo[mid] <= row) lo = mid; else hi = mid;
        }
        const float se = identity ? 1.0f : 1.0f + (float)lo / 256.0f;
        float f[8];
        if (kFp8) {
            const uint2 q = *reinterpret_cast<const uint2 *>(static_cast<const unsigned char *>(recv) +
                                                             (size_t)row * H + (size_t)c * 8);
            const float sc = recv_scale[(size_t)row * (H / 128) + (c * 8) / 128];
            const uint32_t w[2] = {q.x, q.y};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[k >> 1] >> (16 * (k & 1))) & 0xffffu);
                const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
                const float2 fl = __half22float2(__half2(hr));
                f[2 * k] = __fmul_rn(fl.x, sc);
                f[2 * k + 1] = __fmul_rn(fl.y, sc);
            }
        } else {
            const uint4 u = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(recv) +
                                                             (size_t)row * H + (size_t)c * 8);
            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 t = __bfloat1622float2(h2[k]);
                f[2 * k] = t.x;
                f[2 * k + 1] = t.y;
            }
        }
        uint4 pk;
        __nv_bfloat162 *p2 = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
        for (int k = 0; k < 4; ++k) p2[k] = __floats2bfloat162_rn(__fmul_rn(f[2 * k], se), __fmul_rn(f[2 * k + 1], se));
        *reinterpret_cast<uint4 *>(y + (size_t)row * H + (size_t)c * 8) = pk;
    }
}

cudaError_t launch_expert_scale(const void *recv, const float *recv_scale, bool fp8, const int32_t *expert_offsets,
                                int E, int H, int rows, int identity, void *y, cudaStream_t stream) {
    const long long total = (long long)rows * (H / 8);
    long long grid = (total + 255) / 256;
    const long long cap = (long long)device_sm_count() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    const size_t smem = (size_t)(E + 1) * 4;
    __nv_bfloat16 *yb = static_cast<__nv_bfloat16 *>(y);
    if (fp8)
        expert_scale_kernel<true><<<(unsigned)grid, 256, smem, stream>>>(recv, recv_scale, expert_offsets, E, H, rows,
                                                                         identity, yb);
    else
        expert_scale_kernel<false><<<(unsigned)grid, 256, smem, stream>>>(recv, recv_scale, expert_offsets, E, H,
                                                                          rows, identity, yb);
    return cudaGetLastError();
}

}  // namespace moe
