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

constexpr int kExpertThreads = 256;
#ifndef MOE_EXPERT_UNROLL
#define MOE_EXPERT_UNROLL 2   // 16-byte chunks per lane in flight at once
#endif
constexpr int kU = MOE_EXPERT_UNROLL;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even
    return (uint32_t)__bfloat16_as_ushort(h.x) | ((uint32_t)__bfloat16_as_ushort(h.y) << 16);
}

// 8 fp32 values times s_e, rounded to bf16 and packed (first value in the low half).
__device__ __forceinline__ uint4 scale_to_bf16x8(const float *f, float se) {
    return make_uint4(pack_bf16x2(__fmul_rn(f[0], se), __fmul_rn(f[1], se)),
                      pack_bf16x2(__fmul_rn(f[2], se), __fmul_rn(f[3], se)),
                      pack_bf16x2(__fmul_rn(f[4], se), __fmul_rn(f[5], se)),
                      pack_bf16x2(__fmul_rn(f[6], se), __fmul_rn(f[7], se)));
}

// One warp per row (the kernel also walks rows warp-strided, should a caller
// launch fewer blocks).  Lane 0 finds
// the row's expert by binary search over expert_offsets in shared memory.
// FP8: a lane takes 16 e4m3 values (16 bytes) per chunk, decodes them exactly
// through half precision, multiplies by the block scale and by s_e, and
// writes 32 bytes of bf16.  bf16: 8 values (16 bytes) in, 16 bytes out.  Each
// lane issues the loads of kU chunks before converting any of them.
template <bool kFp8>
__global__ void __launch_bounds__(kExpertThreads) expert_scale_kernel(const void *__restrict__ recv,
                                                                      const float *__restrict__ recv_scale,
                                                                      const int32_t *__restrict__ expert_offsets,
                                                                      int E, int H, int rows, int identity,
                                                                      __nv_bfloat16 *__restrict__ y) {
    extern __shared__ int32_t s_eo[];   // [E + 1]
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_eo[i] = expert_offsets[i];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const long long W = (long long)gridDim.x * (blockDim.x >> 5);
    const int nblk = H / 128;
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += W) {
        int e = 0;
        if (lane == 0) {   // s_eo[e] <= row < s_eo[e+1]
            int lo = 0, hi = E;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_eo[mid] <= row) lo = mid; else hi = mid;
            }
            e = lo;
        }
        e = __shfl_sync(0xffffffffu, e, 0);
        const float se = identity ? 1.0f : 1.0f + (float)e / 256.0f;
        __nv_bfloat16 *yr = y + (size_t)row * H;
        if (kFp8) {
            const unsigned char *qr = static_cast<const unsigned char *>(recv) + (size_t)row * H;
            const float *sr = recv_scale + (size_t)row * nblk;
            const int nc = H / 16;
            for (int c0 = lane; c0 < nc; c0 += 32 * kU) {
                uint4 q[kU];
                float sc[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + 32 * u;
                    q[u] = (c < nc) ? ld_stream_v4(qr + (size_t)c * 16) : make_uint4(0u, 0u, 0u, 0u);
                    sc[u] = (c < nc) ? __ldg(sr + (c >> 3)) : 0.0f;   // 8 chunks of 16 per 128-channel block
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + 32 * u;
                    if (c >= nc) break;
                    const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
                    float f[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const __nv_fp8x2_storage_t pair =
                            (__nv_fp8x2_storage_t)((w[k >> 1] >> (16 * (k & 1))) & 0xffffu);
                        const float2 fl = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
                        f[2 * k] = __fmul_rn(fl.x, sc[u]);
                        f[2 * k + 1] = __fmul_rn(fl.y, sc[u]);
                    }
                    st_v4(yr + (size_t)c * 16, scale_to_bf16x8(f, se));
                    st_v4(yr + (size_t)c * 16 + 8, scale_to_bf16x8(f + 8, se));
                }
            }
        } else {
            const __nv_bfloat16 *xr = static_cast<const __nv_bfloat16 *>(recv) + (size_t)row * H;
            const int nc = H / 8;
            for (int c0 = lane; c0 < nc; c0 += 32 * kU) {
                uint4 v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + 32 * u;
                    v[u] = (c < nc) ? ld_stream_v4(xr + (size_t)c * 8) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + 32 * u;
                    if (c >= nc) break;
                    // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32
                    const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                    float f[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        f[2 * k] = __uint_as_float(w[k] << 16);
                        f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
                    }
                    st_v4(yr + (size_t)c * 8, scale_to_bf16x8(f, se));
                }
            }
        }
    }
}

cudaError_t launch_expert_scale(const void *recv, const float *recv_scale, bool fp8, const int32_t *expert_offsets,
                                int E, int H, int rows, int identity, void *y, cudaStream_t stream) {
    const int warps = kExpertThreads / 32;
    const size_t smem = (size_t)(E + 1) * 4;
    // one warp per row and no persistent loop: the hardware hands each SM new
    // rows as its blocks finish (a single resident wave walking the rows was
    // 23 % slower on the FP8 prefill layer)
    long long grid = ((long long)rows + warps - 1) / warps;
    if (grid < 1) grid = 1;
    __nv_bfloat16 *yb = static_cast<__nv_bfloat16 *>(y);
    if (fp8)
        expert_scale_kernel<true><<<(unsigned)grid, kExpertThreads, smem, stream>>>(recv, recv_scale, expert_offsets, E,
                                                                                    H, rows, identity, yb);
    else
        expert_scale_kernel<false><<<(unsigned)grid, kExpertThreads, smem, stream>>>(recv, recv_scale, expert_offsets,
                                                                                     E, H, rows, identity, yb);
    return cudaGetLastError();
}

}  // namespace moe
