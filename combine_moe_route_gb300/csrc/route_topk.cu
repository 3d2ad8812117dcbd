// route_topk.cu -- the router's top-K selection and softmax weights.
//
// Perplexity, "Lower latency and higher throughput with multi-node DeepSeek
// deployment", section "MoE router": the router is a sort that keeps track of
// the indices of the selected scores; section "Expert parallelism": each token
// goes to K routed experts whose outputs are summed with weights.
//
// One warp per token.  Lane l holds logits e = l, l+32, l+64, ... in
// registers.  Each logit becomes a 64-bit key (order-preserving image of the
// fp32 value in the high word, the complement of the expert id in the low
// word, so that a larger key means a larger logit and, on equal logits, a
// smaller id).  K rounds of: per-lane maximum over its not-yet-chosen keys,
// warp-wide maximum by butterfly shuffles, the owning lane marks the winner.
// The weights are a softmax over the K winners, max-subtracted (the first
// winner is the largest), exponentials summed in j order, one IEEE division.
#include "launch.h"

namespace moe {

// fp32 -> uint32 with the same order (+0 and -0 map to the same value).
__device__ __forceinline__ uint32_t ordered_key(float v) {
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0u;   // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

template <int NPL>   // logits per lane: E <= 32 * NPL
__global__ void __launch_bounds__(256) route_topk_kernel(const float *__restrict__ logits, int T, int E, int K,
                                                         int32_t *__restrict__ topk_idx,
                                                         float *__restrict__ topk_w) {
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const long long g = (long long)blockIdx.x * warps + (threadIdx.x >> 5);
    if (g >= T) return;

    const float *row = logits + g * (long long)E;
    uint32_t key[NPL];
    uint32_t avail = 0;   // bit i: slot i holds a not-yet-chosen expert
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            key[i] = ordered_key(__ldg(row + e));
            avail |= 1u << i;
        } else {
            key[i] = 0u;
        }
    }

    int my_e = 0;
    uint32_t my_key = 0;
    for (int k = 0; k < K; ++k) {
        unsigned long long best = 0ull;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            if (avail & (1u << i)) {
                const unsigned long long c =
                    ((unsigned long long)key[i] << 32) | (unsigned long long)(0xffffffffu - (uint32_t)(lane + 32 * i));
                best = c > best ? c : best;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
            best = o > best ? o : best;
        }
        const int e_win = (int)(0xffffffffu - (uint32_t)(best & 0xffffffffull));
        if ((e_win & 31) == lane) avail &= ~(1u << (e_win >> 5));
        if (lane == k) {
            my_e = e_win;
            my_key = (uint32_t)(best >> 32);
        }
    }

    // softmax over the K winners (lane j < K holds winner j)
    const float my_l = key_to_float(my_key);
    const float m = __shfl_sync(0xffffffffu, my_l, 0);
    const float ex = (lane < K) ? expf(my_l - m) : 0.0f;
    float sum = 0.0f;
    for (int j = 0; j < K; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
    if (lane < K) {
        topk_idx[g * K + lane] = my_e;
        topk_w[g * K + lane] = ex / sum;
    }
}

cudaError_t launch_route_topk(const float *logits, int T, int E, int K, int32_t *topk_idx, float *topk_w,
                              cudaStream_t stream) {
    constexpr int kThreads = 256;
    const int warps = kThreads / 32;
    const unsigned grid = (unsigned)((T + warps - 1) / warps);
    if (E <= 32)
        route_topk_kernel<1><<<grid, kThreads, 0, stream>>>(logits, T, E, K, topk_idx, topk_w);
    else if (E <= 64)
        route_topk_kernel<2><<<grid, kThreads, 0, stream>>>(logits, T, E, K, topk_idx, topk_w);
    else if (E <= 128)
        route_topk_kernel<4><<<grid, kThreads, 0, stream>>>(logits, T, E, K, topk_idx, topk_w);
    else if (E <= 256)
        route_topk_kernel<8><<<grid, kThreads, 0, stream>>>(logits, T, E, K, topk_idx, topk_w);
    else if (E <= 384)
        route_topk_kernel<12><<<grid, kThreads, 0, stream>>>(logits, T, E, K, topk_idx, topk_w);
    else if (E <= 512)
        route_topk_kernel<16><<<grid, kThreads, 0, stream>>>(logits, T, E, K, topk_idx, topk_w);
    else
        route_topk_kernel<32><<<grid, kThreads, 0, stream>>>(logits, T, E, K, topk_idx, topk_w);
    return cudaGetLastError();
}

}  // namespace moe
