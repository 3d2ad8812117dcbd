// route_topk.cu -- the router's top-K selection and softmax weights.
//
// Perplexity, "Lower latency and higher throughput with multi-node DeepSeek
// deployment", section "MoE router": the router is a sort that keeps track of
// the indices of the selected scores; section "Expert parallelism": each token
// goes to K routed experts whose outputs are summed with weights.
//
// One warp per token.  Lane l holds logits e = l, l+32, l+64, ... in
// registers as an order-preserving 32-bit image of each fp32 value.  K
// rounds of: per-lane maximum over its not-yet-chosen keys, warp-wide maximum
// of the image by one redux.sync, then the smallest expert id among the lanes
// holding that maximum by a second one; the owning lane marks the winner.
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

constexpr int kRouteThreads = 256;

// G > 1: group-limited routing (Perplexity, "Lower latency and higher
// throughput with multi-node DeepSeek deployment", "MoE router": DeepSeek's
// group top-K, of which the plain top-K is the one-group case).  The E experts
// form G contiguous groups; a group scores its largest logit; the M best
// groups are kept (equal scores: smaller group id) and only their experts
// stay eligible for the K rounds.
template <int NPL>   // logits per lane: E <= 32 * NPL
__global__ void __launch_bounds__(kRouteThreads) route_topk_kernel(const float *__restrict__ logits, int T, int E,
                                                                   int K, int G, int M,
                                                                   int32_t *__restrict__ topk_idx,
                                                                   float *__restrict__ topk_w) {
    __shared__ uint32_t s_gmax[kRouteThreads / 32][32];
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

    // K rounds: each lane offers its best remaining key (on equal keys its
    // lowest slot, i.e. its lowest expert id); the warp keeps the largest key
    // (one redux.sync) and, among the lanes offering it, the smallest id
    // (a second redux.sync).
    if (G > 1) {
        uint32_t *gm = s_gmax[threadIdx.x >> 5];
        const int gs = E / G;
        if (lane < G) gm[lane] = 0u;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < NPL; ++i)
            if (avail & (1u << i)) atomicMax(&gm[(lane + 32 * i) / gs], key[i]);
        __syncwarp();
        const uint32_t gkey = (lane < G) ? gm[lane] : 0u;   // every real group's key is > 0
        bool open = lane < G;
        uint32_t kept = 0u;
        for (int r = 0; r < M; ++r) {
            const uint32_t gmax = __reduce_max_sync(0xffffffffu, open ? gkey : 0u);
            const uint32_t gwin = __reduce_min_sync(0xffffffffu, (open && gkey == gmax) ? (uint32_t)lane : 0xffffffffu);
            kept |= 1u << gwin;
            if ((uint32_t)lane == gwin) open = false;
        }
#pragma unroll
        for (int i = 0; i < NPL; ++i)
            if (!((kept >> ((lane + 32 * i) / gs)) & 1u)) avail &= ~(1u << i);
    }

    int my_e = 0;
    uint32_t my_key = 0;
    for (int k = 0; k < K; ++k) {
        uint32_t bk = 0u;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            if ((avail & (1u << i)) && key[i] > bk) {
                bk = key[i];
                bi = i;
            }
        }
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t cand = (bi >= 0 && bk == kmax) ? (uint32_t)(lane + 32 * bi) : 0xffffffffu;
        const int e_win = (int)__reduce_min_sync(0xffffffffu, cand);
        if ((e_win & 31) == lane) avail &= ~(1u << (e_win >> 5));
        if (lane == k) {
            my_e = e_win;
            my_key = kmax;
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

cudaError_t launch_route_topk(const float *logits, int T, int E, int K, int G, int M, int32_t *topk_idx,
                              float *topk_w, cudaStream_t stream) {
    const int warps = kRouteThreads / 32;
    const unsigned grid = (unsigned)((T + warps - 1) / warps);
#define MOE_ROUTE_LAUNCH(NPL) \
    route_topk_kernel<NPL><<<grid, kRouteThreads, 0, stream>>>(logits, T, E, K, G, M, topk_idx, topk_w)
    if (E <= 32)
        MOE_ROUTE_LAUNCH(1);
    else if (E <= 64)
        MOE_ROUTE_LAUNCH(2);
    else if (E <= 128)
        MOE_ROUTE_LAUNCH(4);
    else if (E <= 256)
        MOE_ROUTE_LAUNCH(8);
    else if (E <= 384)
        MOE_ROUTE_LAUNCH(12);
    else if (E <= 512)
        MOE_ROUTE_LAUNCH(16);
    else
        MOE_ROUTE_LAUNCH(32);
#undef MOE_ROUTE_LAUNCH
    return cudaGetLastError();
}

}  // namespace moe
