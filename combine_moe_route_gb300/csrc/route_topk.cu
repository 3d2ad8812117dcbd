// route_topk.cu -- the router's top-K selection and softmax weights.
//
// Perplexity, "Lower latency and higher throughput with multi-node DeepSeek
// deployment", section "MoE router": the router is a sort that keeps track of
// the indices of the selected scores; section "Expert parallelism": each token
// goes to K routed experts whose outputs are summed with weights.
//
// One warp per token.  Lane l holds logits e = l, l+32, l+64, ... in
// registers as an order-preserving 32-bit image of each fp32 value, sorts
// them once (a bitonic network on (key, expert) pairs) and keeps the sorted
// list in shared memory.  K rounds of: warp-wide maximum of the lanes' list
// heads by one redux.sync, then the smallest expert id among the lanes
// holding that maximum by a second one; the owning lane pops its head.  A
// round therefore costs O(1) per lane instead of a pass over E/32 keys.
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

// Descending bitonic sort of N (a power of two) values held in registers.
template <int N>
__device__ __forceinline__ void bitonic_sort_desc(unsigned long long (&c)[N]) {
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;   // direction of this bitonic run
                    const unsigned long long a = c[i], b = c[j];
                    const bool swap = desc ? (a < b) : (a > b);
                    c[i] = swap ? b : a;
                    c[j] = swap ? a : b;
                }
            }
        }
    }
}

template <int NPL>   // logits per lane: E <= 32 * NPL
struct RouteShape {
    static constexpr int kSlots = (NPL & (NPL - 1)) == 0 ? NPL : (NPL <= 16 ? 16 : 32);   // NPL padded to 2^n
    static constexpr int kWarps = kSlots >= 32 ? 4 : 8;                                     // 32 KB list at most
};

// G > 1: group-limited routing (Perplexity, "Lower latency and higher
// throughput with multi-node DeepSeek deployment", "MoE router": DeepSeek's
// group top-K, of which the plain top-K is the one-group case).  The E experts
// form G contiguous groups; a group scores its largest logit; the M best
// groups are kept (equal scores: smaller group id) and only their experts
// stay eligible for the K rounds.
template <int NPL>
__global__ void __launch_bounds__(RouteShape<NPL>::kWarps * 32) route_topk_kernel(const float *__restrict__ logits,
                                                                                  int T, int E, int K, int G, int M,
                                                                                  int32_t *__restrict__ topk_idx,
                                                                                  float *__restrict__ topk_w) {
    constexpr int NS = RouteShape<NPL>::kSlots;
    constexpr int kWarps = RouteShape<NPL>::kWarps;
    __shared__ uint32_t s_gmax[kWarps][32];
    __shared__ unsigned long long s_list[kWarps][NS * 32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const long long g = (long long)blockIdx.x * kWarps + warp;
    if (g >= T) return;

    const float *row = logits + g * (long long)E;
    uint32_t key[NPL];
    uint32_t avail = 0;   // bit i: slot i holds an eligible expert
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

    if (G > 1) {   // keep the M best groups; the experts of the others leave the race
        uint32_t *gm = s_gmax[warp];
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

    // Each lane sorts its eligible candidates once, descending, as 64-bit
    // (key, ~expert) composites -- on equal keys the smaller expert comes
    // first -- and parks the sorted list in shared memory, interleaved by
    // lane.  Then K rounds: every lane offers the head of its list; the warp
    // keeps the largest key (redux.sync) and, among the lanes offering it, the
    // smallest expert id (a second redux.sync); the winning lane's head moves
    // one entry on.  Empty entries are 0 and never win (every real key is > 0).
    unsigned long long c[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i)
        c[i] = (i < NPL && (avail & (1u << i)))
                   ? ((unsigned long long)key[i] << 32) | (unsigned long long)(~(uint32_t)(lane + 32 * i))
                   : 0ull;
    bitonic_sort_desc<NS>(c);
    unsigned long long *list = s_list[warp];
#pragma unroll
    for (int i = 0; i < NS; ++i) list[i * 32 + lane] = c[i];
    __syncwarp();
    int head = 0;
    int my_e = 0;
    uint32_t my_key = 0;
    for (int k = 0; k < K; ++k) {
        const unsigned long long h = (head < NS) ? list[head * 32 + lane] : 0ull;
        const uint32_t hk = (uint32_t)(h >> 32);
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, hk);
        const uint32_t cand = (hk == kmax && hk != 0u) ? ~(uint32_t)h : 0xffffffffu;
        const uint32_t e_win = __reduce_min_sync(0xffffffffu, cand);
        if ((int)(e_win & 31u) == lane) ++head;
        if (lane == k) {
            my_e = (int)e_win;
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
#define MOE_ROUTE_LAUNCH(NPL)                                                                       \
    route_topk_kernel<NPL><<<(unsigned)((T + RouteShape<NPL>::kWarps - 1) / RouteShape<NPL>::kWarps), \
                             RouteShape<NPL>::kWarps * 32, 0, stream>>>(logits, T, E, K, G, M, topk_idx, topk_w)
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
