// route_topk.cu -- the router's top-K selection and softmax weights.
//
// Perplexity, "Lower latency and higher throughput with multi-node DeepSeek
// deployment", section "MoE router": the router is a sort that keeps track of
// the indices of the selected scores; section "Expert parallelism": each token
// goes to K routed experts whose outputs are summed with weights.
//
// One warp per token.  Lane l holds logits e = l, l+32, l+64, ... in
// registers as an order-preserving 32-bit image of each fp32 value.  The
// K-th largest lane maximum, its lowest 5 bits replaced by a lane tag so that
// K rounds of one redux.sync each find it, gives tau, a lower bound of the
// row's K-th largest key, so the top K is among the candidates key >= tau --
// on random rows K plus a few.  The candidates are
// compacted into shared memory and each one's output position is the number
// of candidates ahead of it (larger key, or equal key and smaller id).  Rows
// with more than kMaxCandidates candidates (many equal keys) instead take K
// rounds of (lane best, redux.sync max of the key, redux.sync min of the id).
// The weights are a softmax over the K winners, max-subtracted (the first
// winner is the largest), exponentials summed by a warp butterfly, one IEEE
// division.  A warp takes several tokens in turn (with up to 12 logits per
// lane it loads the next token's logits while it selects the current one's);
// when E = 32 * NPL is a multiple of 128, the logits are read 16 bytes at a
// time, four consecutive experts per lane; with groups that layout serves group
// sizes that are whole runs of lanes of a 128-expert block or whole blocks.
#include <atomic>

#include "launch.h"

namespace moe {

// fp32 -> uint32 with the same order (+0 and -0 map to the same value).
// Adding +0 turns -0 into +0 and leaves every other value unchanged (round to
// nearest, denormals kept); then negative values have all bits flipped and
// non-negative ones their sign bit set.
__device__ __forceinline__ uint32_t ordered_key(float v) {
    const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

struct RouteShape {
    static constexpr int kWarps = 8;   // tokens (warps) per block
};

// Candidates ranked in shared memory; a row with more candidates than this
// (many equal keys) takes the K-round path instead.
constexpr int kMaxCandidates = 64;

// The expert in slot i of a lane.  Interleaved: lane + 32 i.  With 16-byte
// loads (plain routing, E = 32 * NPL a multiple of 128): each lane holds four
// consecutive experts of every 128, 128 (i / 4) + 4 lane + i % 4.
template <bool kVec>
__device__ __forceinline__ int slot_expert(int lane, int i) {
    return kVec ? ((i >> 2) << 7) + (lane << 2) + (i & 3) : lane + 32 * i;
}

// One row of logits into the lane's slots (0 past E).
template <int NPL, bool kVec>
__device__ __forceinline__ void load_row(const float *__restrict__ row, int E, int lane, float (&v)[NPL]) {
    if (kVec) {
#pragma unroll
        for (int q = 0; q < NPL / 4; ++q) {
            const float4 f = __ldg(reinterpret_cast<const float4 *>(row + q * 128 + lane * 4));
            v[4 * q] = f.x;
            v[4 * q + 1] = f.y;
            v[4 * q + 2] = f.z;
            v[4 * q + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            v[i] = (e < E) ? __ldg(row + e) : 0.0f;
        }
    }
}

// G > 1: group-limited routing (Perplexity, "Lower latency and higher
// throughput with multi-node DeepSeek deployment", "MoE router": DeepSeek's
// group top-K, of which the plain top-K is the one-group case).  The E experts
// form G contiguous groups; a group scores its largest logit; the M best
// groups are kept (equal scores: smaller group id) and only their experts
// stay eligible for the K rounds.
template <int NPL, bool kVec, bool kVecGroups>   // logits per lane: E <= 32 * NPL
__global__ void __launch_bounds__(RouteShape::kWarps * 32) route_topk_kernel(const float *__restrict__ logits,
                                                                                  int T, int E, int K, int G, int M,
                                                                                  int32_t *__restrict__ topk_idx,
                                                                                  float *__restrict__ topk_w) {
    constexpr int kWarps = RouteShape::kWarps;
    __shared__ uint32_t s_gmax[kWarps][32];
    __shared__ unsigned long long s_cand[kWarps][kMaxCandidates];
    __shared__ unsigned long long s_win[kWarps][MOE_MAX_TOPK];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    // the warp takes tokens g, g + stride, ...; with up to 12 logits per lane
    // each token's logits are loaded while the previous token's selection runs
    // (with more, the extra registers cost more occupancy than the prefetch gains)
    constexpr bool kPrefetch = NPL <= 12;
    const long long stride = (long long)gridDim.x * kWarps;
    long long g = (long long)blockIdx.x * kWarps + warp;
    if (g >= T) return;
    float nxt[NPL];
    if (kPrefetch) load_row<NPL, kVec>(logits + g * (long long)E, E, lane, nxt);
    for (;; g += stride) {
        if (!kPrefetch) load_row<NPL, kVec>(logits + g * (long long)E, E, lane, nxt);
        uint32_t key[NPL];
        uint32_t avail = 0;   // bit i: slot i holds an eligible expert
        // (the 16-byte-load layout runs only over exactly E = 32 * NPL experts,
        // so there every slot is in range)
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            if (kVec || slot_expert<kVec>(lane, i) < E) {
                key[i] = ordered_key(nxt[i]);
                avail |= 1u << i;
            } else {
                key[i] = 0u;
            }
        }
        const bool more = g + stride < T;
        if (kPrefetch && more) load_row<NPL, kVec>(logits + (g + stride) * (long long)E, E, lane, nxt);

        // keep the M best groups; the experts of the others leave the race
        if constexpr (kVec && kVecGroups) {
            // 16-byte layout: lane l's slots 4m..4m+3 hold experts 128m + 4l .. +3.
            // A group of gs < 128 experts is gs/4 consecutive lanes of one
            // 128-expert block m (gs/4 a power of two); a group of gs >= 128 is
            // gs/128 whole blocks.  vm[m]: the lane's largest key of block m.
            const int gs = E / G;
            uint32_t vm[NPL / 4];
#pragma unroll
            for (int m = 0; m < NPL / 4; ++m)
                vm[m] = max(max(key[4 * m], key[4 * m + 1]), max(key[4 * m + 2], key[4 * m + 3]));
            uint32_t gkey = 0u;   // lane q < G: the largest key of group q (every real key is > 0)
            int lpg = 0, gpm = 0, bpg = 0;
            if (gs < 128) {
                lpg = gs >> 2;     // lanes per group
                gpm = 128 / gs;    // groups per block
#pragma unroll
                for (int m = 0; m < NPL / 4; ++m)
                    for (int off = 1; off < lpg; off <<= 1)
                        vm[m] = max(vm[m], __shfl_xor_sync(0xffffffffu, vm[m], off));
                // group q = m * gpm + s sits in lanes s * lpg .. s * lpg + lpg - 1 of block m
                const int src = (lane % gpm) * lpg;
#pragma unroll
                for (int m = 0; m < NPL / 4; ++m) {
                    const uint32_t t = __shfl_sync(0xffffffffu, vm[m], src);
                    if (lane / gpm == m) gkey = t;
                }
            } else {
                bpg = gs >> 7;     // blocks per group
#pragma unroll
                for (int m = 0; m < NPL / 4; ++m) {
                    const uint32_t t = __reduce_max_sync(0xffffffffu, vm[m]);
                    if (lane == m / bpg) gkey = max(gkey, t);
                }
            }
            bool open = lane < G;
            uint32_t kept = 0u;
            for (int r = 0; r < M; ++r) {
                const uint32_t gmax = __reduce_max_sync(0xffffffffu, open ? gkey : 0u);
                const uint32_t gwin =
                    __reduce_min_sync(0xffffffffu, (open && gkey == gmax) ? (uint32_t)lane : 0xffffffffu);
                kept |= 1u << gwin;
                if ((uint32_t)lane == gwin) open = false;
            }
#pragma unroll
            for (int m = 0; m < NPL / 4; ++m) {
                const int q = (gs < 128) ? m * gpm + lane / lpg : m / bpg;
                if (!((kept >> q) & 1u)) avail &= ~(0xfu << (4 * m));
            }
        }
        if (!kVec && G > 1) {
            const int gs = E / G;
            // group of slot i, when every slot lies inside one group (group size a
            // multiple of 32): slots 0..spg-1 are group 0, and so on
            const bool whole_slots = (gs & 31) == 0;
            int slot_group[NPL];
            uint32_t gkey = 0u;   // lane q < G: the largest key of group q (every real key is > 0)
            if (whole_slots) {
                const int spg = gs >> 5;
                int q = 0, c = 0;
#pragma unroll
                for (int i = 0; i < NPL; ++i) {
                    slot_group[i] = q;
                    if (++c == spg) {
                        c = 0;
                        ++q;
                    }
                }
#pragma unroll
                for (int i = 0; i < NPL; ++i) {
                    const uint32_t m = __reduce_max_sync(0xffffffffu, (avail & (1u << i)) ? key[i] : 0u);
                    if (lane == slot_group[i]) gkey = max(gkey, m);
                }
            } else {
#pragma unroll
                for (int i = 0; i < NPL; ++i) slot_group[i] = (lane + 32 * i) / gs;
                uint32_t *gm = s_gmax[warp];
                if (lane < G) gm[lane] = 0u;
                __syncwarp();
#pragma unroll
                for (int i = 0; i < NPL; ++i)
                    if (avail & (1u << i)) atomicMax(&gm[slot_group[i]], key[i]);
                __syncwarp();
                if (lane < G) gkey = gm[lane];
            }
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
                if (slot_group[i] >= 32 || !((kept >> slot_group[i]) & 1u)) avail &= ~(1u << i);
        }

        // Threshold.  Each lane's maximum keeps its upper 27 bits and takes the
        // tag 31 - lane in its lower 5, so the 32 tagged values are distinct and
        // each of K rounds retires exactly one of them with a single redux.sync.
        // tau = the upper 27 bits of the K-th largest tagged value.  The K retired
        // lanes each hold a key >= tau, so the K-th largest key of the row is
        // >= tau, and every member of the top K (ties included) is a candidate:
        // an eligible key >= tau.  Truncating only lowers tau, which admits a few
        // more candidates, never fewer.  If fewer than K lanes hold a key, the
        // rounds run out (top = 0) and every eligible key is a candidate.  On
        // random rows only a few keys beyond K pass.
        uint32_t ek[NPL];   // eligible keys; 0 = not eligible (every real key is > 0)
        uint32_t lmax = 0u;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            // the plain top-K keeps every in-range slot; key[i] is already 0 past E
            ek[i] = ((kVec && !kVecGroups) || (!kVec && G <= 1) || (avail & (1u << i))) ? key[i] : 0u;
            lmax = max(lmax, ek[i]);
        }
        uint32_t v = lmax ? ((lmax & ~31u) | (uint32_t)(31 - lane)) : 0u;
        uint32_t top = 0u;
        for (int k = 0; k < K; ++k) {
            top = __reduce_max_sync(0xffffffffu, v);
            if (v == top) v = 0u;   // the one lane holding top (top = 0: nothing left, no change)
        }
        // at least 1, so that one compare also drops the ineligible slots (key 0)
        const uint32_t tau = max(top & ~31u, 1u);
        uint32_t cm = 0u;   // bit i: slot i is a candidate
#pragma unroll
        for (int i = 0; i < NPL; ++i)
            if (ek[i] >= tau) cm |= 1u << i;
        const int cnt = __popc(cm);
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const int n = __shfl_sync(0xffffffffu, incl, 31);

        int my_e = 0;
        uint32_t my_key = 0;
        if (n <= kMaxCandidates) {
            // rank each candidate by the 64-bit (key, ~expert) composite: a larger
            // composite is a larger key or, on equal keys, a smaller expert id
            unsigned long long *cand = s_cand[warp];
            int pos = incl - cnt;
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (cm & (1u << i))
                    cand[pos++] = ((unsigned long long)ek[i] << 32) |
                                  (unsigned long long)(~(uint32_t)slot_expert<kVec>(lane, i));
            __syncwarp();
            for (int c = lane; c < n; c += 32) {
                const unsigned long long me = cand[c];
                int r = 0;
                for (int m = 0; m < n; ++m) r += (cand[m] > me) ? 1 : 0;
                if (r < K) s_win[warp][r] = me;
            }
            __syncwarp();
            if (lane < K) {
                const unsigned long long wv = s_win[warp][lane];
                my_key = (uint32_t)(wv >> 32);
                my_e = (int)~(uint32_t)wv;
            }
        } else {
            // many equal keys: K rounds of (each lane's best remaining key, the
            // warp's largest by redux.sync, the smallest expert id among the lanes
            // holding it by a second redux.sync; the owner retires it)
            for (int k = 0; k < K; ++k) {
                uint32_t bk = 0u;
                int bi = -1;
#pragma unroll
                for (int i = 0; i < NPL; ++i)
                    if (ek[i] > bk) {
                        bk = ek[i];
                        bi = i;
                    }
                const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
                uint32_t cand = 0xffffffffu;
#pragma unroll
                for (int i = 0; i < NPL; ++i)
                    if (i == bi && bk == kmax) cand = (uint32_t)slot_expert<kVec>(lane, i);
                const uint32_t e_win = __reduce_min_sync(0xffffffffu, cand);
#pragma unroll
                for (int i = 0; i < NPL; ++i)
                    if ((uint32_t)slot_expert<kVec>(lane, i) == e_win) ek[i] = 0u;
                if (lane == k) {
                    my_e = (int)e_win;
                    my_key = kmax;
                }
            }
        }

        // softmax over the K winners (lane j < K holds winner j); the exponentials
        // are summed by a butterfly, which leaves the same sum in every lane
        const float my_l = key_to_float(my_key);
        const float m = __shfl_sync(0xffffffffu, my_l, 0);
        const float ex = (lane < K) ? expf(my_l - m) : 0.0f;
        float sum = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane < K) {
            topk_idx[g * K + lane] = my_e;
            topk_w[g * K + lane] = ex / sum;
        }
        if (!more) break;
        __syncwarp();   // s_cand / s_win are refilled for the next token
    }
}

#ifndef MOE_ROUTE_WAVES
#define MOE_ROUTE_WAVES 2   // resident waves of blocks; each warp then walks its share of the tokens
#endif

// One block per 8 tokens, capped at MOE_ROUTE_WAVES resident waves of blocks
// when the kernel prefetches (measured on the DeepSeek-V3 prefill logits: 2
// waves 19.4 us, 3 waves 19.8 us, 4 waves 20.5 us; on an earlier build 1 wave
// was 23.0 us and one token per warp 23.3 us against 21.5 us for 2 waves).
template <int NPL, bool kVec, bool kVecGroups>
static cudaError_t launch_npl(const float *logits, int T, int E, int K, int G, int M, int32_t *topk_idx,
                              float *topk_w, cudaStream_t stream) {
    static std::atomic<int> per_sm_cache[64];
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return ce;
    if (dev < 0 || dev >= 64) dev = 0;
    int per_sm = per_sm_cache[dev].load(std::memory_order_relaxed);
    if (per_sm == 0) {
        ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_topk_kernel<NPL, kVec, kVecGroups>,
                                                           RouteShape::kWarps * 32, 0);
        if (ce != cudaSuccess) return ce;
        if (per_sm < 1) per_sm = 1;
        per_sm_cache[dev].store(per_sm, std::memory_order_relaxed);
    }
    long long grid = ((long long)T + RouteShape::kWarps - 1) / RouteShape::kWarps;
    const long long cap = (long long)device_sm_count() * per_sm * MOE_ROUTE_WAVES;
    if (NPL <= 12 && grid > cap) grid = cap;
    route_topk_kernel<NPL, kVec, kVecGroups><<<(unsigned)grid, RouteShape::kWarps * 32, 0, stream>>>(
        logits, T, E, K, G, M, topk_idx, topk_w);
    return cudaGetLastError();
}

template <int NPL>
static cudaError_t launch_layout(const float *logits, int T, int E, int K, int G, int M, int32_t *topk_idx,
                                 float *topk_w, cudaStream_t stream) {
    // 16-byte loads: exactly 32 * NPL experts, a multiple of 128, aligned rows; groups
    // that are whole lane runs of a 128-expert block (gs/4 lanes, a power of two) or
    // whole blocks
    if constexpr (NPL % 4 == 0) {
        if (E == 32 * NPL && (reinterpret_cast<uintptr_t>(logits) & 15) == 0) {
            if (G <= 1) return launch_npl<NPL, true, false>(logits, T, E, K, G, M, topk_idx, topk_w, stream);
            const int gs = E / G;
            const bool runs = gs < 128 && gs % 4 == 0 && 128 % gs == 0;
            if (runs || gs % 128 == 0)
                return launch_npl<NPL, true, true>(logits, T, E, K, G, M, topk_idx, topk_w, stream);
        }
    }
    return launch_npl<NPL, false, false>(logits, T, E, K, G, M, topk_idx, topk_w, stream);
}

cudaError_t launch_route_topk(const float *logits, int T, int E, int K, int G, int M, int32_t *topk_idx,
                              float *topk_w, cudaStream_t stream) {
    if (E <= 32) return launch_layout<1>(logits, T, E, K, G, M, topk_idx, topk_w, stream);
    if (E <= 64) return launch_layout<2>(logits, T, E, K, G, M, topk_idx, topk_w, stream);
    if (E <= 128) return launch_layout<4>(logits, T, E, K, G, M, topk_idx, topk_w, stream);
    if (E <= 256) return launch_layout<8>(logits, T, E, K, G, M, topk_idx, topk_w, stream);
    if (E <= 384) return launch_layout<12>(logits, T, E, K, G, M, topk_idx, topk_w, stream);
    if (E <= 512) return launch_layout<16>(logits, T, E, K, G, M, topk_idx, topk_w, stream);
    return launch_layout<32>(logits, T, E, K, G, M, topk_idx, topk_w, stream);
}

}  // namespace moe
