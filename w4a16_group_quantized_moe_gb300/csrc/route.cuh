// route.cuh -- the per-token router shared by the routing kernels: softmax
// over E logits, the k most probable experts (ties to the lower index), and
// their probabilities renormalised over the k.  One warp per token; see
// route.cu for the method.
#pragma once
#include "common.cuh"

namespace moe {

// Monotone map fp32 -> u32, shifted by one so that 0 means "no candidate":
// a < b as floats (after -0 -> +0) iff key(a) < key(b); NaN maps to 1,
// below -inf.
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0;                                        // -0 -> +0
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 1;  // NaN
    return ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) + 1u;
}

// The largest untaken key of a lane and its slot (the lowest slot among
// equal keys), by a pairwise tree: blocks of 2, 4, ... slots, the right block
// winning only when strictly larger, so the depth is log2(PER), not PER.
template <int PER>
__device__ __forceinline__ void lane_best(const uint32_t (&key)[PER], uint32_t taken, uint32_t &bk,
                                          int &bj) {
    uint32_t kk[PER];
    int jj[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        kk[j] = ((taken >> j) & 1u) ? 0u : key[j];
        jj[j] = j;
    }
#pragma unroll
    for (int st = 1; st < PER; st *= 2)
#pragma unroll
        for (int j = 0; j + st < PER; j += 2 * st) {
            const bool r = kk[j + st] > kk[j];
            kk[j] = r ? kk[j + st] : kk[j];
            jj[j] = r ? jj[j + st] : jj[j];
        }
    bk = kk[0];
    bj = jj[0];
}

// A logit: through the read-only cache, or (FRESH: written earlier in the
// same kernel by other CTAs) from L2.
template <bool FRESH>
__device__ __forceinline__ float load_logit(const float *p) {
    return FRESH ? __ldcg(p) : __ldg(p);
}

// Routes one token with one warp.  PER = logits held per lane (E <= 32*PER).
// Writes ids and weights of token t to every destination given (non-null):
// topk_ids / topk_w at [t*k + j], and s_ids / s_w at [t*k + j].
template <int PER, bool FRESH = false>
__device__ __forceinline__ void route_token(const float *__restrict__ row, int E, int k, int t,
                                            int32_t *__restrict__ topk_ids, float *__restrict__ topk_w,
                                            int *s_ids, float *s_w = nullptr) {
    const int lane = threadIdx.x & 31;
    uint32_t key[PER];  // 0 = no candidate
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        key[j] = e < E ? order_key(load_logit<FRESH>(row + e)) : 0u;
    }
    // this lane's best untaken candidate (first maximum in index order)
    uint32_t bk, taken = 0;
    int bj;
    lane_best<PER>(key, taken, bk, bj);

    int my_id = 0;  // lane s keeps the s-th selection
    for (int s = 0; s < k; ++s) {
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t mine = (bk == kmax) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu;
        const int win = (int)__reduce_min_sync(0xffffffffu, mine);
        if (lane == s) my_id = win;
        if ((win & 31) == lane) {
            taken |= 1u << (win >> 5);
            lane_best<PER>(key, taken, bk, bj);
        }
    }

    // weights: softmax over the selected logits (rank 0 holds the maximum)
    const float my_logit = lane < k ? load_logit<FRESH>(row + my_id) : 0.f;
    const float m = __shfl_sync(0xffffffffu, my_logit, 0);
    const float ex = (lane < k) ? expf(my_logit - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) {
        const float w = ex / sum;
        if (topk_ids) topk_ids[(size_t)t * k + lane] = my_id;
        if (topk_w) topk_w[(size_t)t * k + lane] = w;
        if (s_ids) s_ids[t * k + lane] = my_id;
        if (s_w) s_w[t * k + lane] = w;
    }
}

// The same routing as route_token, written for a cold instruction cache: a
// kernel that routes once per launch runs this code once, and each 128-byte
// line of straight-line code costs an L2 round trip on first use, so the
// selection is a short loop over keys kept in shared memory (s_key: E
// words of this warp) instead of unrolled register code.  Each of the k
// rounds scans the lane's keys in ascending expert order (first maximum =
// lowest index), takes the warp maximum and, among lanes holding it, the
// lowest expert index; the winner's key is cleared.  Results are identical
// to route_token's.  E <= 1024.  With pub_n, every round also publishes its
// winner at once: pub_id[s] = expert of rank s, then (after a block-scope
// fence) *pub_n = s + 1, so other warps of the CTA can act on the first
// ranks while the later ones are still being chosen.
template <bool FRESH = false>
__device__ __forceinline__ void route_token_compact(const float *__restrict__ row, int E, int k, int t,
                                                    int32_t *__restrict__ topk_ids,
                                                    float *__restrict__ topk_w, int *s_ids, float *s_w,
                                                    uint32_t *s_key, int *pub_id = nullptr,
                                                    volatile int *pub_n = nullptr) {
    const int lane = threadIdx.x & 31;
    {
        // every load first (one memory round trip), then the keys
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = lane + 32 * j < E ? load_logit<FRESH>(row + lane + 32 * j) : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (lane + 32 * j < E) s_key[lane + 32 * j] = order_key(v[j]);
    }
    __syncwarp();
    int my_id = 0;
    for (int s = 0; s < k; ++s) {
        // two interleaved scans (even and odd strides), merged keeping the lower index on ties
        uint32_t b0 = 0, b1 = 0;
        int e0 = 0x7fffffff, e1 = 0x7fffffff;
        for (int e = lane; e < E; e += 64) {
            const uint32_t v0 = s_key[e];
            if (v0 > b0) { b0 = v0; e0 = e; }
            if (e + 32 < E) {
                const uint32_t v1 = s_key[e + 32];
                if (v1 > b1) { b1 = v1; e1 = e + 32; }
            }
        }
        if (b1 > b0 || (b1 == b0 && e1 < e0)) { b0 = b1; e0 = e1; }
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, b0);
        const int win = (int)__reduce_min_sync(0xffffffffu, b0 == kmax ? (uint32_t)e0 : 0xffffffffu);
        if (lane == s) my_id = win;
        if (lane == (win & 31)) s_key[win] = 0u;
        if (pub_n && lane == 0) {
            pub_id[s] = win;
            __threadfence_block();
            *pub_n = s + 1;
        }
        __syncwarp();
    }
    const float my_logit = lane < k ? load_logit<FRESH>(row + my_id) : 0.f;
    const float m = __shfl_sync(0xffffffffu, my_logit, 0);
    const float ex = (lane < k) ? expf(my_logit - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) {
        const float w = ex / sum;
        if (topk_ids) topk_ids[(size_t)t * k + lane] = my_id;
        if (topk_w) topk_w[(size_t)t * k + lane] = w;
        if (s_ids) s_ids[t * k + lane] = my_id;
        if (s_w) s_w[t * k + lane] = w;
    }
}

}  // namespace moe
