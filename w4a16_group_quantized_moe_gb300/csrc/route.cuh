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
// words of this warp) instead of unrolled register code.  Every lane keeps
// the best of its keys (scanned in ascending expert order: first maximum =
// lowest index); each of the k rounds takes the warp maximum and, among
// lanes holding it, the lowest expert index, clears the winner's key, and
// only the winning lane scans its keys again.  Results are identical to
// route_token's.  E <= 1024.  With pub_n, every round also publishes its
// winner at once: pub_id[s] = expert of rank s, then (after a block-scope
// fence) *pub_n = s + 1, so other warps of the CTA can act on the first
// ranks while the later ones are still being chosen.
//
// With lbar (an mbarrier of this warp's own, in shared memory), a row that
// starts on a 16-byte boundary with E a multiple of 4 arrives by one bulk
// copy into s_key and is turned into keys in place by a short loop: the
// straight-line code of 32 loads per lane is the longest stretch of cold
// code in a kernel that routes once.  The winners' logits are recovered
// from their keys (order_key is invertible up to -0 -> +0 and the NaN
// payload), so the row is read once.
__device__ __forceinline__ float key_value(uint32_t key) {
    const uint32_t u = key - 1u;
    return __uint_as_float((u & 0x80000000u) ? (u ^ 0x80000000u) : ~u);
}

template <bool FRESH = false>
__device__ __forceinline__ void route_token_compact(const float *__restrict__ row, int E, int k, int t,
                                                    int32_t *__restrict__ topk_ids,
                                                    float *__restrict__ topk_w, int *s_ids, float *s_w,
                                                    uint32_t *s_key, int *pub_id = nullptr,
                                                    volatile int *pub_n = nullptr, uint64_t *lbar = nullptr) {
    const int lane = threadIdx.x & 31;
    bool loaded = false;
    if (lbar && ((reinterpret_cast<uintptr_t>(row) | (uintptr_t)E * 4u) & 15u) == 0) {
        if (lane == 0) {
            mbar_init(lbar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(lbar, (uint32_t)E * 4u);
            bulk_g2s(s_key, row, (uint32_t)E * 4u, lbar);
        }
        __syncwarp();
        // a wait that expires (about a second; never with a working copy
        // engine) falls back to the loads below
        loaded = mbar_wait_bounded(lbar, 0, nullptr);
        if (loaded)
            for (int e = lane; e < E; e += 32) s_key[e] = order_key(__uint_as_float(s_key[e]));
    }
    if (!loaded) {
        // every load first (one memory round trip), then the keys
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = lane + 32 * j < E ? load_logit<FRESH>(row + lane + 32 * j) : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (lane + 32 * j < E) s_key[lane + 32 * j] = order_key(v[j]);
    }
    __syncwarp();
    // each lane's best untaken key and its expert (the first maximum in
    // ascending expert order, so the lowest index among equal keys); only the
    // lane whose candidate a round takes scans its keys again
    uint32_t bk = 0;
    int be = 0x7fffffff;
    auto lane_scan = [&]() {
        bk = 0;
        be = 0x7fffffff;
        for (int e0 = lane; e0 < E; e0 += 256) {
            uint32_t v[8];  // eight loads in flight, then the compares in ascending order
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = e0 + 32 * u < E ? s_key[e0 + 32 * u] : 0u;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (v[u] > bk) {
                    bk = v[u];
                    be = e0 + 32 * u;
                }
            }
        }
    };
    lane_scan();
    int my_id = 0;
    uint32_t my_key = 0;
    for (int s = 0; s < k; ++s) {
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
        const int win = (int)__reduce_min_sync(0xffffffffu, bk == kmax ? (uint32_t)be : 0xffffffffu);
        if (lane == s) {
            my_id = win;
            my_key = kmax;
        }
        if (pub_n && lane == 0) {
            pub_id[s] = win;
            __threadfence_block();
            *pub_n = s + 1;
        }
        if (lane == (win & 31)) {
            s_key[win] = 0u;
            lane_scan();
        }
        __syncwarp();
    }
    const float my_logit = lane < k ? key_value(my_key) : 0.f;
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
