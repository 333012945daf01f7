// route.cu -- step 1: softmax router with top-k selection and renormalised
// weights.  Geometry from "[Model][SM70] Adapt Qwen3.8 Flash Next NVFP4",
// section Implemented route (512 experts, top-10); ties go to the lower
// expert index.
//
// One warp per token.  The token's E logits are held in registers (lane l
// holds experts l, l+32, ...), turned into order-preserving integer keys,
// and k rounds of a warp arg-max pick the experts in rank order.  The
// renormalised weights are a softmax over the k selected logits: the full
// softmax denominator cancels when the selected probabilities are divided
// by their sum.
#include "common.cuh"

namespace moe {

constexpr int kRouteWarpsPerBlock = 4;
constexpr int kRouteMaxE = 1024;
constexpr int kRoutePerLane = kRouteMaxE / 32;

// Monotone map fp32 -> u32: a < b as floats (after -0 -> +0) iff key(a) <
// key(b); every NaN maps to 0, below -inf.
__device__ inline uint32_t order_key(float v) {
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0;                                        // -0 -> +0
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0;  // NaN
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kRouteWarpsPerBlock * 32)
route_kernel(const float *__restrict__ logits, int T, int E, int k,
             int32_t *__restrict__ topk_ids, float *__restrict__ topk_w) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *row = logits + (size_t)t * E;

    uint32_t key[kRoutePerLane];
    uint32_t taken = 0;  // bit j: expert lane + 32 j already selected (or absent)
#pragma unroll
    for (int j = 0; j < kRoutePerLane; ++j) {
        const int e = lane + 32 * j;
        if (e < E) {
            key[j] = order_key(__ldg(row + e));
        } else {
            key[j] = 0;
            taken |= 1u << j;
        }
    }

    int my_id = -1;        // lane s keeps the s-th selection
    float my_logit = 0.f;
    for (int s = 0; s < k; ++s) {
        // best untaken expert of this lane (first max in index order)
        uint32_t bk = 0;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kRoutePerLane; ++j) {
            const bool cand = !((taken >> j) & 1u);
            if (cand && (bi == 0x7fffffff || key[j] > bk)) {
                bk = key[j];
                bi = lane + 32 * j;
            }
        }
        // warp arg-max: larger key, then lower index
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const uint32_t ok = __shfl_xor_sync(0xffffffffu, bk, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ok > bk || (ok == bk && oi < bi)) {
                bk = ok;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == s) {
            my_id = bi;
            my_logit = __ldg(row + bi);
        }
    }

    // weights: softmax over the selected logits (rank 0 holds the maximum)
    const float m = __shfl_sync(0xffffffffu, my_logit, 0);
    float ex = (lane < k) ? expf(my_logit - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) {
        topk_ids[(size_t)t * k + lane] = my_id;
        topk_w[(size_t)t * k + lane] = ex / sum;
    }
}

cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                         cudaStream_t stream) {
    const int blocks = (T + kRouteWarpsPerBlock - 1) / kRouteWarpsPerBlock;
    route_kernel<<<blocks, kRouteWarpsPerBlock * 32, 0, stream>>>(logits, T, E, k, ids, w);
    return cudaGetLastError();
}

}  // namespace moe
