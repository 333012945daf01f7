// route.cu -- step 1: softmax router with top-k selection and renormalised
// weights.  Geometry from "[Model][SM70] Adapt Qwen3.8 Flash Next NVFP4",
// section Implemented route (512 experts, top-10); ties go to the lower
// expert index.
//
// One warp per token.  The token's E logits are held in registers (lane l
// holds experts l, l+32, ...) as order-preserving integer keys.  Each of the
// k rounds takes the warp maximum of the lanes' current best keys with one
// redux.sync, resolves equal keys to the lowest expert index with a second
// one, and lets only the winning lane rescan its candidates.  The
// renormalised weights are a softmax over the k selected logits: the full
// softmax denominator cancels when the selected probabilities are divided by
// their sum.
#include "common.cuh"

namespace moe {

constexpr int kRouteWarpsPerBlock = 4;

// Monotone map fp32 -> u32, shifted by one so that 0 means "no candidate":
// a < b as floats (after -0 -> +0) iff key(a) < key(b); NaN maps to 1,
// below -inf.
__device__ inline uint32_t order_key(float v) {
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0;                                        // -0 -> +0
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 1;  // NaN
    return ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) + 1u;
}

// PER = logits held per lane (E <= 32 * PER).
template <int PER>
__global__ void __launch_bounds__(kRouteWarpsPerBlock * 32)
route_kernel(const float *__restrict__ logits, int T, int E, int k,
             int32_t *__restrict__ topk_ids, float *__restrict__ topk_w) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *row = logits + (size_t)t * E;

    uint32_t key[PER];  // 0 = no candidate
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        key[j] = e < E ? order_key(__ldg(row + e)) : 0u;
    }
    // this lane's best untaken candidate (first maximum in index order)
    uint32_t bk = 0, taken = 0;
    int bj = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j)
        if (key[j] > bk) {
            bk = key[j];
            bj = j;
        }

    int my_id = 0;  // lane s keeps the s-th selection
    for (int s = 0; s < k; ++s) {
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t mine = (bk == kmax) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu;
        const int win = (int)__reduce_min_sync(0xffffffffu, mine);
        if (lane == s) my_id = win;
        if ((win & 31) == lane) {
            taken |= 1u << (win >> 5);
            bk = 0;
            bj = 0;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const uint32_t c = ((taken >> j) & 1u) ? 0u : key[j];
                if (c > bk) {
                    bk = c;
                    bj = j;
                }
            }
        }
    }

    // weights: softmax over the selected logits (rank 0 holds the maximum)
    const float my_logit = lane < k ? __ldg(row + my_id) : 0.f;
    const float m = __shfl_sync(0xffffffffu, my_logit, 0);
    const float ex = (lane < k) ? expf(my_logit - m) : 0.f;
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
    const int threads = kRouteWarpsPerBlock * 32;
    if (E <= 64) return launch_pdl(route_kernel<2>, blocks, threads, 0, stream, logits, T, E, k, ids, w);
    if (E <= 128) return launch_pdl(route_kernel<4>, blocks, threads, 0, stream, logits, T, E, k, ids, w);
    if (E <= 256) return launch_pdl(route_kernel<8>, blocks, threads, 0, stream, logits, T, E, k, ids, w);
    if (E <= 512) return launch_pdl(route_kernel<16>, blocks, threads, 0, stream, logits, T, E, k, ids, w);
    return launch_pdl(route_kernel<32>, blocks, threads, 0, stream, logits, T, E, k, ids, w);
}

}  // namespace moe
