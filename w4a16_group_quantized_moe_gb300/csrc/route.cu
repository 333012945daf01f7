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
#include "route.cuh"

namespace moe {

constexpr int kRouteWarpsPerBlock = 4;

template <int PER>
__global__ void __launch_bounds__(kRouteWarpsPerBlock * 32)
route_kernel(const float *__restrict__ logits, int T, int E, int k,
             int32_t *__restrict__ topk_ids, float *__restrict__ topk_w) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * kRouteWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= T) return;
    route_token<PER>(logits + (size_t)t * E, E, k, t, topk_ids, topk_w, nullptr);
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
