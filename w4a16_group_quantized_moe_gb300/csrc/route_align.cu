// route_align.cu -- steps 1 and 2 in one launch for small batches.
//
// At decode size both steps are a chain of short dependent phases, and a
// kernel launch plus a global-memory round trip between them costs more
// than either step.  One CTA routes every token (one warp per token, the
// router of route.cuh) into shared memory as well as to the outputs, then
// groups the pairs with the block routine of align.cuh reading the ids from
// shared memory.  The outputs are exactly those of moe_topk_route followed
// by moe_align_offsets.
#include "align.cuh"
#include "route.cuh"

namespace moe {

constexpr int kFusedMaxT = 32;

template <int PER>
__global__ void route_align_kernel(const float *__restrict__ logits, int T, int E, int k, int WS,
                                   int32_t *__restrict__ topk_ids, float *__restrict__ topk_w,
                                   int32_t *__restrict__ expert_offsets,
                                   int32_t *__restrict__ sorted_pair,
                                   int32_t *__restrict__ active_experts,
                                   int32_t *__restrict__ num_active, uint32_t *err) {
    extern __shared__ int sm[];
    int *s_ids = sm;                        // [T*k]
    int *s_align = sm + ((T * k + 31) & ~31);
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5;
    if (warp < T) route_token<PER>(logits + (size_t)warp * E, E, k, warp, topk_ids, topk_w, s_ids);
    __syncthreads();
    align_block(s_ids, T * k, E, WS, expert_offsets, sorted_pair, active_experts, num_active, err,
                s_align);
}

bool route_align_fusable(int T, int E, int k, size_t smem_limit) {
    const int P = T * k, WS = align_slices(P);
    return T >= 1 && T <= kFusedMaxT && 32 * T <= 1024 &&
           (((size_t)(P + 31) & ~(size_t)31) + align_smem_ints(WS, E)) * sizeof(int) <= smem_limit;
}

cudaError_t launch_route_align(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                               int32_t *offsets, int32_t *sorted_pair, int32_t *active,
                               int32_t *num_active, uint32_t *err, cudaStream_t stream) {
    const int P = T * k, WS = align_slices(P);
    const size_t smem = (((size_t)(P + 31) & ~(size_t)31) + align_smem_ints(WS, E)) * sizeof(int);
    int threads = align_threads(WS, E);
    if (threads < 32 * T) threads = 32 * T;
    static int configured[5][128];
#define MOE_RA(PER, IDX)                                                                         \
    do {                                                                                         \
        cudaError_t e = ensure_smem(route_align_kernel<PER>, configured[IDX], smem);             \
        if (e != cudaSuccess) return e;                                                          \
        return launch_pdl(route_align_kernel<PER>, 1, threads, smem, stream, logits, T, E, k, WS, \
                          ids, w, offsets, sorted_pair, active, num_active, err);                \
    } while (0)
    if (E <= 64) MOE_RA(2, 0);
    if (E <= 128) MOE_RA(4, 1);
    if (E <= 256) MOE_RA(8, 2);
    if (E <= 512) MOE_RA(16, 3);
    MOE_RA(32, 4);
#undef MOE_RA
}

}  // namespace moe
