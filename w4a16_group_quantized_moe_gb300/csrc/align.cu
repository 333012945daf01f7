// align.cu -- step 2: active-expert segments.  "Multi-row active-expert
// segments and offsets-based scheduling" ("[Perf][SM70] Narrow Qwen3.8 AWQ
// active grouped decode", section Purpose): the P = T*k token-expert pairs
// are grouped by expert with a stable counting sort, and the list of experts
// that received any pair is compacted.
//
// One CTA.  Pair ids are split into WS contiguous slices, one per scatter
// warp, so that walking slices in warp order walks pairs in id order:
//   1. per-slice histograms hist[w][e] (shared-memory atomics);
//   2. per expert (one thread each), the counts become per-slice starting
//      cursors (exclusive prefix over w) and a total;
//   3. a block-wide exclusive scan of the totals gives expert_offsets, and a
//      scan of (total > 0) gives each active expert's slot;
//   4. each scatter warp re-walks its slice 32 pairs at a time; lanes with the
//      same expert find their rank among themselves (ballots over the id bits), so
//      the scatter keeps pair-id order inside every segment.
#include "align.cuh"

namespace moe {

__global__ void align_kernel(const int32_t *__restrict__ topk_ids, int P, int E, int WS,
                             int32_t *__restrict__ expert_offsets,
                             int32_t *__restrict__ sorted_pair,
                             int32_t *__restrict__ active_experts,
                             int32_t *__restrict__ num_active, uint32_t *err) {
    extern __shared__ int sm[];
    pdl_wait();
    pdl_trigger();
    align_block(topk_ids, P, E, WS, expert_offsets, sorted_pair, active_experts, num_active, err, sm);
}

cudaError_t launch_align(const int32_t *ids, int P, int E, int32_t *offsets, int32_t *sorted_pair,
                         int32_t *active, int32_t *num_active, uint32_t *err, size_t smem_limit,
                         cudaStream_t stream) {
    int WS = align_slices(P);
    while (WS > 1 && align_smem_ints(WS, E) * sizeof(int) > smem_limit) --WS;
    const size_t smem = align_smem_ints(WS, E) * sizeof(int);
    static int configured[128];
    cudaError_t e = ensure_smem(align_kernel, configured, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(align_kernel, 1, align_threads(WS, E), smem, stream, ids, P, E, WS, offsets,
                      sorted_pair, active, num_active, err);
}

}  // namespace moe
