// align.cu -- step 2: active-expert segments.  "Multi-row active-expert
// segments and offsets-based scheduling" ("[Perf][SM70] Narrow Qwen3.8 AWQ
// active grouped decode", section Purpose): the P = T*k token-expert pairs
// are grouped by expert with a stable counting sort, and the list of experts
// that received any pair is compacted.
//
// One CTA of W warps.  Pair ids are split into W contiguous slices, one per
// warp, so that walking slices in warp order walks pairs in id order:
//   1. per-warp histograms hist[w][e] (shared-memory atomics);
//   2. per expert, the counts are turned into per-warp starting cursors
//      (exclusive prefix over w) and a total;
//   3. a block-wide exclusive scan of the totals gives expert_offsets, and a
//      scan of (total > 0) gives each active expert's slot;
//   4. each warp re-walks its slice 32 pairs at a time; lanes with the same
//      expert find their rank among themselves with __match_any_sync, so the
//      scatter keeps pair-id order inside every segment.
#include "common.cuh"

namespace moe {

// Block-wide exclusive scan of two int arrays of length n held in shared
// memory (in place).  Returns the totals.  Every thread must call it.
__device__ int2 block_exclusive_scan2(int *a, int *b, int n, int *scratch) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int nw = nt >> 5;
    const int per = (n + nt - 1) / nt;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int sa = 0, sb = 0;
    for (int i = lo; i < hi; ++i) {
        sa += a[i];
        sb += b[i];
    }
    // inclusive warp scan of the thread sums
    int ia = sa, ib = sb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int ta = __shfl_up_sync(0xffffffffu, ia, off);
        const int tb = __shfl_up_sync(0xffffffffu, ib, off);
        if (lane >= off) {
            ia += ta;
            ib += tb;
        }
    }
    if (lane == 31) {
        scratch[2 * warp] = ia;
        scratch[2 * warp + 1] = ib;
    }
    __syncthreads();
    if (warp == 0) {
        int wa = lane < nw ? scratch[2 * lane] : 0;
        int wb = lane < nw ? scratch[2 * lane + 1] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int ta = __shfl_up_sync(0xffffffffu, wa, off);
            const int tb = __shfl_up_sync(0xffffffffu, wb, off);
            if (lane >= off) {
                wa += ta;
                wb += tb;
            }
        }
        if (lane < nw) {
            scratch[64 + 2 * lane] = wa;  // inclusive warp prefix
            scratch[64 + 2 * lane + 1] = wb;
        }
    }
    __syncthreads();
    const int wpa = warp ? scratch[64 + 2 * (warp - 1)] : 0;
    const int wpb = warp ? scratch[64 + 2 * (warp - 1) + 1] : 0;
    int ra = wpa + ia - sa, rb = wpb + ib - sb;  // exclusive prefix of this thread
    for (int i = lo; i < hi; ++i) {
        const int va = a[i], vb = b[i];
        a[i] = ra;
        b[i] = rb;
        ra += va;
        rb += vb;
    }
    const int2 tot = make_int2(scratch[64 + 2 * (nw - 1)], scratch[64 + 2 * (nw - 1) + 1]);
    __syncthreads();
    return tot;
}

__global__ void align_kernel(const int32_t *__restrict__ topk_ids, int P, int E,
                             int32_t *__restrict__ expert_offsets,
                             int32_t *__restrict__ sorted_pair,
                             int32_t *__restrict__ active_experts,
                             int32_t *__restrict__ num_active, uint32_t *err) {
    extern __shared__ int sm[];
    const int W = blockDim.x >> 5;
    int *hist = sm;                 // [W][E]
    int *offs = hist + W * E;       // [E]  counts -> exclusive offsets
    int *slot = offs + E;           // [E]  active flags -> active slots
    int *scratch = slot + E;        // [128]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    pdl_wait();
    pdl_trigger();
    for (int i = tid; i < W * E; i += blockDim.x) hist[i] = 0;
    __syncthreads();

    const int lo = (int)((long long)P * warp / W), hi = (int)((long long)P * (warp + 1) / W);
    bool bad = false;
    for (int p = lo + lane; p < hi; p += 32) {
        const int e = topk_ids[p];
        if (e >= 0 && e < E)
            atomicAdd(&hist[warp * E + e], 1);
        else
            bad = true;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, MOE_DEVERR_BAD_EXPERT_ID);
    __syncthreads();

    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < W; ++w) {
            const int c = hist[w * E + e];
            hist[w * E + e] = run;
            run += c;
        }
        offs[e] = run;
        slot[e] = run > 0;
    }
    __syncthreads();
    // counts are read back from the cursors' totals after the scan, so keep them
    const int2 tot = block_exclusive_scan2(offs, slot, E, scratch);
    const int total = tot.x, nact = tot.y;

    for (int e = tid; e < E; e += blockDim.x) {
        expert_offsets[e] = offs[e];
        const int next = (e + 1 < E) ? offs[e + 1] : total;
        if (next > offs[e]) active_experts[slot[e]] = e;
    }
    for (int a = nact + tid; a < E; a += blockDim.x) active_experts[a] = -1;
    if (tid == 0) {
        expert_offsets[E] = total;
        num_active[0] = nact;
    }

    // stable scatter: warps in slice order, lanes in pair order
    for (int base = lo; base < hi; base += 32) {
        const int p = base + lane;
        int e = (p < hi) ? topk_ids[p] : -1;
        const bool ok = (p < hi) && e >= 0 && e < E;
        if (!ok) e = -1 - lane;  // unique key: matches only itself
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & ((1u << lane) - 1u));
        int cur = 0;
        if (ok) {
            cur = hist[warp * E + e];
            sorted_pair[offs[e] + cur + rank] = p;
        }
        __syncwarp();
        if (ok && lane == 31 - __clz(same)) hist[warp * E + e] = cur + __popc(same);
        __syncwarp();
    }
    // pairs with bad ids leave holes at the end; mark them
    for (int r = total + tid; r < P; r += blockDim.x) sorted_pair[r] = -1;
}

size_t align_smem_bytes(int W, int E) { return sizeof(int) * ((size_t)W * E + 2 * E + 128); }

int align_warps(int P, int E, size_t smem_limit) {
    int W = (P + 255) / 256;
    W = W < 1 ? 1 : (W > 32 ? 32 : W);
    while (W > 1 && align_smem_bytes(W, E) > smem_limit) --W;
    return W;
}

cudaError_t launch_align(const int32_t *ids, int P, int E, int32_t *offsets, int32_t *sorted_pair,
                         int32_t *active, int32_t *num_active, uint32_t *err, size_t smem_limit,
                         cudaStream_t stream) {
    const int W = align_warps(P, E, smem_limit);
    const size_t smem = align_smem_bytes(W, E);
    static int configured[128];
    cudaError_t e = ensure_smem(align_kernel, configured, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(align_kernel, 1, W * 32, smem, stream, ids, P, E, offsets, sorted_pair, active,
                      num_active, err);
}

}  // namespace moe
