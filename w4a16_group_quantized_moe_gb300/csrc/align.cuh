// align.cuh -- the grouping step as a block-level routine shared by the
// grouping kernels; see align.cu for the method.
#pragma once
#include "common.cuh"

namespace moe {

// Block-wide exclusive scan of two int arrays of length n held in shared
// memory (in place).  Returns the totals.  Every thread must call it.
__device__ __forceinline__ int2 block_exclusive_scan2(int *a, int *b, int n, int *scratch) {
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

// Shared ints needed by align_block: WS per-slice histograms of E experts,
// offsets and slots of E experts, scan scratch.
__host__ __device__ inline size_t align_smem_ints(int WS, int E) { return (size_t)WS * E + 2 * E + 128; }

// Groups the P pairs whose expert ids are ids[0..P) (global or shared
// memory).  Every thread of the block calls it; WS (<= warps of the block)
// warps scatter, one contiguous slice of pairs each; the other loops are
// spread over all threads.
__device__ __forceinline__ void align_block(const int32_t *ids, int P, int E, int WS,
                                            int32_t *__restrict__ expert_offsets,
                                            int32_t *__restrict__ sorted_pair,
                                            int32_t *__restrict__ active_experts,
                                            int32_t *__restrict__ num_active, uint32_t *err, int *sm) {
    int *hist = sm;                 // [WS][E]
    int *offs = hist + WS * E;      // [E]  counts -> exclusive offsets
    int *slot = offs + E;           // [E]  active flags -> active slots
    int *scratch = slot + E;        // [128]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;

    for (int i = tid; i < WS * E; i += nt) hist[i] = 0;
    __syncthreads();

    const int lo = warp < WS ? (int)((long long)P * warp / WS) : 0;
    const int hi = warp < WS ? (int)((long long)P * (warp + 1) / WS) : 0;
    constexpr int kBatch = 8;  // rounds of 32 ids loaded before any is used
    bool bad = false;
    for (int base = lo; base < hi; base += 32 * kBatch) {
        int ev[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int p = base + 32 * u + lane;
            ev[u] = p < hi ? ids[p] : 0;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (base + 32 * u + lane >= hi) continue;
            const int e = ev[u];
            if (e >= 0 && e < E)
                atomicAdd(&hist[warp * E + e], 1);
            else
                bad = true;
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, MOE_DEVERR_BAD_EXPERT_ID);
    __syncthreads();

    for (int e = tid; e < E; e += nt) {
        int run = 0;
        for (int w = 0; w < WS; ++w) {
            const int c = hist[w * E + e];
            hist[w * E + e] = run;
            run += c;
        }
        offs[e] = run;
        slot[e] = run > 0;
    }
    __syncthreads();
    const int2 tot = block_exclusive_scan2(offs, slot, E, scratch);
    const int total = tot.x, nact = tot.y;

    for (int e = tid; e < E; e += nt) {
        expert_offsets[e] = offs[e];
        const int next = (e + 1 < E) ? offs[e + 1] : total;
        if (next > offs[e]) active_experts[slot[e]] = e;
    }
    for (int a = nact + tid; a < E; a += nt) active_experts[a] = -1;
    if (tid == 0) {
        expert_offsets[E] = total;
        num_active[0] = nact;
    }

    // stable scatter: warps in slice order, lanes in pair order
    const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;  // bits of an expert id
    if (warp < WS) {
        for (int b0 = lo; b0 < hi; b0 += 32 * kBatch) {
            int ev[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int p = b0 + 32 * u + lane;
                ev[u] = p < hi ? ids[p] : -1;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int base = b0 + 32 * u;
                if (base >= hi) break;  // warp-uniform
                const int p = base + lane;
                int e = ev[u];
                const bool ok = (p < hi) && e >= 0 && e < E;
                // lanes holding the same expert: valid lanes agreeing on every
                // bit of the id (one ballot per bit; cheaper than a match)
                unsigned same = __ballot_sync(0xffffffffu, ok);
                for (int bit = 0; bit < nbits; ++bit) {
                    const bool v = (e >> bit) & 1;
                    const unsigned bm = __ballot_sync(0xffffffffu, v);
                    same &= v ? bm : ~bm;
                }
                if (!ok) same = 1u << lane;
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
        }
    }
    // pairs with bad ids leave holes at the end; mark them
    for (int r = total + tid; r < P; r += nt) sorted_pair[r] = -1;
}

// Scatter slices for P pairs: one warp per 256 pairs, 1..32.
__host__ __device__ inline int align_slices(int P) {
    int W = (P + 255) / 256;
    return W < 1 ? 1 : (W > 32 ? 32 : W);
}

// Threads of a grouping block: enough for the slices and for one expert each.
__host__ __device__ inline int align_threads(int WS, int E) {
    int n = 32 * WS;
    const int e32 = ((E < 1024 ? E : 1024) + 31) / 32 * 32;
    return n > e32 ? n : e32;
}

}  // namespace moe
