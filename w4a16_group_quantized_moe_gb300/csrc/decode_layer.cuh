// decode_layer.cuh -- the whole layer for decode batches (T <= 8) in one
// cooperative launch: routing, grouping, gate/up + SiLU, down and the
// weighted combine.  The kernel template lives in this header so that its
// instantiations compile in separate translation units (decode_layer_*.cu);
// decode_layer.cu plans and dispatches the launch.
//
// At decode size the layer streams a few tens of megabytes of packed
// weights, a few microseconds of HBM time, while each step boundary of the
// four-call path costs a launch, a global round trip for the step's inputs
// and a ramp-up of the weight stream.  Here every CTA (one per SM, all
// resident) does the following, and the only waits between CTAs are the two
// true data dependencies of the method:
//
//  1. Routes every token itself (the router of route.cuh, one warp per
//     token, from the fp32 logits) and groups the T*k pairs by expert in
//     shared memory, one thread per pair.  The routing of "Sparse MoE
//     layer" (softmax, top-k, renormalised) and the grouping into
//     active-expert segments with offsets of "Active grouped decode" are
//     recomputed per CTA: that is cheaper than publishing them.
//  2. Takes a contiguous share of the gate/up tasks (RT1 row pairs of one
//     active expert) and of the down tasks (RT2 rows), dealt over its warps.
//     Each warp streams its task sequence through its own two-slot ring of
//     bulk-copy buffers, so down weights are already in flight while the
//     gate/up tasks finish.
//  3. Gate/up writes h = silu(gate) * up of every pair of the expert's
//     segment to the workspace, already in the pair-interleaved shared-cache
//     layout, and counts finished row pairs per expert.  Between the two
//     steps each CTA publishes its counts (one fence) and waits only for the
//     experts its own down tasks read, then copies those h rows into shared
//     memory.
//  4. Down writes each pair's fp32 projection and counts rows per 8-row
//     output block; whichever CTA completes a block sums its k terms per
//     token in order (deterministic) and writes fp16.
//
// Every cross-CTA wait is bounded: on expiry it sets MOE_DEVERR_WAIT_TIMEOUT
// in the error word and the kernel finishes without the dependent work.  The
// workspace's diagnostic words set the wait limit and an offset added to the
// wait targets (so that a test can make the waits run out), and can switch
// on a timeline of global-timer stamps of the kernel's phases.
// The last CTA to leave resets the per-expert counters, so consecutive calls
// on one stream share a workspace without clearing it.
#pragma once
#include "decode_common.cuh"
#include "route.cuh"

namespace moe {

constexpr int kLayerMaxWarps = 16;
constexpr int kLayerMinWarps = 8;
constexpr int kLayerMaxT = 8;
constexpr int kLayerMaxPairs = 256;
constexpr int kLayerSlots = 2;  // task buffers per warp
constexpr int kLayerRoutePer = 32;  // logits per lane in the router (E <= 1024)
constexpr uint32_t kPollTries = 1u << 20;  // bounded wait (about a second) for other CTAs

// Stamps of the optional phase timeline (8 per CTA, global timer, ns).
enum { kLtEntry = 0, kLtGrouped, kLtFirstIssue, kLtFirstLanded, kLtGateUpDone, kLtDownReady, kLtDownDone, kLtExit };

// Named barriers of the pair-segment path (0 is __syncthreads): the staging
// warps' hand-off of the x rows to the routing warps, and the staging warps'
// own barrier.
enum { kBarXReady = 1, kBarStagers = 2 };

struct LayerArgs {
    const float *logits;  // [T][E]
    const __half *x;      // [T][H]
    const uint32_t *q13;  // gate/up packed codes  [E][2I][H/8]
    const __half *s13;    //                scales [E][2I][H/32]
    const uint32_t *z13;  //                zeros  [E][2I/8][H/32]
    const uint32_t *q2;   // down packed codes     [E][H][I/8]
    const __half *s2;     //                scales [E][H][I/32]
    const uint32_t *z2;   //                zeros  [E][H/8][I/32]
    int T, E, k, H, I, P;
    int32_t *topk_ids;    // [T][k] (written by CTA 0)
    float *topk_w;        // [T][k] (written by CTA 0)
    __half *out;          // [T][H]
    __half *h;            // workspace [P][I], sorted rows, cache layout
    float *y;             // workspace [P][H]
    uint32_t *blkctr;     // workspace [H/8]
    uint32_t *done;       // workspace [P]: finished gate/up row pairs per active slot
    uint32_t *exitctr;    // workspace [1]
    uint32_t *err;
    int nw;               // warps per CTA
    int hrows;            // h rows the shared cache holds
    uint32_t slot_bytes;  // one task buffer
    int pair_mode;        // 1: one-row segment per pair, in pair order (see the kernel)
};

// Shared memory: meta ints (ids, weights, sorted pairs, active experts,
// segment bounds, per-expert counts, grouping scratch, misc), per-block row
// counts and completed-block list, the activation cache (x rows in step 3,
// h rows in step 4), the per-warp rings and their mbarriers.
struct LayerLayout {
    uint32_t meta, blk, cache, ring, bars, total;
};

__host__ __device__ inline LayerLayout layer_layout(int T, int H, int I, int P, int hrows, int nw,
                                                    uint32_t slot_bytes) {
    LayerLayout L;
    L.meta = 0;
    L.blk = (uint32_t)align_up((size_t)(11 * P + 8) * 4, 128);
    L.cache = L.blk + (uint32_t)align_up((size_t)(H / 8) * 4, 128);
    const size_t xc = (size_t)T * H * 2, hc = (size_t)hrows * I * 2;
    L.ring = L.cache + (uint32_t)align_up(xc > hc ? xc : hc, 128);
    L.bars = L.ring + (uint32_t)nw * kLayerSlots * slot_bytes;
    L.total = L.bars + (uint32_t)(nw * kLayerSlots + kLayerMaxT) * 8;  // + one per routing warp
    return L;
}

// Index of h[row][i] within a row of the cache layout (dec_xoff with the
// pair interleave of each 8-element block: [a0 a4 a1 a5 a2 a6 a3 a7]).
__device__ __forceinline__ int h_cache_index(int i, int G) {
    const int kb = i >> 3, j = i & 7;
    return ((kb & 3) * G + (kb >> 2)) * 8 + (j < 4 ? 2 * j : 2 * (j - 4) + 1);
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Gate/up end of a token pass: reduce over the L lanes of each row pair and
// write h = silu(g) * u for the pass's rows (cache layout, sorted rows).
template <int L, int NT>
__device__ __forceinline__ void layer_finish_gate_up(float (&acc)[1][2][kDecPass], const Cursor &c,
                                                     const LayerArgs &a, int G2, int lane) {
    const int ks = lane % L, us = lane / L;
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int off = L / 2; off > 0; off >>= 1)
                acc[0][b][t] += __shfl_xor_sync(0xffffffffu, acc[0][b][t], off);
    const int lr = us;
    const int unit = c.unit0 + lr;
    const int hi = h_cache_index(unit, G2);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int r = c.r0 + c.tb + t;
        if (lr < c.cnt && (t % L) == ks) {
            const float gv = acc[0][0][t], uv = acc[0][1][t];
            const float hv = gv / (1.0f + __expf(-gv)) * uv;
            a.h[(size_t)r * a.I + hi] = __float2half_rn(hv);
        }
    }
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int t = 0; t < kDecPass; ++t) acc[0][b][t] = 0.f;
}

// Down end of a token pass: reduce and write y[pair][row] in fp32.
template <int L, int NT>
__device__ __forceinline__ void layer_finish_down(float (&acc)[2][1][kDecPass], const Cursor &c,
                                                  const int *s_pairs, const LayerArgs &a, int lane) {
    using Tr = DecTraits<kDecDown, L, 2>;
    const int ks = lane % L, us = lane / L;
#pragma unroll
    for (int ru = 0; ru < 2; ++ru)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int off = L / 2; off > 0; off >>= 1)
                acc[ru][0][t] += __shfl_xor_sync(0xffffffffu, acc[ru][0][t], off);
#pragma unroll
    for (int ru = 0; ru < 2; ++ru) {
        const int lr = us + ru * Tr::UPW;
        const int unit = c.unit0 + lr;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int p = s_pairs[c.r0 + c.tb + t];
            if (lr < c.cnt && (t % L) == ks) a.y[(size_t)p * a.H + unit] = acc[ru][0][t];
        }
    }
#pragma unroll
    for (int ru = 0; ru < 2; ++ru)
#pragma unroll
        for (int t = 0; t < kDecPass; ++t) acc[ru][0][t] = 0.f;
}

// Position of a task in one of the two flat task lists (expert-major): the
// active slot and the task's index within that expert.
struct TaskPos {
    int ai, li;
};

// Advances a position by `step` tasks in a list of tpe tasks per expert.
__device__ __forceinline__ void task_advance(TaskPos &p, int step, int tpe) {
    p.li += step;
    while (p.li >= tpe) {
        p.li -= tpe;
        ++p.ai;
    }
}

// First task of a CTA's share: tasks are weighted by (1 + rows of their
// expert's segment), the dequantisation being worth about one row of
// products (measured on the Qwen4Exp geometry at 8 tokens: 79.0 us per
// layer against 81.9 with 2 + rows, 81.4 with rows alone, 84.9 with
// 4 + rows), and CTA c owns the tasks whose weighted start lies in
// [c W / NC, (c+1) W / NC).  The weighted start of expert a's first task is
// tpe * (a + lo[a]) (lo: first sorted row of the segment).
__device__ __forceinline__ void share_start(long long w, int A, int tpe, const int *s_lo, const int *s_hi,
                                            int *s_out, int tid, int nth) {
    for (int a = tid; a < A; a += nth) {
        const long long pa = (long long)tpe * (a + s_lo[a]);
        const long long pn = (long long)tpe * (a + 1 + s_hi[a]);
        if (pa <= w && w < pn) {
            const long long cost = 1 + s_hi[a] - s_lo[a];
            *s_out = a * tpe + (int)((w - pa + cost - 1) / cost);
        }
    }
}

template <int L1, int GT1, int L2, int GT2, int FMT, bool PAIRS>
__global__ void __launch_bounds__(kLayerMaxWarps * 32, 1) decode_layer_kernel(const LayerArgs a) {
    using T1 = DecTraits<kDecGateUp, L1, 1>;
    using T2 = DecTraits<kDecDown, L2, 2>;
    constexpr int RT1 = T1::RT, RT2 = T2::RT;
    extern __shared__ __align__(128) uint8_t smem[];
    const int NW = a.nw, NTH = NW * 32;
    const int G1 = GT1 ? GT1 : a.H / 32, G2 = GT2 ? GT2 : a.I / 32;
    const int H = 32 * G1, I = 32 * G2, P = a.P, k = a.k;
    const int nblk = H / 8;
    const LayerLayout Ly = layer_layout(a.T, H, I, P, a.hrows, NW, a.slot_bytes);
    int *s_ids = reinterpret_cast<int *>(smem + Ly.meta);
    float *s_w = reinterpret_cast<float *>(s_ids + P);
    int *s_pairs = reinterpret_cast<int *>(s_w + P);
    int *s_act = s_pairs + P;   // [A] active experts, ascending
    int *s_lo = s_act + P;      // [A] first sorted row of the segment
    int *s_hi = s_lo + P;       // [A] one past its last row
    int *s_cnt1 = s_hi + P;     // [A] gate/up row pairs this CTA finished
    int *g_less = s_cnt1 + P;   // grouping scratch per pair
    int *g_same = g_less + P;
    int *g_first = g_same + P;
    int *s_tok = g_first + P;   // token of each sorted row
    volatile int *s_misc = s_tok + P;  // [0] A, [2] h not ready, [3] give up, [4..7] share bounds
    int *s_blk = reinterpret_cast<int *>(smem + Ly.blk);  // [nblk] rows counted per output block
    uint8_t *cache = smem + Ly.cache;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t *ring = smem + Ly.ring + (size_t)warp * kLayerSlots * a.slot_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Ly.bars) + warp * kLayerSlots;
    // the routing warp's logits copy (warps < T)
    uint64_t *lbar = reinterpret_cast<uint64_t *>(smem + Ly.bars) + NW * kLayerSlots + (warp & (kLayerMaxT - 1));
    const WarpGeom wg1 = warp_geom(RT1, 2, H), wg2 = warp_geom(RT2, 1, I);
    const int cta = blockIdx.x, NC = gridDim.x;

    // diagnostics of the control block: wait limit, wait-target offset, timeline
    const uint64_t t_entry = global_timer_ns();
    const uint32_t polls = a.err[kCtrlWaitPolls] ? a.err[kCtrlWaitPolls] : kPollTries;
    const uint32_t extra = a.err[kCtrlWaitExtra];
    uint64_t *tl = reinterpret_cast<uint64_t *>(
        *reinterpret_cast<const unsigned long long *>(a.err + kCtrlTimeline));
    auto stamp = [&](int i) {
        if (tl) tl[cta * 8 + i] = global_timer_ns();
    };
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kLayerSlots; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    for (int i = tid; i < nblk; i += NTH) s_blk[i] = 0;
    for (int i = tid; i < P; i += NTH) s_cnt1[i] = 0;
    if (tid < 8) s_misc[tid] = 0;
    pdl_wait();
    pdl_trigger();

    // Pair segments (a.pair_mode; always with one token, where it changes
    // nothing else): every pair p = t*k + j is its own one-row segment, in
    // pair order, even when two tokens chose the same expert (that expert's
    // weights are then streamed once per pair).  Every CTA's task shares then
    // follow from P alone, each routing warp publishes its token's ranks as
    // its rounds decide them, and the other warps compute their shares
    // meanwhile and issue each task's copies as soon as its pair is ranked.
    // h, y and the combine are indexed by pair, so the arithmetic per pair is
    // that of the grouped path.
    constexpr bool one = PAIRS;  // a separate instantiation: the grouped path carries none of it
    volatile int *s_ranked = g_less;  // [T] ranks published per token (pair segments)
    int A, b1, e1, b2, e2;
    const int TPE1 = (I + RT1 - 1) / RT1, TPE2 = (H + RT2 - 1) / RT2;
    if (one) {
        A = P;
        for (int t = tid; t < a.T; t += NTH) s_ranked[t] = 0;
        __syncthreads();  // the zeroed counters are visible before anyone polls them
        if (warp < a.T) {
            if (lane < k) {
                const int p = warp * k + lane;
                s_lo[p] = p;
                s_hi[p] = p + 1;
                s_pairs[p] = p;
                s_tok[p] = warp;
            }
            const bool lead = cta == 0;
            route_token_compact(a.logits + (size_t)warp * a.E, a.E, k, warp, lead ? a.topk_ids : nullptr,
                                lead ? a.topk_w : nullptr, s_ids, s_w, reinterpret_cast<uint32_t *>(ring),
                                s_act + warp * k, s_ranked + warp, lbar);
        } else {
            dec_stage_rows(a.x, a.T, H, G1, cache, tid - 32 * a.T, NTH - 32 * a.T);
            named_barrier_arrive(kBarXReady, NTH);        // the routing warps sync on it later
            named_barrier(kBarStagers, NTH - 32 * a.T);   // x visible to every staging warp
        }
        // shares: A = P one-row segments, every task weighs 3, segment p's
        // tasks start at weight 3 p tpe (the closed form of share_start)
        auto share1 = [&](long long w, int tpe) {
            const long long a3 = 3LL * tpe;
            const int ax = (int)(w / a3);
            return ax * tpe + (int)((w - ax * a3 + 2) / 3);
        };
        const long long W1 = 3LL * TPE1 * P, W2 = 3LL * TPE2 * P;
        b1 = share1(W1 * cta / NC, TPE1);
        e1 = cta + 1 < NC ? share1(W1 * (cta + 1) / NC, TPE1) : P * TPE1;
        b2 = share1(W2 * cta / NC, TPE2);
        e2 = cta + 1 < NC ? share1(W2 * (cta + 1) / NC, TPE2) : P * TPE2;
        if (tid == 0 && tl) {
            tl[cta * 8 + kLtEntry] = t_entry;
            stamp(kLtGrouped);
        }
    } else {
        // ---- 1. route (warps < T) while the other warps stage the x rows
        if (warp < a.T) {
            const bool lead = cta == 0;
            const float *row = a.logits + (size_t)warp * a.E;
            int32_t *ids = lead ? a.topk_ids : nullptr;
            float *w = lead ? a.topk_w : nullptr;
            // keys in this warp's task ring, which no copy has touched yet
            route_token_compact(row, a.E, k, warp, ids, w, s_ids, s_w, reinterpret_cast<uint32_t *>(ring), nullptr,
                                nullptr, lbar);
        } else if (NTH > 32 * a.T) {  // the host keeps NW > T
            dec_stage_rows(a.x, a.T, H, G1, cache, tid - 32 * a.T, NTH - 32 * a.T);
        }
        __syncthreads();

        // ---- group the pairs: rank of pair p = #(expert < e) + #(earlier pairs of e)
        for (int p = tid; p < P; p += NTH) {
            const int e = s_ids[p];
            int less = 0, same = 0, before = 0;
            for (int q = 0; q < P; ++q) {
                const int f = s_ids[q];
                less += f < e;
                same += f == e;
                before += (f == e) & (q < p);
            }
            s_pairs[less + before] = p;
            s_tok[less + before] = p / k;
            g_less[p] = less;
            g_same[p] = same;
            g_first[p] = before == 0;
            if (before == 0) atomicAdd(const_cast<int *>(&s_misc[0]), 1);
        }
        __syncthreads();
        for (int p = tid; p < P; p += NTH) {
            if (!g_first[p]) continue;
            const int e = s_ids[p];
            int slot = 0;
            for (int q = 0; q < P; ++q) slot += g_first[q] & (s_ids[q] < e);
            s_act[slot] = e;
            s_lo[slot] = g_less[p];
            s_hi[slot] = g_less[p] + g_same[p];
        }
        __syncthreads();

        if (tid == 0 && tl) {
            tl[cta * 8 + kLtEntry] = t_entry;
            stamp(kLtGrouped);
        }

        // ---- 2. this CTA's shares of both task lists (weighted, contiguous)
        A = s_misc[0];
        {
            const long long W1 = (long long)TPE1 * (A + P), W2 = (long long)TPE2 * (A + P);
            if (tid == 0) {
                s_misc[4] = 0; s_misc[5] = A * TPE1; s_misc[6] = 0; s_misc[7] = A * TPE2;
            }
            __syncthreads();
            int *sm = const_cast<int *>(s_misc);
            share_start(W1 * cta / NC, A, TPE1, s_lo, s_hi, sm + 4, tid, NTH);
            if (cta + 1 < NC) share_start(W1 * (cta + 1) / NC, A, TPE1, s_lo, s_hi, sm + 5, tid, NTH);
            share_start(W2 * cta / NC, A, TPE2, s_lo, s_hi, sm + 6, tid, NTH);
            if (cta + 1 < NC) share_start(W2 * (cta + 1) / NC, A, TPE2, s_lo, s_hi, sm + 7, tid, NTH);
            __syncthreads();
        }
        b1 = s_misc[4]; e1 = s_misc[5]; b2 = s_misc[6]; e2 = s_misc[7];
    }
    // this warp's tasks: b1 + gw + i*gNW (i < n1), then b2 + warp + j*NW; with
    // pair segments the routing warps take no gate/up task (gw = warp - T
    // over the other NW - T warps), so no task waits for a router to finish
    const int gw = one ? warp - a.T : warp, gNW = one ? NW - a.T : NW;
    const int n1 = (gw >= 0 && e1 - b1 > gw) ? (e1 - b1 - gw + gNW - 1) / gNW : 0;
    const int n2 = e2 - b2 > warp ? (e2 - b2 - warp + NW - 1) / NW : 0;
    const int ntask = n1 + n2;

    // positions of the next task to issue and of the two tasks in the slots
    int iss = 0;
    TaskPos ip{gw >= 0 ? (b1 + gw) / TPE1 : 0, gw >= 0 ? (b1 + gw) % TPE1 : 0};
    if (n1 == 0) ip = TaskPos{(b2 + warp) / TPE2, (b2 + warp) % TPE2};
    TaskPos q0{0, 0}, q1{0, 0};  // tasks in flight, oldest first

    auto make_cursor = [&](const TaskPos &tp, bool gate, Cursor &cu) {
        const int rt = gate ? RT1 : RT2, rows = gate ? I : H;
        cu.unit0 = tp.li * rt;
        cu.cnt = min(rt, rows - cu.unit0);
        cu.e = s_act[tp.ai];
        cu.r0 = s_lo[tp.ai];
        cu.ne = s_hi[tp.ai] - cu.r0;
        cu.tb = 0;
    };
    // fetch task `iss` (position ip) into slot iss % 2, then advance ip.
    // Lane 0 posts the expected bytes; lanes 0-5 (gate/up: codes, scales,
    // zeros of gate and up) or 0-2 (down) then issue one bulk copy each.
    bool dead = false;
    auto issue = [&]() {
        if (one) {
            // pair segments: this task's pair may still be being ranked
            const int pt = ip.ai / k, pj = ip.ai - pt * k;
            uint32_t it = 0;
            while (s_ranked[pt] <= pj && ++it < polls) __nanosleep(32);
            __threadfence_block();
            if (!__all_sync(0xffffffffu, it < polls)) {
                if (lane == 0) set_error(a.err, MOE_DEVERR_WAIT_TIMEOUT);
                dead = true;
                return;
            }
        }
        const bool gate = iss < n1;
        Cursor cu;
        make_cursor(ip, gate, cu);
        uint8_t *wb = ring + (size_t)(iss % kLayerSlots) * a.slot_bytes;
        uint64_t *bar = bars + iss % kLayerSlots;
        const int nmat = gate ? 2 : 1;
        const int N = gate ? 2 * I : H, K = gate ? H : I;
        const WarpGeom &wg = gate ? wg1 : wg2;
        const int b = lane % nmat, kind = lane / nmat;  // kind 0 codes, 1 scales, 2 zeros
        const WarpCopy cp = warp_copy(cu.e, cu.unit0 + b * I, cu.cnt, N, K);
        // NVFP4: no zero words (z13 / z2 hold the per-expert scales)
        const int nkind = FMT == kFmtNvfp4 ? 2 : 3;
        uint32_t tx = cp.q_len + cp.s_len + (FMT == kFmtNvfp4 ? 0u : cp.z_len);
        if (gate) tx += __shfl_xor_sync(0xffffffffu, tx, 1);
        if (lane == 0) mbar_arrive_expect_tx(bar, tx);
        __syncwarp();
        if (kind < nkind) {
            fence_proxy_async();  // this warp's earlier reads of the slot come first
            const uint8_t *src;
            uint32_t dst, len;
            if (kind == 0) {
                src = reinterpret_cast<const uint8_t *>(gate ? (const void *)a.q13 : (const void *)a.q2) + cp.q_off;
                dst = b * wg.q_bytes;
                len = cp.q_len;
            } else if (kind == 1) {
                src = reinterpret_cast<const uint8_t *>(gate ? (const void *)a.s13 : (const void *)a.s2) + cp.s_a;
                dst = nmat * wg.q_bytes + b * wg.s_bytes;
                len = cp.s_len;
            } else {
                src = reinterpret_cast<const uint8_t *>(gate ? (const void *)a.z13 : (const void *)a.z2) + cp.z_a;
                dst = nmat * (wg.q_bytes + wg.s_bytes) + b * wg.z_bytes;
                len = cp.z_len;
            }
            bulk_g2s(wb + dst, src, len, bar);
        }
        // record and advance (every lane keeps the same positions)
        if (iss == 0) q0 = ip; else q1 = ip;
        ++iss;
        if (iss == n1) ip = TaskPos{(b2 + warp) / TPE2, (b2 + warp) % TPE2};
        else task_advance(ip, iss < n1 ? gNW : NW, iss < n1 ? TPE1 : TPE2);
    };

    const int nfirst = ntask < kLayerSlots ? ntask : kLayerSlots;
    for (int i = 0; i < nfirst && !(one && dead); ++i) issue();
    if (tid == 0) stamp(kLtFirstIssue);
    if (one && warp < a.T) named_barrier(kBarXReady, NTH);  // routers compute after x is staged
    int consumed = 0;

    const TaskDims td1{2 * I, H, I, P, k}, td2{H, I, H, P, k};
    float acc1[1][2][kDecPass], acc2[2][1][kDecPass];
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int t = 0; t < kDecPass; ++t) acc1[0][b][t] = acc2[b][0][t] = 0.f;
    int hrow0 = 0;

    for (int i = 0; i <= ntask; ++i) {
        if (i == n1) {
            // ---- 3. between the steps (every warp passes here once)
            __syncthreads();  // this CTA's h values are written
            if (tid == 0) stamp(kLtGateUpDone);
            if (e1 > b1) {
                const int lo = b1 / TPE1, hi = (e1 - 1) / TPE1;
                for (int s = lo + tid; s <= hi; s += NTH) {
                    const int c = s_cnt1[s];
                    if (c) {
                        __threadfence();
                        atomicAdd(a.done + s, (unsigned)c);
                    }
                }
            }
            __syncthreads();
            if (e2 > b2) {
                const int lo = b2 / TPE2, hi = (e2 - 1) / TPE2;
                for (int s = lo + tid; s <= hi; s += NTH) {
                    uint32_t it = 0;
                    while (ld_acquire_u32(a.done + s) < (uint32_t)I + extra && ++it < polls) __nanosleep(64);
                    if (it >= polls) {
                        set_error(a.err, MOE_DEVERR_WAIT_TIMEOUT);
                        s_misc[2] = 1;
                    }
                }
            }
            __syncthreads();
            if (e2 > b2) {
                hrow0 = s_lo[b2 / TPE2];
                const int nh = s_hi[(e2 - 1) / TPE2] - hrow0;
                if (nh > a.hrows) {
                    if (tid == 0) {
                        set_error(a.err, MOE_DEVERR_BAD_METADATA);
                        s_misc[2] = 1;
                    }
                } else {
                    const uint4 *src = reinterpret_cast<const uint4 *>(a.h + (size_t)hrow0 * I);
                    uint4 *dst = reinterpret_cast<uint4 *>(cache);
                    const int nv = nh * I / 8;
                    for (int v = tid; v < nv; v += NTH) dst[v] = __ldcg(src + v);
                }
            }
            __syncthreads();
            if (tid == 0) stamp(kLtDownReady);
            if (s_misc[2]) dead = true;
        }
        if (i == ntask) break;
        if (dead) {  // a dead warp still passes the step boundary once
            if (i < n1) continue;
            break;
        }

        const int s = i % kLayerSlots;
        if (!mbar_wait_bounded(bars + s, (uint32_t)((i / kLayerSlots) & 1), nullptr)) {
            if (lane == 0) set_error(a.err, MOE_DEVERR_WAIT_TIMEOUT);
            dead = true;
            continue;
        }
        consumed = i + 1;
        if (i == 0 && tid == 0) stamp(kLtFirstLanded);
        const uint8_t *wb = ring + (size_t)s * a.slot_bytes;
        const TaskPos tp = q0;
        q0 = q1;
        Cursor cu;
        make_cursor(tp, i < n1, cu);
        const float gsc = FMT == kFmtNvfp4
                              ? __ldg(reinterpret_cast<const float *>(i < n1 ? a.z13 : a.z2) + cu.e)
                              : 1.f;
        if (i < n1) {
            for (cu.tb = 0; cu.tb < cu.ne;) {
                const int nt = cu.ne - cu.tb;
                if (nt >= 4) {
                    dec_compute<kDecGateUp, L1, 1, GT1, 4, FMT>(wb, wg1, acc1, cu, s_pairs, cache, 0, nullptr, td1, lane, s_tok, gsc);
                    layer_finish_gate_up<L1, 4>(acc1, cu, a, G2, lane);
                    cu.tb += 4;
                } else if (nt >= 2) {
                    dec_compute<kDecGateUp, L1, 1, GT1, 2, FMT>(wb, wg1, acc1, cu, s_pairs, cache, 0, nullptr, td1, lane, s_tok, gsc);
                    layer_finish_gate_up<L1, 2>(acc1, cu, a, G2, lane);
                    cu.tb += 2;
                } else {
                    dec_compute<kDecGateUp, L1, 1, GT1, 1, FMT>(wb, wg1, acc1, cu, s_pairs, cache, 0, nullptr, td1, lane, s_tok, gsc);
                    layer_finish_gate_up<L1, 1>(acc1, cu, a, G2, lane);
                    cu.tb += 1;
                }
            }
            if (lane == 0) atomicAdd(&s_cnt1[tp.ai], cu.cnt);
        } else {
            for (cu.tb = 0; cu.tb < cu.ne;) {
                const int nt = cu.ne - cu.tb;
                if (nt >= 4) {
                    dec_compute<kDecDown, L2, 2, GT2, 4, FMT>(wb, wg2, acc2, cu, s_pairs, cache, hrow0, nullptr, td2, lane, nullptr, gsc);
                    layer_finish_down<L2, 4>(acc2, cu, s_pairs, a, lane);
                    cu.tb += 4;
                } else if (nt >= 2) {
                    dec_compute<kDecDown, L2, 2, GT2, 2, FMT>(wb, wg2, acc2, cu, s_pairs, cache, hrow0, nullptr, td2, lane, nullptr, gsc);
                    layer_finish_down<L2, 2>(acc2, cu, s_pairs, a, lane);
                    cu.tb += 2;
                } else {
                    dec_compute<kDecDown, L2, 2, GT2, 1, FMT>(wb, wg2, acc2, cu, s_pairs, cache, hrow0, nullptr, td2, lane, nullptr, gsc);
                    layer_finish_down<L2, 1>(acc2, cu, s_pairs, a, lane);
                    cu.tb += 1;
                }
            }
            if (lane == 0) {
                const int n_lo = cu.unit0, n_hi = cu.unit0 + cu.cnt;
                for (int nb = n_lo / 8; nb <= (n_hi - 1) / 8; ++nb)
                    atomicAdd(&s_blk[nb], min(n_hi, nb * 8 + 8) - max(n_lo, nb * 8));
            }
        }
        __syncwarp();
        if (iss < ntask) issue();  // a warp that found a wait timed out left the loop above
    }
    // never leave with a copy in flight into this CTA's shared memory
    for (int j = consumed; j < iss; ++j)
        mbar_wait_bounded(bars + j % kLayerSlots, (uint32_t)((j / kLayerSlots) & 1), nullptr);

    // ---- 4. publish this CTA's row counts per output block, then combine
    // this CTA's slice of blocks once every active expert's rows are in
    __syncthreads();
    if (tid == 0) stamp(kLtDownDone);
    if (!dead) {
        for (int nb = tid; nb < nblk; nb += NTH) {
            const int c = s_blk[nb];
            if (c == 0) continue;
            __threadfence();
            atomicAdd(a.blkctr + nb, (unsigned)c);
        }
    }
    const int q_lo = (int)((long long)nblk * cta / NC), q_hi = (int)((long long)nblk * (cta + 1) / NC);
    const int units = (q_hi - q_lo) * a.T;  // (block, token) pairs
    const int o = lane & 7, js = lane >> 3;
    for (int u = warp; u < units; u += NW) {
        const int nb = q_lo + u / a.T, t = u - (u / a.T) * a.T;
        if (s_misc[3]) break;  // an earlier wait of this CTA expired
        // every lane waits (acquire) for all rows of the block
        uint32_t it = 0;
        while (ld_acquire_u32(a.blkctr + nb) < (uint32_t)A * 8u + extra && ++it < polls) __nanosleep(64);
        if (__any_sync(0xffffffffu, it >= polls)) {
            if (lane == 0) {
                set_error(a.err, MOE_DEVERR_WAIT_TIMEOUT);
                s_misc[3] = 1;
            }
            break;
        }
        // out[t][n] = sum_j w[t][j] y[t*k+j][n]: lanes (o, js) sum j = js, js+4, ...,
        // then a fixed shuffle tree over js (deterministic order)
        // (every load of a lane issued before the first product: one L2
        // round trip instead of one per term)
        const int n = nb * 8 + o;
        float accv = 0.f;
        for (int j0 = js; j0 < k; j0 += 32) {
            float yv[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + 4 * jj;
                yv[jj] = j < k ? __ldcg(a.y + (size_t)(t * k + j) * H + n) : 0.f;
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + 4 * jj;
                if (j < k) accv = fmaf(s_w[t * k + j], yv[jj], accv);
            }
        }
        accv += __shfl_xor_sync(0xffffffffu, accv, 8);
        accv += __shfl_xor_sync(0xffffffffu, accv, 16);
        if (js == 0) a.out[(size_t)t * H + n] = __float2half_rn(accv);
    }
    __syncthreads();  // every poll of this CTA's blocks is done
    for (int nb = q_lo + tid; nb < q_hi; nb += NTH) a.blkctr[nb] = 0u;

    // ---- the last CTA to leave resets the per-expert counters
    __syncthreads();
    if (tid == 0) stamp(kLtExit);
    if (tid == 0) {
        __threadfence();
        const unsigned old = atomicAdd(a.exitctr, 1u);
        if (old == (unsigned)NC - 1u) {
            for (int s = 0; s < P; ++s) a.done[s] = 0u;
            *a.exitctr = 0u;
            __threadfence();
        }
    }
}

// ---------------------------------------------------------------- launch
// Launch shape of the layer kernel for one problem size.
struct LayerPlan {
    bool ok;
    int nw, hrows, L1, L2;
    uint32_t slot_bytes;
    size_t smem;
};

// Cooperative launch of one instantiation: one CTA per SM, all resident.
template <typename K>
cudaError_t launch_layer_k(K kern, int *configured, const LayerArgs &a, const LayerPlan &pl, int num_sms,
                           cudaStream_t stream) {
    cudaError_t e = ensure_smem(kern, configured, pl.smem);
    if (e != cudaSuccess) return e;
    // the cooperative launch itself fails (cudaErrorCooperativeLaunchTooLarge)
    // unless every CTA can be resident at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(pl.nw * 32);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Pair segments (a.pair_mode) are compiled for the geometries with a
// compile-time group count only; elsewhere the grouped path runs.
template <int L1, int GT1, int L2, int GT2, int FMT>
cudaError_t launch_layer_t(const LayerArgs &a, const LayerPlan &pl, int num_sms, cudaStream_t stream) {
    if constexpr (GT1 != 0) {
        if (a.pair_mode) {
            static int configured_p[128];
            return launch_layer_k(decode_layer_kernel<L1, GT1, L2, GT2, FMT, true>, configured_p, a, pl, num_sms,
                                  stream);
        }
    }
    static int configured[128];
    return launch_layer_k(decode_layer_kernel<L1, GT1, L2, GT2, FMT, false>, configured, a, pl, num_sms, stream);
}

#define MOE_LAYER_INSTANCES(X) \
    X(16, 80, 4, 20)           \
    X(16, 80, 1, 5)            \
    X(16, 0, 4, 0)             \
    X(16, 0, 1, 0)             \
    X(4, 0, 4, 0)              \
    X(4, 0, 1, 0)              \
    X(1, 0, 4, 0)              \
    X(1, 0, 1, 0)

#define MOE_LAYER_EXTERN(L1, GT1, L2, GT2)                                                              \
    extern template cudaError_t launch_layer_t<L1, GT1, L2, GT2, kFmtW4A16>(const LayerArgs &, const LayerPlan &, \
                                                                            int, cudaStream_t);               \
    extern template cudaError_t launch_layer_t<L1, GT1, L2, GT2, kFmtNvfp4>(const LayerArgs &, const LayerPlan &, \
                                                                            int, cudaStream_t);
MOE_LAYER_INSTANCES(MOE_LAYER_EXTERN)
#undef MOE_LAYER_EXTERN

}  // namespace moe
