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
// in the error word and the kernel finishes without the dependent work.
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
    L.blk = (uint32_t)align_up((size_t)(10 * P + 8) * 4, 128);
    L.cache = L.blk + (uint32_t)align_up((size_t)(2 * (H / 8)) * 4, 128);
    const size_t xc = (size_t)T * H * 2, hc = (size_t)hrows * I * 2;
    L.ring = L.cache + (uint32_t)align_up(xc > hc ? xc : hc, 128);
    L.bars = L.ring + (uint32_t)nw * kLayerSlots * slot_bytes;
    L.total = L.bars + (uint32_t)nw * kLayerSlots * 8;
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

template <int L1, int GT1, int L2, int GT2>
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
    int *s_misc = g_first + P;  // [0] A, [1] completed blocks, [2] h not ready
    int *s_blk = reinterpret_cast<int *>(smem + Ly.blk);  // [nblk] counts, [nblk] completed list
    uint8_t *cache = smem + Ly.cache;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t *ring = smem + Ly.ring + (size_t)warp * kLayerSlots * a.slot_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Ly.bars) + warp * kLayerSlots;
    const WarpGeom wg1 = warp_geom(RT1, 2, H), wg2 = warp_geom(RT2, 1, I);

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kLayerSlots; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    for (int i = tid; i < 2 * nblk; i += NTH) s_blk[i] = 0;
    for (int i = tid; i < P; i += NTH) s_cnt1[i] = 0;
    if (tid < 8) s_misc[tid] = 0;
    pdl_wait();
    pdl_trigger();

    // ---- 1. route (warps < T) while the other warps stage the x rows
    if (warp < a.T) {
        const bool lead = blockIdx.x == 0;
        route_token<kLayerRoutePer>(a.logits + (size_t)warp * a.E, a.E, k, warp, lead ? a.topk_ids : nullptr,
                                    lead ? a.topk_w : nullptr, s_ids, s_w);
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
        g_less[p] = less;
        g_same[p] = same;
        g_first[p] = before == 0;
        if (before == 0) atomicAdd(&s_misc[0], 1);
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

    // ---- 2. this CTA's tasks: contiguous shares of both task lists
    const int A = s_misc[0];
    const int TPE1 = (I + RT1 - 1) / RT1, TPE2 = (H + RT2 - 1) / RT2;
    const int U1 = A * TPE1, U2 = A * TPE2;
    const int cta = blockIdx.x, NC = gridDim.x;
    const int b1 = (int)((long long)U1 * cta / NC), e1 = (int)((long long)U1 * (cta + 1) / NC);
    const int b2 = (int)((long long)U2 * cta / NC), e2 = (int)((long long)U2 * (cta + 1) / NC);
    const int n1 = e1 - b1 > warp ? (e1 - b1 - warp + NW - 1) / NW : 0;
    const int n2 = e2 - b2 > warp ? (e2 - b2 - warp + NW - 1) / NW : 0;
    const int ntask = n1 + n2;

    auto cursor = [&](int i, Cursor &cu) -> int {  // returns the active slot
        int ai;
        if (i < n1) {
            const int uu = b1 + warp + i * NW;
            ai = uu / TPE1;
            cu.unit0 = (uu - ai * TPE1) * RT1;
            cu.cnt = min(RT1, I - cu.unit0);
        } else {
            const int uu = b2 + warp + (i - n1) * NW;
            ai = uu / TPE2;
            cu.unit0 = (uu - ai * TPE2) * RT2;
            cu.cnt = min(RT2, H - cu.unit0);
        }
        cu.e = s_act[ai];
        cu.r0 = s_lo[ai];
        cu.ne = s_hi[ai] - cu.r0;
        cu.tb = 0;
        return ai;
    };
    // lane 0 fetches task i into slot i % kLayerSlots
    auto issue = [&](int i) {
        if (lane != 0) return;
        Cursor cu;
        cursor(i, cu);
        uint8_t *wb = ring + (size_t)(i % kLayerSlots) * a.slot_bytes;
        uint64_t *bar = bars + i % kLayerSlots;
        fence_proxy_async();  // this warp's earlier reads of the slot come first
        if (i < n1) {
            WarpCopy cp[2];
            uint32_t tx = 0;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                cp[b] = warp_copy(cu.e, cu.unit0 + b * I, cu.cnt, 2 * I, H);
                tx += cp[b].q_len + cp[b].s_len + cp[b].z_len;
            }
            mbar_arrive_expect_tx(bar, tx);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                bulk_g2s(wb + b * wg1.q_bytes, reinterpret_cast<const uint8_t *>(a.q13) + cp[b].q_off,
                         cp[b].q_len, bar);
                bulk_g2s(wb + 2 * wg1.q_bytes + b * wg1.s_bytes,
                         reinterpret_cast<const uint8_t *>(a.s13) + cp[b].s_a, cp[b].s_len, bar);
                bulk_g2s(wb + 2 * (wg1.q_bytes + wg1.s_bytes) + b * wg1.z_bytes,
                         reinterpret_cast<const uint8_t *>(a.z13) + cp[b].z_a, cp[b].z_len, bar);
            }
        } else {
            const WarpCopy cp = warp_copy(cu.e, cu.unit0, cu.cnt, H, I);
            mbar_arrive_expect_tx(bar, cp.q_len + cp.s_len + cp.z_len);
            bulk_g2s(wb, reinterpret_cast<const uint8_t *>(a.q2) + cp.q_off, cp.q_len, bar);
            bulk_g2s(wb + wg2.q_bytes, reinterpret_cast<const uint8_t *>(a.s2) + cp.s_a, cp.s_len, bar);
            bulk_g2s(wb + wg2.q_bytes + wg2.s_bytes, reinterpret_cast<const uint8_t *>(a.z2) + cp.z_a,
                     cp.z_len, bar);
        }
    };

    const int nfirst = ntask < kLayerSlots ? ntask : kLayerSlots;
    for (int i = 0; i < nfirst; ++i) issue(i);
    int issued = nfirst, consumed = 0;

    const TaskDims td1{2 * I, H, I, P, k}, td2{H, I, H, P, k};
    float acc1[1][2][kDecPass], acc2[2][1][kDecPass];
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int t = 0; t < kDecPass; ++t) acc1[0][b][t] = acc2[b][0][t] = 0.f;
    bool dead = false;
    int hrow0 = 0;

    for (int i = 0; i <= ntask; ++i) {
        if (i == n1) {
            // ---- 3. between the steps (every warp passes here once)
            __syncthreads();  // this CTA's h values are written
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
                    while (ld_acquire_u32(a.done + s) < (uint32_t)I && ++it < kPollTries) __nanosleep(64);
                    if (it >= kPollTries) {
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
        const uint8_t *wb = ring + (size_t)s * a.slot_bytes;
        Cursor cu;
        const int ai = cursor(i, cu);
        if (i < n1) {
            for (cu.tb = 0; cu.tb < cu.ne; cu.tb += kDecPass) {
                const int nt = min(kDecPass, cu.ne - cu.tb);
                switch (nt) {
                    case 1:
                        dec_compute<kDecGateUp, L1, 1, GT1, 1>(wb, wg1, acc1, cu, s_pairs, cache, 0, nullptr, td1, lane);
                        layer_finish_gate_up<L1, 1>(acc1, cu, a, G2, lane);
                        break;
                    case 2:
                        dec_compute<kDecGateUp, L1, 1, GT1, 2>(wb, wg1, acc1, cu, s_pairs, cache, 0, nullptr, td1, lane);
                        layer_finish_gate_up<L1, 2>(acc1, cu, a, G2, lane);
                        break;
                    case 3:
                        dec_compute<kDecGateUp, L1, 1, GT1, 3>(wb, wg1, acc1, cu, s_pairs, cache, 0, nullptr, td1, lane);
                        layer_finish_gate_up<L1, 3>(acc1, cu, a, G2, lane);
                        break;
                    default:
                        dec_compute<kDecGateUp, L1, 1, GT1, 4>(wb, wg1, acc1, cu, s_pairs, cache, 0, nullptr, td1, lane);
                        layer_finish_gate_up<L1, 4>(acc1, cu, a, G2, lane);
                        break;
                }
            }
            if (lane == 0) atomicAdd(&s_cnt1[ai], cu.cnt);
        } else {
            for (cu.tb = 0; cu.tb < cu.ne; cu.tb += kDecPass) {
                const int nt = min(kDecPass, cu.ne - cu.tb);
                switch (nt) {
                    case 1:
                        dec_compute<kDecDown, L2, 2, GT2, 1>(wb, wg2, acc2, cu, s_pairs, cache, hrow0, nullptr, td2, lane);
                        layer_finish_down<L2, 1>(acc2, cu, s_pairs, a, lane);
                        break;
                    case 2:
                        dec_compute<kDecDown, L2, 2, GT2, 2>(wb, wg2, acc2, cu, s_pairs, cache, hrow0, nullptr, td2, lane);
                        layer_finish_down<L2, 2>(acc2, cu, s_pairs, a, lane);
                        break;
                    case 3:
                        dec_compute<kDecDown, L2, 2, GT2, 3>(wb, wg2, acc2, cu, s_pairs, cache, hrow0, nullptr, td2, lane);
                        layer_finish_down<L2, 3>(acc2, cu, s_pairs, a, lane);
                        break;
                    default:
                        dec_compute<kDecDown, L2, 2, GT2, 4>(wb, wg2, acc2, cu, s_pairs, cache, hrow0, nullptr, td2, lane);
                        layer_finish_down<L2, 4>(acc2, cu, s_pairs, a, lane);
                        break;
                }
            }
            if (lane == 0) {
                const int n_lo = cu.unit0, n_hi = cu.unit0 + cu.cnt;
                for (int nb = n_lo / 8; nb <= (n_hi - 1) / 8; ++nb)
                    atomicAdd(&s_blk[nb], min(n_hi, nb * 8 + 8) - max(n_lo, nb * 8));
            }
        }
        __syncwarp();
        if (issued < ntask) issue(issued++);
    }
    // never leave with a copy in flight into this CTA's shared memory
    for (int j = consumed; j < issued; ++j)
        mbar_wait_bounded(bars + j % kLayerSlots, (uint32_t)((j / kLayerSlots) & 1), nullptr);

    // ---- 4. publish row counts; combine the blocks this CTA completes
    __syncthreads();
    int *s_done = s_blk + nblk;
    if (!dead) {
        for (int nb = tid; nb < nblk; nb += NTH) {
            const int c = s_blk[nb];
            if (c == 0) continue;
            __threadfence();
            const unsigned old = atomicAdd(a.blkctr + nb, (unsigned)c);
            if (old + c == (unsigned)A * 8u) {
                __threadfence();
                s_done[atomicAdd(&s_misc[1], 1)] = nb;
            }
        }
    }
    __syncthreads();
    const int ndone = s_misc[1];
    if (ndone > 0) __threadfence();
    for (int d = warp; d < ndone; d += NW) {
        const int nb = s_done[d];
        for (int idx = lane; idx < a.T * 8; idx += 32) {
            const int t = idx >> 3, n = nb * 8 + (idx & 7);
            float accv = 0.f;
#pragma unroll 8
            for (int j = 0; j < k; ++j) {  // unrolled: the loads go out together
                const int p = t * k + j;
                accv = fmaf(s_w[p], __ldcg(a.y + (size_t)p * H + n), accv);
            }
            a.out[(size_t)t * H + n] = __float2half_rn(accv);
        }
        __syncwarp();
        if (lane == 0) atomicExch(a.blkctr + nb, 0u);
    }

    // ---- the last CTA to leave resets the per-expert counters
    __syncthreads();
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
template <int L1, int GT1, int L2, int GT2>
cudaError_t launch_layer_t(const LayerArgs &a, const LayerPlan &pl, int num_sms, cudaStream_t stream) {
    auto kern = decode_layer_kernel<L1, GT1, L2, GT2>;
    static int configured[128];
    cudaError_t e = ensure_smem(kern, configured, pl.smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, pl.nw * 32, pl.smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
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

#define MOE_LAYER_INSTANCES(X) \
    X(16, 80, 4, 20)           \
    X(16, 80, 1, 5)            \
    X(16, 0, 4, 0)             \
    X(16, 0, 1, 0)             \
    X(4, 0, 4, 0)              \
    X(4, 0, 1, 0)              \
    X(1, 0, 4, 0)              \
    X(1, 0, 1, 0)

#define MOE_LAYER_EXTERN(L1, GT1, L2, GT2)                                                         \
    extern template cudaError_t launch_layer_t<L1, GT1, L2, GT2>(const LayerArgs &, const LayerPlan &, \
                                                                 int, cudaStream_t);
MOE_LAYER_INSTANCES(MOE_LAYER_EXTERN)
#undef MOE_LAYER_EXTERN

}  // namespace moe
