// decode_gemv.cuh -- steps 3 and 4 for decode batches (T <= 16, as far as the
// shared-memory layout allows): the
// latency-first weight stream.
//
// "Active grouped decode" ("[Perf][SM70] Narrow Qwen3.8 AWQ active grouped
// decode", section Purpose) runs 2-8 tokens through only the experts they
// selected.  At that size the whole step is a few tens of megabytes, so what
// matters is how soon every SM has its share in flight and how many
// independent instructions each warp can issue:
//
//  * One CTA per SM, of 14 warps (fewer, down to 6, when step 3's cache of
//    every x row leaves too little room for 14 task buffers: on the
//    Qwen4Exp geometry 12 warps at 11-15 tokens, 10 at 16).  A prologue, run by every thread with all loads
//    issued before any store, brings the routing metadata (active list,
//    offsets, pair ids) and the activations (every x row in step 3, every h
//    row in step 4 when they fit) into shared memory in a single round trip.
//  * Work is cut into warp tasks: RT consecutive row units (gate/up row pairs
//    in step 3, output rows in step 4) of one active expert, L lanes per row
//    unit.  Tasks are dealt round-robin over CTAs, then over their warps, so
//    every SM gets the same share whatever the active experts.
//  * Each warp owns a shared-memory buffer and an mbarrier.  A task's rows
//    are contiguous in every packed tensor, so lane 0 fetches the whole task
//    (codes, scales, zero words of its gate and up rows, or of its down
//    rows) with a handful of bulk asynchronous copies; the warp's lanes then
//    dequantise from shared memory.  With 14 warps per SM that many tasks are
//    in flight at once, without spending registers on them.  The kGPI groups
//    of a row are worked on together, with independent fp16 chains, to keep
//    the issue slots busy.
//  * Dequantisation and arithmetic are those of common.cuh: code - zero in
//    fp16 pairs, fp16 products summed per group, fp32 group accumulation.
//  * For the geometries the layer is specified on, the number of groups per
//    row is a compile-time constant, so every shared-memory offset of a
//    task is an immediate and each lane's group loop unrolls completely.
//  * Step 4 writes each pair's fp32 projection to the workspace and counts
//    finished rows per 8-row output block in shared memory.  At the end each
//    CTA publishes its counts (one fence, parallel atomics); whichever CTA
//    completes a block sums the block's k terms per token in order and writes
//    fp16 (deterministic, no extra launch).
#pragma once
#include "decode_common.cuh"

namespace moe {

constexpr int kDecWarps = 14;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecMinWarps = 6;
// batches these kernels can take: T <= kDecMaxT when the layout fits in
// shared memory (on the Qwen4Exp geometry, with fewer warps past 10 tokens,
// up to 29).  Which batches they are chosen for is the dispatch's business.
#ifndef DEC_MAX_T
#define DEC_MAX_T 32
#endif
constexpr int kDecMaxT = DEC_MAX_T;

struct DecodeArgs {
    const uint32_t *q;   // packed codes  [E][N][K/8]
    const __half *s;     // scales        [E][N][K/32]
    const uint32_t *z;   // packed zeros  [E][N/8][K/32]
    int E, N, K;         // N: matrix rows per expert, K: reduction length
    int rows;            // row units per expert: I (gate/up pairs) or H
    const __half *vin;   // step 3: x [T][K]; step 4: h [P][K]
    int T, k, P;
    const int32_t *offsets, *sorted_pair, *active, *num_active;
    __half *h_out;       // step 3: [P][I]
    float *y_out;        // step 4: [P][H]
    const float *topk_w; // step 4
    __half *out;         // step 4: [T][H]
    uint32_t *counters;  // step 4: [H/8]
    uint32_t *err;
    int slots;           // activation rows held in shared memory (step 4: P or 0)
    int nblk;            // step 4: 8-row output blocks (H/8); step 3: 0
    uint32_t wbytes;     // per-warp task buffer
};

// meta: [A | pad3 | active E | offsets E+1 | pairs P] ints; blk: 2*nblk ints
// (per-block row counts, then the list of blocks this CTA completed); xc:
// activation cache; wbuf: per-warp task buffers; bars: per-warp mbarriers.
struct DecLayout {
    uint32_t meta, blk, xc, wbuf, bars, total;
};

__host__ __device__ inline DecLayout dec_layout(int E, int P, int nblk, int slots, int K, uint32_t wbytes,
                                                 int nw = kDecWarps) {
    DecLayout L;
    L.meta = 0;
    L.blk = (uint32_t)align_up((size_t)(4 + E + E + 1 + P) * 4, 128);
    L.xc = L.blk + (uint32_t)align_up((size_t)(2 * nblk + 4) * 4, 128);
    L.wbuf = L.xc + (uint32_t)align_up((size_t)slots * K * 2, 128);
    L.bars = L.wbuf + (uint32_t)nw * wbytes;
    L.total = L.bars + nw * 8;
    return L;
}

// Warps of a decode launch: kDecWarps, else the most of 12, 10, 8 or 6 whose
// task buffers fit beside the activation cache (step 3 keeps every x row of
// the batch, so larger batches leave room for fewer buffers); 0 if none fits.
__host__ __device__ inline int dec_warps(int E, int P, int nblk, int slots, int K, uint32_t wbytes,
                                         size_t smem_limit) {
    for (int nw = kDecWarps; nw >= kDecMinWarps; nw -= 2)
        if (dec_layout(E, P, nblk, slots, K, wbytes, nw).total <= smem_limit) return nw;
    return 0;
}

// End of a token pass: finish the dot products across the L lanes of each
// row unit and write h (step 3) or y (step 4) for the pass's rows.
template <int MODE, int L, int RU, int NT>
__device__ __forceinline__ void dec_finish(float (&acc)[RU][DecTraits<MODE, L, RU>::nmat][kDecPass],
                                           const Cursor &c, const int *s_pairs, const DecodeArgs &a,
                                           int lane) {
    using Tr = DecTraits<MODE, L, RU>;
    constexpr int nmat = Tr::nmat;
    const int ks = lane % L, us = lane / L;
#pragma unroll
    for (int ru = 0; ru < RU; ++ru)
#pragma unroll
        for (int b = 0; b < nmat; ++b)
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int off = L / 2; off > 0; off >>= 1)
                    acc[ru][b][t] += __shfl_xor_sync(0xffffffffu, acc[ru][b][t], off);
#pragma unroll
    for (int ru = 0; ru < RU; ++ru) {
        const int lr = us + ru * Tr::UPW;
        const int unit = c.unit0 + lr;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int r = c.r0 + c.tb + t;
            const int p = s_pairs[r];
            if (lr < c.cnt && (t % L) == ks) {
                if (p < 0 || p >= a.P) {
                    set_error(a.err, MOE_DEVERR_BAD_METADATA);
                } else if (MODE == kDecGateUp) {
                    const float gv = acc[ru][0][t], uv = acc[ru][nmat - 1][t];
                    const float hv = gv / (1.0f + __expf(-gv)) * uv;
                    a.h_out[(size_t)r * a.rows + unit] = __float2half_rn(hv);
                } else {
                    a.y_out[(size_t)p * a.N + unit] = acc[ru][0][t];
                }
            }
        }
    }
#pragma unroll
    for (int ru = 0; ru < RU; ++ru)
#pragma unroll
        for (int b = 0; b < nmat; ++b)
#pragma unroll
            for (int t = 0; t < kDecPass; ++t) acc[ru][b][t] = 0.f;
}

template <int MODE, int L, int RU, int GT, int FMT>
__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(const DecodeArgs a) {
    using Tr = DecTraits<MODE, L, RU>;
    constexpr int nmat = Tr::nmat;
    extern __shared__ __align__(128) uint8_t smem[];
    const int G = GT ? GT : a.K / 32;
    const int K = 32 * G;
    // warps of this launch (kDecWarps, or fewer where their buffers and a
    // larger activation cache would not fit together)
    const int NW = blockDim.x >> 5, NTH = NW * 32;
    const DecLayout Ly = dec_layout(a.E, a.P, a.nblk, a.slots, K, a.wbytes, NW);
    const WarpGeom wg = warp_geom(Tr::RT, nmat, K);
    int *s_meta = reinterpret_cast<int *>(smem + Ly.meta);
    int *s_active = s_meta + 4;
    int *s_offs = s_active + a.E;
    int *s_pairs = s_offs + a.E + 1;
    int *s_blk = reinterpret_cast<int *>(smem + Ly.blk);  // [nblk] counts, [nblk] done list, [1] n done
    uint8_t *xcb = smem + Ly.xc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t *wb = smem + Ly.wbuf + (size_t)warp * a.wbytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Ly.bars) + warp;

    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    for (int i = tid; i < 2 * a.nblk + 1; i += NTH) s_blk[i] = 0;
    pdl_wait();
    pdl_trigger();

    // ---- prologue: metadata and activations, all loads first
    {
        const int nmeta = a.E + (a.E + 1) + a.P;  // active | offsets | pairs
        for (int base = 0; base < nmeta; base += 4 * NTH) {
            int v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = base + tid + c * NTH;
                v[c] = 0;
                if (i < a.E)
                    v[c] = __ldg(a.active + i);
                else if (i < 2 * a.E + 1)
                    v[c] = __ldg(a.offsets + (i - a.E));
                else if (i < nmeta)
                    v[c] = __ldg(a.sorted_pair + (i - 2 * a.E - 1));
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = base + tid + c * NTH;
                if (i < nmeta) s_active[i] = v[c];  // active, offsets, pairs are contiguous
            }
        }
        if (tid == 0) s_meta[0] = __ldg(a.num_active);
        // step 3: every x row; step 4: every h row when the cache holds them
        if (MODE == kDecGateUp || a.slots >= a.P) dec_stage_rows(a.vin, MODE == kDecGateUp ? a.T : a.P, K, G, xcb, tid, NTH);
    }
    __syncthreads();
    const bool hc = MODE == kDecDown && a.slots >= a.P;
    const TaskDims td{a.N, K, a.rows, a.P, a.k};

    int A = s_meta[0];
    A = A < 0 ? 0 : (A > a.E ? a.E : A);
    const int TPE = (a.rows + Tr::RT - 1) / Tr::RT;  // tasks per expert
    const int U = A * TPE;
    // tasks dealt round-robin: CTA first, then warp
    const int ustride = gridDim.x * NW;
    int u = blockIdx.x + gridDim.x * warp;

    // task u's expert and segment; false if the metadata is bad
    auto task = [&](int uu, Cursor &c) -> bool {
        const int ai = uu / TPE;
        c.e = s_active[ai];
        if (c.e < 0 || c.e >= a.E) return false;
        c.r0 = s_offs[c.e];
        const int r1 = s_offs[c.e + 1];
        if (c.r0 < 0 || r1 > a.P || r1 <= c.r0) return false;
        c.ne = r1 - c.r0;
        c.unit0 = (uu - ai * TPE) * Tr::RT;
        c.cnt = min(Tr::RT, a.rows - c.unit0);
        c.tb = 0;
        return true;
    };
    // lane 0 fetches the whole task into this warp's buffer
    auto issue = [&](const Cursor &c) {
        if (lane != 0) return;
        fence_proxy_async();  // this warp's earlier reads of the buffer come first
        WarpCopy cp[nmat];
        uint32_t tx = 0;
#pragma unroll
        for (int b = 0; b < nmat; ++b) {
            cp[b] = warp_copy(c.e, c.unit0 + b * a.rows, c.cnt, a.N, K);
            tx += cp[b].q_len + cp[b].s_len + (FMT == kFmtNvfp4 ? 0u : cp[b].z_len);
        }
        mbar_arrive_expect_tx(bar, tx);
#pragma unroll
        for (int b = 0; b < nmat; ++b) {
            bulk_g2s(wb + b * wg.q_bytes, reinterpret_cast<const uint8_t *>(a.q) + cp[b].q_off, cp[b].q_len, bar);
            bulk_g2s(wb + nmat * wg.q_bytes + b * wg.s_bytes, reinterpret_cast<const uint8_t *>(a.s) + cp[b].s_a,
                     cp[b].s_len, bar);
            if (FMT != kFmtNvfp4)  // NVFP4: no zero words (a.z holds the per-expert scales)
                bulk_g2s(wb + nmat * (wg.q_bytes + wg.s_bytes) + b * wg.z_bytes,
                         reinterpret_cast<const uint8_t *>(a.z) + cp[b].z_a, cp[b].z_len, bar);
        }
    };

    Cursor cur;
    while (u < U && !task(u, cur)) {
        if (lane == 0) set_error(a.err, MOE_DEVERR_BAD_METADATA);
        u += ustride;
    }
    if (u < U) issue(cur);

    float acc[Tr::RT > 0 ? RU : 1][nmat][kDecPass];
#pragma unroll
    for (int ru = 0; ru < RU; ++ru)
#pragma unroll
        for (int b = 0; b < nmat; ++b)
#pragma unroll
            for (int t = 0; t < kDecPass; ++t) acc[ru][b][t] = 0.f;
    uint32_t phase = 0;
    bool dead = false;
    while (u < U) {
        if (!mbar_wait_bounded(bar, phase, nullptr)) {
            if (lane == 0) set_error(a.err, MOE_DEVERR_WAIT_TIMEOUT);
            mbar_wait_bounded(bar, phase, nullptr);  // never leave with a copy in flight
            dead = true;
            break;
        }
        phase ^= 1u;
        const float gsc = FMT == kFmtNvfp4 ? __ldg(reinterpret_cast<const float *>(a.z) + cur.e) : 1.f;
        // segments longer than a pass (several tokens on one expert) take more passes
        for (cur.tb = 0; cur.tb < cur.ne; cur.tb += kDecPass) {
            const int nt = min(kDecPass, cur.ne - cur.tb);
            switch (nt) {
                case 1:
                    dec_compute<MODE, L, RU, GT, 1, FMT>(wb, wg, acc, cur, s_pairs, xcb, 0, hc ? nullptr : a.vin, td, lane,
                                                         nullptr, gsc);
                    dec_finish<MODE, L, RU, 1>(acc, cur, s_pairs, a, lane);
                    break;
                case 2:
                    dec_compute<MODE, L, RU, GT, 2, FMT>(wb, wg, acc, cur, s_pairs, xcb, 0, hc ? nullptr : a.vin, td, lane,
                                                         nullptr, gsc);
                    dec_finish<MODE, L, RU, 2>(acc, cur, s_pairs, a, lane);
                    break;
                case 3:
                    dec_compute<MODE, L, RU, GT, 3, FMT>(wb, wg, acc, cur, s_pairs, xcb, 0, hc ? nullptr : a.vin, td, lane,
                                                         nullptr, gsc);
                    dec_finish<MODE, L, RU, 3>(acc, cur, s_pairs, a, lane);
                    break;
                default:
                    dec_compute<MODE, L, RU, GT, 4, FMT>(wb, wg, acc, cur, s_pairs, xcb, 0, hc ? nullptr : a.vin, td, lane,
                                                         nullptr, gsc);
                    dec_finish<MODE, L, RU, 4>(acc, cur, s_pairs, a, lane);
                    break;
            }
        }
        if (MODE == kDecDown && lane == 0) {
            // count this task's rows into its 8-row output blocks (shared)
            const int n_lo = cur.unit0, n_hi = cur.unit0 + cur.cnt;
            for (int nb = n_lo / 8; nb <= (n_hi - 1) / 8; ++nb)
                atomicAdd(&s_blk[nb], min(n_hi, nb * 8 + 8) - max(n_lo, nb * 8));
        }
        __syncwarp();
        // next valid task of this warp
        for (u += ustride; u < U && !task(u, cur); u += ustride)
            if (lane == 0) set_error(a.err, MOE_DEVERR_BAD_METADATA);
        if (u < U) issue(cur);
    }

    if (MODE == kDecDown) {
        // Publish this CTA's row counts: the y rows of every warp precede the
        // barrier, the barrier precedes each publishing thread's fence and
        // atomic.  A thread whose atomic completes a block queues it.
        __syncthreads();
        int *s_done = s_blk + a.nblk, *s_ndone = s_blk + 2 * a.nblk;
        for (int nb = tid; nb < a.nblk; nb += NTH) {
            const int cnt = s_blk[nb];
            if (cnt == 0 || dead) continue;
            __threadfence();
            const unsigned old = atomicAdd(a.counters + nb, (unsigned)cnt);
            if (old + cnt == (unsigned)A * 8u) {
                __threadfence();
                s_done[atomicAdd(s_ndone, 1)] = nb;
            }
        }
        __syncthreads();
        const int ndone = *s_ndone;
        if (ndone > 0) __threadfence();
        // each completed block: out[t][8 rows] = sum_j w[t][j] * y[t*k+j] in j order
        for (int d = warp; d < ndone; d += NW) {
            const int nb = s_done[d];
            for (int idx = lane; idx < a.T * 8; idx += 32) {
                const int t = idx >> 3, n = nb * 8 + (idx & 7);
                float accv = 0.f;
#pragma unroll 8
                for (int jj = 0; jj < a.k; ++jj) {  // unrolled: the loads go out together
                    const int p = t * a.k + jj;
                    accv = fmaf(__ldg(a.topk_w + p), __ldcg(a.y_out + (size_t)p * a.N + n), accv);
                }
                a.out[(size_t)t * a.N + n] = __float2half_rn(accv);
            }
            __syncwarp();
            if (lane == 0) atomicExch(a.counters + nb, 0u);
        }
    }
}

// ---------------------------------------------------------------- launchers
template <int MODE, int L, int RU, int GT, int FMT>
inline cudaError_t launch_decode_t(DecodeArgs a, int num_sms, size_t smem_limit, cudaStream_t stream) {
    using Tr = DecTraits<MODE, L, RU>;
    a.wbytes = warp_geom(Tr::RT, Tr::nmat, a.K).bytes;
    const int nw = dec_warps(a.E, a.P, a.nblk, a.slots, a.K, a.wbytes, smem_limit);
    if (nw == 0) return cudaErrorInvalidConfiguration;
    const size_t smem = dec_layout(a.E, a.P, a.nblk, a.slots, a.K, a.wbytes, nw).total;
    static int configured[128];
    cudaError_t e = ensure_smem(decode_kernel<MODE, L, RU, GT, FMT>, configured, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_kernel<MODE, L, RU, GT, FMT>, num_sms, nw * 32, smem, stream, a);
}

// Lanes per row unit: a power of two giving each lane about five groups.
inline int lanes_for(int G) { return G >= 40 ? 8 : (G >= 20 ? 4 : (G >= 10 ? 2 : 1)); }

// Per-warp buffer of the decode kernels (step 3: a task of 32/L row pairs;
// step 4: a task of 2*32/L rows).
inline uint32_t decode_wbytes(int H, int I, bool gate_up) {
    const int G = (gate_up ? H : I) / 32, L = lanes_for(G);
    return gate_up ? warp_geom(32 / L, 2, H).bytes : warp_geom(2 * (32 / L), 1, I).bytes;
}

// step 4 caches every h row when they fit next to its task buffers
inline int down_slots(int T, int E, int k, int H, int I, size_t smem_limit) {
    const int P = T * k;
    const uint32_t wb = decode_wbytes(H, I, false);
    return dec_layout(E, P, H / 8, P, I, wb).total <= smem_limit ? P : 0;
}

inline bool decode_supported_impl(int T, int E, int k, int H, int I, size_t smem_limit) {
    const int P = T * k;
    return T >= 1 && T <= kDecMaxT && dec_warps(E, P, 0, T, H, decode_wbytes(H, I, true), smem_limit) > 0 &&
           dec_warps(E, P, H / 8, down_slots(T, E, k, H, I, smem_limit), I, decode_wbytes(H, I, false),
                     smem_limit) > 0;
}

template <int FMT>
cudaError_t launch_gate_up_decode_f(const __half *x, const uint32_t *q, const __half *s, const uint32_t *z,
                                  const int32_t *offsets, const int32_t *sorted_pair,
                                  const int32_t *active, const int32_t *num_active, int T, int E, int k,
                                  int H, int I, __half *h, uint32_t *err, int num_sms, size_t smem_limit,
                                  cudaStream_t stream) {
    DecodeArgs a{};
    a.q = q; a.s = s; a.z = z;
    a.E = E; a.N = 2 * I; a.K = H; a.rows = I;
    a.vin = x; a.T = T; a.k = k; a.P = T * k;
    a.offsets = offsets; a.sorted_pair = sorted_pair; a.active = active; a.num_active = num_active;
    a.h_out = h; a.err = err;
    a.slots = T;
    a.nblk = 0;
    const int G = H / 32;
    if (G == 80) return launch_decode_t<kDecGateUp, 8, 1, 80, FMT>(a, num_sms, smem_limit, stream);
    switch (lanes_for(G)) {
        case 8: return launch_decode_t<kDecGateUp, 8, 1, 0, FMT>(a, num_sms, smem_limit, stream);
        case 4: return launch_decode_t<kDecGateUp, 4, 1, 0, FMT>(a, num_sms, smem_limit, stream);
        case 2: return launch_decode_t<kDecGateUp, 2, 1, 0, FMT>(a, num_sms, smem_limit, stream);
        default: return launch_decode_t<kDecGateUp, 1, 1, 0, FMT>(a, num_sms, smem_limit, stream);
    }
}

template <int FMT>
cudaError_t launch_down_decode_f(const __half *h, const uint32_t *q, const __half *s, const uint32_t *z,
                               const int32_t *offsets, const int32_t *sorted_pair, const int32_t *active,
                               const int32_t *num_active, const float *topk_w, int T, int E, int k, int H,
                               int I, __half *out, float *y, uint32_t *counters, uint32_t *err,
                               int num_sms, size_t smem_limit, cudaStream_t stream) {
    DecodeArgs a{};
    a.q = q; a.s = s; a.z = z;
    a.E = E; a.N = H; a.K = I; a.rows = H;
    a.vin = h; a.T = T; a.k = k; a.P = T * k;
    a.offsets = offsets; a.sorted_pair = sorted_pair; a.active = active; a.num_active = num_active;
    a.y_out = y; a.topk_w = topk_w; a.out = out; a.counters = counters; a.err = err;
    a.slots = down_slots(T, E, k, H, I, smem_limit);
    a.nblk = H / 8;
    const int G = I / 32;
    if (G == 20) return launch_decode_t<kDecDown, 4, 2, 20, FMT>(a, num_sms, smem_limit, stream);
    if (G == 5) return launch_decode_t<kDecDown, 1, 2, 5, FMT>(a, num_sms, smem_limit, stream);
    switch (lanes_for(G)) {
        case 8: return launch_decode_t<kDecDown, 8, 2, 0, FMT>(a, num_sms, smem_limit, stream);
        case 4: return launch_decode_t<kDecDown, 4, 2, 0, FMT>(a, num_sms, smem_limit, stream);
        case 2: return launch_decode_t<kDecDown, 2, 2, 0, FMT>(a, num_sms, smem_limit, stream);
        default: return launch_decode_t<kDecDown, 1, 2, 0, FMT>(a, num_sms, smem_limit, stream);
    }
}

}  // namespace moe
