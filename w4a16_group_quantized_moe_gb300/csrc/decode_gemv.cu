// decode_gemv.cu -- steps 3 and 4 for decode batches (T <= 8): the
// latency-first weight stream.
//
// "Active grouped decode" ("[Perf][SM70] Narrow Qwen3.8 AWQ active grouped
// decode", section Purpose) runs 2-8 tokens through only the experts they
// selected.  At that size the whole step is a few tens of megabytes, so what
// matters is how soon every SM has its share in flight and how many
// independent instructions each warp can issue:
//
//  * One 16-warp CTA per SM.  A prologue, run by every thread with all loads
//    issued before any store, brings the routing metadata (active list,
//    offsets, pair ids) and, in step 3, every x row into shared memory in a
//    single round trip.  Step 4 caches the h rows of the CTA's segments (one
//    contiguous run of sorted rows) the same way.
//  * Work is cut into warp tasks: RT consecutive row units (gate/up row pairs
//    in step 3, output rows in step 4) of one active expert, L lanes per row
//    unit.  Task lists are split into equal contiguous ranges per warp.
//  * A warp walks its tasks in steps of kGPI groups per row: the loads of a
//    step (16-byte code words plus the matching scale and zero words) go
//    straight into registers one step ahead, so the next step (of this or
//    the next task) is in flight while the current one is dequantised and
//    multiplied.  The step's groups are worked on together, with independent
//    fp16 chains, to keep the issue slots busy.  No staging barriers.
//  * Dequantisation and arithmetic are those of common.cuh: code - zero in
//    fp16 pairs, fp16 products summed per group, fp32 group accumulation.
//  * Step 4 writes each pair's fp32 projection to the workspace and counts
//    finished rows per 8-row output block; the warp that completes a block
//    sums the block's k terms per token in order and writes fp16.
#include "common.cuh"

namespace moe {

constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecMaxT = 8;   // decode batches: T <= 8
constexpr int kDecPass = 4;   // activation rows per compute pass
constexpr int kGPI = 2;       // groups per lane per pipeline step

enum { kDecGateUp = 0, kDecDown = 1 };

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
    int slots;           // activation rows held in shared memory
};

struct DecLayout {
    uint32_t meta, xc, total;
};

__host__ __device__ inline DecLayout dec_layout(int E, int P, int slots, int K) {
    DecLayout L;
    L.meta = 0;
    L.xc = (uint32_t)align_up((size_t)(4 + E + E + 1 + P) * 4, 128);
    L.total = L.xc + (uint32_t)align_up((size_t)slots * K * 2, 128);
    return L;
}

// shared activation cache: slot s, 8-element block kb = 4*g + wd stored at
// ((s*4 + wd)*G + g)*16 bytes (consecutive groups -> consecutive banks)
__device__ __forceinline__ uint32_t dec_xoff(int slot, int kb, int G) {
    return (uint32_t)(((slot * 4 + (kb & 3)) * G + (kb >> 2)) * 16);
}

__device__ __forceinline__ uint32_t dec_word(const uint4 &w, int i) {
    return i == 0 ? w.x : (i == 1 ? w.y : (i == 2 ? w.z : w.w));
}

// Position of a warp in its work list: task u (RT row units of expert e
// from unit0), token pass tb (activation rows r0+tb .. r0+tb+3) and group
// step gs (groups gs*L*kGPI + ks + L*i, i < kGPI, of every row).
struct Cursor {
    int u, e, unit0, r0, ne, tb, gs;
};

// Registers of one load step: per row unit, matrix and group, the 16-byte
// code word, the scale and the packed zero word.
template <int RU, int NMAT>
struct Step {
    uint4 w[RU][NMAT][kGPI];
    float sc[RU][NMAT][kGPI];
    uint32_t zw[RU][NMAT][kGPI];
};

template <int MODE, int L, int RU>
struct DecTraits {
    static constexpr int nmat = MODE == kDecGateUp ? 2 : 1;
    static constexpr int UPW = 32 / L;  // row units per warp step
    static constexpr int RT = UPW * RU; // row units per task
};

// Moves c to the first valid task at or after u (c.u = t1 when none is left).
template <int MODE, int L, int RU>
__device__ __forceinline__ void cursor_task(Cursor &c, int u, int t1, int TPE, const int *s_active,
                                            const int *s_offs, const DecodeArgs &a, int lane) {
    for (; u < t1; ++u) {
        const int ai = u / TPE;
        const int e = s_active[ai];
        if (e >= 0 && e < a.E) {
            const int r0 = s_offs[e], r1 = s_offs[e + 1];
            if (r0 >= 0 && r1 <= a.P && r1 > r0) {
                c.u = u;
                c.e = e;
                c.unit0 = (u - ai * TPE) * DecTraits<MODE, L, RU>::RT;
                c.r0 = r0;
                c.ne = r1 - r0;
                c.tb = 0;
                c.gs = 0;
                return;
            }
        }
        if (lane == 0) set_error(a.err, MOE_DEVERR_BAD_METADATA);
    }
    c.u = t1;
}

template <int MODE, int L, int RU>
__device__ __forceinline__ void cursor_next(Cursor &c, int t1, int TPE, int nsteps, const int *s_active,
                                            const int *s_offs, const DecodeArgs &a, int lane) {
    if (++c.gs < nsteps) return;
    c.gs = 0;
    c.tb += kDecPass;
    if (c.tb < c.ne) return;
    cursor_task<MODE, L, RU>(c, c.u + 1, t1, TPE, s_active, s_offs, a, lane);
}

// Issue every load of the step at cursor c.  Groups past G and rows past
// the expert load nothing: zero codes, zero point 0 and scale 0.
template <int MODE, int L, int RU>
__device__ __forceinline__ void dec_issue(Step<RU, DecTraits<MODE, L, RU>::nmat> &st, const Cursor &c,
                                          const DecodeArgs &a, int lane) {
    using Tr = DecTraits<MODE, L, RU>;
    const int G = a.K / 32, KW = a.K / 8;
    const int ks = lane % L, us = lane / L;
#pragma unroll
    for (int ru = 0; ru < RU; ++ru) {
        const int unit = c.unit0 + us + ru * Tr::UPW;
#pragma unroll
        for (int b = 0; b < Tr::nmat; ++b) {
            const int n = unit + b * a.rows;  // matrix row
            const size_t row = (size_t)c.e * a.N + n;
            const uint4 *qp = reinterpret_cast<const uint4 *>(a.q + row * KW);
            const __half *sp = a.s + row * G;
            const uint32_t *zp = a.z + ((size_t)c.e * (a.N / 8) + n / 8) * G;
#pragma unroll
            for (int i = 0; i < kGPI; ++i) {
                const int g = c.gs * L * kGPI + ks + L * i;
                const bool ok = unit < a.rows && g < G;
                st.w[ru][b][i] = ok ? ldg_stream(qp + g) : make_uint4(0, 0, 0, 0);
                st.sc[ru][b][i] = ok ? __half2float(__ldg(sp + g)) : 0.f;
                st.zw[ru][b][i] = ok ? __ldg(zp + g) : 0u;
            }
        }
    }
}

// Dequantise the step at cursor c and accumulate against NT activation rows.
// The kGPI groups of every row are worked on together, each product sum in
// up to four independent fp16 chains, to keep enough independent
// instructions in flight.
template <int MODE, int L, int RU, int NT>
__device__ __forceinline__ void dec_compute(const Step<RU, DecTraits<MODE, L, RU>::nmat> &st,
                                            float (&acc)[RU][DecTraits<MODE, L, RU>::nmat][kDecPass],
                                            const Cursor &c, const int *s_pairs, const uint8_t *xcb,
                                            int hbase, bool hc, const DecodeArgs &a, int lane) {
    using Tr = DecTraits<MODE, L, RU>;
    constexpr int nmat = Tr::nmat;
    constexpr int CH = NT == 1 ? 4 : (NT == 2 ? 2 : 1);  // independent chains per product sum
    const int K = a.K, G = K / 32;
    const int ks = lane % L, us = lane / L;
    uint32_t xrow[NT];  // byte offset of each activation row in the cache
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int r = c.r0 + c.tb + t;
        const int p = s_pairs[r];
        const int slot = MODE == kDecGateUp ? ((p >= 0 && p < a.P) ? p / a.k : 0) : r - hbase;
        xrow[t] = (uint32_t)(slot * 4 * G * 16);
    }
#pragma unroll
    for (int ru = 0; ru < RU; ++ru) {
        const int unit = c.unit0 + us + ru * Tr::UPW;
        ZeroPoint zp[nmat][kGPI];
#pragma unroll
        for (int b = 0; b < nmat; ++b)
#pragma unroll
            for (int i = 0; i < kGPI; ++i)
                zp[b][i] = make_zero_point((st.zw[ru][b][i] >> (4 * ((unit + b * a.rows) & 7))) & 0xFu);
        __half2 hs[kGPI][nmat][NT][CH];
#pragma unroll
        for (int i = 0; i < kGPI; ++i)
#pragma unroll
            for (int b = 0; b < nmat; ++b)
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int ch = 0; ch < CH; ++ch) hs[i][b][t][ch] = __float2half2_rn(0.f);
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
            for (int i = 0; i < kGPI; ++i) {
                const int g = c.gs * L * kGPI + ks + L * i;
                const bool gok = g < G;
                __half2 dq[nmat][4];
#pragma unroll
                for (int b = 0; b < nmat; ++b) dequant_word(dec_word(st.w[ru][b][i], wd), zp[b][i], dq[b]);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    // groups past G have zero codes and scale 0; their
                    // activations read as zero so the sums stay finite
                    uint4 X = make_uint4(0, 0, 0, 0);
                    if (gok) {
                        if (MODE == kDecGateUp || hc) {
                            X = *reinterpret_cast<const uint4 *>(xcb + xrow[t] + (uint32_t)((wd * G + g) * 16));
                        } else {
                            X = pair_interleave(__ldg(reinterpret_cast<const uint4 *>(
                                a.vin + (size_t)(c.r0 + c.tb + t) * K + g * 32 + wd * 8)));
                        }
                    }
#pragma unroll
                    for (int b = 0; b < nmat; ++b) {
                        __half2 &h = hs[i][b][t][wd % CH];
                        h = __hfma2(dq[b][0], u32_as_half2(X.x), h);
                        h = __hfma2(dq[b][1], u32_as_half2(X.y), h);
                        h = __hfma2(dq[b][2], u32_as_half2(X.z), h);
                        h = __hfma2(dq[b][3], u32_as_half2(X.w), h);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kGPI; ++i)
#pragma unroll
            for (int b = 0; b < nmat; ++b)
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    __half2 s2 = hs[i][b][t][0];
#pragma unroll
                    for (int ch = 1; ch < CH; ++ch) s2 = __hadd2(s2, hs[i][b][t][ch]);
                    const float2 f = __half22float2(s2);
                    acc[ru][b][t] = fmaf(st.sc[ru][b][i], f.x + f.y, acc[ru][b][t]);
                }
    }
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
        const int unit = c.unit0 + us + ru * Tr::UPW;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int r = c.r0 + c.tb + t;
            const int p = s_pairs[r];
            if (unit < a.rows && (t % L) == ks) {
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

// Step 4, after a task's last pass: count its rows into their 8-row output
// blocks; the warp that completes a block sums each token's k terms in order.
// Every lane's y writes precede lane 0's fence and atomic (__syncwarp), and
// the completing warp fences before reading the other warps' y rows.
__device__ __forceinline__ void dec_combine(int n_lo, int n_hi, int A, const DecodeArgs &a, int lane) {
    __syncwarp();
    for (int nb = n_lo / 8; nb <= (n_hi - 1) / 8; ++nb) {
        const int covered = min(n_hi, nb * 8 + 8) - max(n_lo, nb * 8);
        unsigned old = 0;
        if (lane == 0) {
            __threadfence();
            old = atomicAdd(a.counters + nb, (unsigned)covered);
        }
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old + covered == (unsigned)A * 8u) {
            __threadfence();
            for (int idx = lane; idx < a.T * 8; idx += 32) {
                const int t = idx >> 3, n = nb * 8 + (idx & 7);
                float accv = 0.f;
                for (int jj = 0; jj < a.k; ++jj) {
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

// compute + (at the end of a pass) finish + (at the end of a task) combine
// for the step at cursor c
template <int MODE, int L, int RU>
__device__ __forceinline__ void dec_consume(const Step<RU, DecTraits<MODE, L, RU>::nmat> &st,
                                            float (&acc)[RU][DecTraits<MODE, L, RU>::nmat][kDecPass],
                                            const Cursor &c, int nsteps, const int *s_pairs,
                                            const uint8_t *xcb, int hbase, bool hcached, int A,
                                            const DecodeArgs &a, int lane) {
    using Tr = DecTraits<MODE, L, RU>;
    const int nt = min(kDecPass, c.ne - c.tb);
    const bool hc = hcached && c.r0 >= hbase && c.r0 + c.ne - hbase <= a.slots;
    switch (nt) {
        case 1: dec_compute<MODE, L, RU, 1>(st, acc, c, s_pairs, xcb, hbase, hc, a, lane); break;
        case 2: dec_compute<MODE, L, RU, 2>(st, acc, c, s_pairs, xcb, hbase, hc, a, lane); break;
        case 3: dec_compute<MODE, L, RU, 3>(st, acc, c, s_pairs, xcb, hbase, hc, a, lane); break;
        default: dec_compute<MODE, L, RU, 4>(st, acc, c, s_pairs, xcb, hbase, hc, a, lane); break;
    }
    if (c.gs + 1 < nsteps) return;
    switch (nt) {
        case 1: dec_finish<MODE, L, RU, 1>(acc, c, s_pairs, a, lane); break;
        case 2: dec_finish<MODE, L, RU, 2>(acc, c, s_pairs, a, lane); break;
        case 3: dec_finish<MODE, L, RU, 3>(acc, c, s_pairs, a, lane); break;
        default: dec_finish<MODE, L, RU, 4>(acc, c, s_pairs, a, lane); break;
    }
    if (MODE == kDecDown && c.tb + kDecPass >= c.ne)
        dec_combine(c.unit0, min(c.unit0 + Tr::RT, a.rows), A, a, lane);
}

// Cooperative copy of n activation rows (starting at src) into cache slots
// 0..n-1, pair-interleaved; every thread issues its loads before any store.
__device__ __forceinline__ void dec_stage_rows(const __half *src, int n, int K, int G, uint8_t *xcb,
                                               int tid) {
    const int KB = K / 8, nx = n * KB;
    for (int base = 0; base < nx; base += 4 * kDecThreads) {
        uint4 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int i = base + tid + c * kDecThreads;
            v[c] = i < nx ? __ldg(reinterpret_cast<const uint4 *>(src) + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int i = base + tid + c * kDecThreads;
            if (i < nx) *reinterpret_cast<uint4 *>(xcb + dec_xoff(i / KB, i % KB, G)) = pair_interleave(v[c]);
        }
    }
}

template <int MODE, int L, int RU>
__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(const DecodeArgs a) {
    using Tr = DecTraits<MODE, L, RU>;
    constexpr int nmat = Tr::nmat;
    extern __shared__ __align__(128) uint8_t smem[];
    const int K = a.K, G = K / 32;
    const DecLayout Ly = dec_layout(a.E, a.P, a.slots, K);
    int *s_meta = reinterpret_cast<int *>(smem + Ly.meta);
    int *s_active = s_meta + 4;
    int *s_offs = s_active + a.E;
    int *s_pairs = s_offs + a.E + 1;
    uint8_t *xcb = smem + Ly.xc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_wait();
    pdl_trigger();

    // ---- prologue: metadata (+ every x row in step 3), all loads first
    {
        const int nmeta = a.E + (a.E + 1) + a.P;  // active | offsets | pairs
        for (int base = 0; base < nmeta; base += 4 * kDecThreads) {
            int v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = base + tid + c * kDecThreads;
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
                const int i = base + tid + c * kDecThreads;
                if (i < nmeta) s_active[i] = v[c];  // active, offsets, pairs are contiguous
            }
        }
        if (tid == 0) s_meta[0] = __ldg(a.num_active);
        if (MODE == kDecGateUp) dec_stage_rows(a.vin, a.T, K, G, xcb, tid);
    }
    __syncthreads();

    int A = s_meta[0];
    A = A < 0 ? 0 : (A > a.E ? a.E : A);
    const int TPE = (a.rows + Tr::RT - 1) / Tr::RT;  // tasks per expert
    const long long U = (long long)A * TPE;
    const long long NW = (long long)gridDim.x * kDecWarps;
    const long long gw = (long long)blockIdx.x * kDecWarps + warp;
    const int t0 = (int)(U * gw / NW), t1 = (int)(U * (gw + 1) / NW);
    const int nsteps = (G + L * kGPI - 1) / (L * kGPI);  // group steps per row

    // the first step of this warp goes out before anything else is waited for
    Cursor cur;
    cursor_task<MODE, L, RU>(cur, t0, t1, TPE, s_active, s_offs, a, lane);
    Step<RU, nmat> bA, bB;
    if (cur.u < t1) dec_issue<MODE, L, RU>(bA, cur, a, lane);

    // ---- step 4: cache the h rows of every segment this CTA touches
    int hbase = 0;
    bool hcached = false;
    if (MODE == kDecDown) {
        const int c0 = (int)(U * blockIdx.x * kDecWarps / NW);
        const int c1 = (int)(U * (blockIdx.x + 1) * kDecWarps / NW);
        if (c1 > c0) {
            const int e0 = s_active[c0 / TPE], e1 = s_active[(c1 - 1) / TPE];
            if (e0 >= 0 && e0 < a.E && e1 >= 0 && e1 < a.E) {
                const int R0 = s_offs[e0], R1 = s_offs[e1 + 1];
                if (R0 >= 0 && R0 <= R1 && R1 <= a.P && R1 - R0 <= a.slots) {
                    dec_stage_rows(a.vin + (size_t)R0 * K, R1 - R0, K, G, xcb, tid);
                    hbase = R0;
                    hcached = true;
                }
            }
        }
        __syncthreads();
    }

    // ---- one-step-ahead register pipeline over this warp's work
    float acc[RU][nmat][kDecPass];
#pragma unroll
    for (int ru = 0; ru < RU; ++ru)
#pragma unroll
        for (int b = 0; b < nmat; ++b)
#pragma unroll
            for (int t = 0; t < kDecPass; ++t) acc[ru][b][t] = 0.f;
    while (cur.u < t1) {
        Cursor nxt = cur;
        cursor_next<MODE, L, RU>(nxt, t1, TPE, nsteps, s_active, s_offs, a, lane);
        if (nxt.u < t1) dec_issue<MODE, L, RU>(bB, nxt, a, lane);
        dec_consume<MODE, L, RU>(bA, acc, cur, nsteps, s_pairs, xcb, hbase, hcached, A, a, lane);
        if (nxt.u >= t1) break;
        cur = nxt;
        cursor_next<MODE, L, RU>(nxt, t1, TPE, nsteps, s_active, s_offs, a, lane);
        if (nxt.u < t1) dec_issue<MODE, L, RU>(bA, nxt, a, lane);
        dec_consume<MODE, L, RU>(bB, acc, cur, nsteps, s_pairs, xcb, hbase, hcached, A, a, lane);
        cur = nxt;
    }
}

// ---------------------------------------------------------------- launchers
template <int MODE, int L, int RU>
static cudaError_t launch_decode_t(DecodeArgs a, int num_sms, size_t smem_limit, cudaStream_t stream) {
    const size_t smem = dec_layout(a.E, a.P, a.slots, a.K).total;
    if (smem > smem_limit) return cudaErrorInvalidConfiguration;
    static int configured[128];
    cudaError_t e = ensure_smem(decode_kernel<MODE, L, RU>, configured, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_kernel<MODE, L, RU>, num_sms, kDecThreads, smem, stream, a);
}

// Lanes per row unit: a power of two giving each lane about five groups.
static int lanes_for(int G) { return G >= 40 ? 8 : (G >= 20 ? 4 : (G >= 10 ? 2 : 1)); }

bool decode_supported(int T, int E, int k, int H, int I, size_t smem_limit) {
    const int P = T * k;
    return T >= 1 && T <= kDecMaxT && dec_layout(E, P, T, H).total <= smem_limit &&
           dec_layout(E, P, 4 * T, I).total <= smem_limit;
}

cudaError_t launch_gate_up_decode(const __half *x, const uint32_t *q, const __half *s, const uint32_t *z,
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
    switch (lanes_for(H / 32)) {
        case 8: return launch_decode_t<kDecGateUp, 8, 1>(a, num_sms, smem_limit, stream);
        case 4: return launch_decode_t<kDecGateUp, 4, 1>(a, num_sms, smem_limit, stream);
        case 2: return launch_decode_t<kDecGateUp, 2, 1>(a, num_sms, smem_limit, stream);
        default: return launch_decode_t<kDecGateUp, 1, 1>(a, num_sms, smem_limit, stream);
    }
}

cudaError_t launch_down_decode(const __half *h, const uint32_t *q, const __half *s, const uint32_t *z,
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
    a.slots = 4 * T;  // h rows of a few segments; more fall back to direct reads
    switch (lanes_for(I / 32)) {
        case 8: return launch_decode_t<kDecDown, 8, 2>(a, num_sms, smem_limit, stream);
        case 4: return launch_decode_t<kDecDown, 4, 2>(a, num_sms, smem_limit, stream);
        case 2: return launch_decode_t<kDecDown, 2, 2>(a, num_sms, smem_limit, stream);
        default: return launch_decode_t<kDecDown, 1, 2>(a, num_sms, smem_limit, stream);
    }
}

}  // namespace moe
