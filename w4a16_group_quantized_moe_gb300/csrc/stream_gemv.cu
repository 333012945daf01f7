// stream_gemv.cu -- steps 3 and 4 for the batches that neither the decode
// kernels' shared-memory layout nor one 128-row tensor-core chunk fits (on
// the Qwen4Exp geometry 11-12 tokens): the weight-streaming expert
// projections.
//
// With few tokens per expert ("2-8 input tokens", "[Perf][SM70] Narrow
// Qwen3.8 AWQ active grouped decode", section Purpose) the layer is bound
// by reading the active experts' packed weights once from HBM.  The kernel
// is built around that stream:
//
//  * Work is the list of active experts' rows (gate/up row pairs for step 3,
//    output rows for step 4), flattened expert-major and cut into one
//    contiguous, equal-length range per CTA (one persistent CTA per SM), so
//    every SM streams the same number of bytes whatever the segment sizes.
//  * One producer thread moves each stage (<= RS rows of one expert: int4
//    codes, fp16 scales, packed zeros) into a shared-memory ring with bulk
//    asynchronous copies completing on an mbarrier; consumer warps release a
//    stage with a second mbarrier.  Several stages stay in flight per SM.
//  * Consumers: S lanes per row, each lane owns groups g = ks, ks+S, ... .
//    A 16-byte load is exactly one 32-code group.  Codes become fp16
//    (code - zero) pairs without conversions (common.cuh), are multiplied by
//    the activations in fp16 within the group, and each group sum is scaled
//    and accumulated in fp32.  S-lane shuffles finish the dot products.
//  * Activations (x rows for step 3, h rows for step 4) sit in a small
//    shared cache, pair-interleaved to match the dequantised codes.  For
//    T <= 8 every x row is cached once per CTA.
//  * Step 4 writes each pair's fp32 projection y_p to the workspace.  For
//    T <= 8 the weighted combine is fused: each 8-row output block counts
//    arriving rows in a workspace counter, and whoever completes a block
//    sums its tokens' k terms in order and writes fp16 (no ordering races,
//    no extra launch).  Larger T uses combine_kernel.
#include "common.cuh"

namespace moe {

enum { kGateUp = 0, kDown = 1 };

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kStreamThreads = kConsumerThreads + 32;
constexpr int kXSlots = 8;
constexpr int kMaxStages = 4;
constexpr int kConsumerBarrier = 1;

struct StreamArgs {
    const uint32_t *q;   // packed codes  [E][N][K/8]
    const __half *s;     // scales        [E][N][K/32]
    const uint32_t *z;   // packed zeros  [E][N/8][K/32]
    int E, N, K;         // N: matrix rows per expert, K: reduction length
    int rows;            // work rows per expert: I (row pairs) or H
    const __half *vin;   // step 3: x [T][K]; step 4: h [P][K]
    int T, k, P;
    const int32_t *offsets, *sorted_pair, *active, *num_active;
    __half *h_out;       // step 3: [P][I]
    float *y_out;        // step 4: [P][H]
    const float *topk_w; // step 4, fused combine
    __half *out;         // step 4, fused combine: [T][H]
    uint32_t *counters;  // step 4, fused combine: [H/8]
    int fuse_combine;
    uint32_t *err;
    int nstages;
};

// Shared-memory geometry of one stage: nmat blocks (gate, up | down) of
// RS rows: codes, then scales, then zero words.  Scale and zero copies are
// widened to 16-byte boundaries, hence the slack.
struct StageGeom {
    uint32_t q_bytes, s_bytes, z_bytes, bytes;
};

template <int MODE, int S>
__host__ __device__ inline StageGeom stage_geom(int K) {
    constexpr int RS = kConsumerThreads / S;
    constexpr int nmat = MODE == kGateUp ? 2 : 1;
    const int G = K / 32;
    StageGeom g;
    g.q_bytes = (uint32_t)(RS * K / 2);
    g.s_bytes = (uint32_t)align_up((size_t)RS * G * 2 + 32, 16);
    g.z_bytes = (uint32_t)align_up((size_t)(RS / 8 + 2) * G * 4 + 32, 16);
    g.bytes = (uint32_t)align_up((size_t)nmat * (g.q_bytes + g.s_bytes + g.z_bytes), 128);
    return g;
}

__host__ __device__ inline size_t xcache_bytes(int K) { return align_up((size_t)kXSlots * K * 2, 128); }

// Byte ranges (from the tensor bases) a stage block copies, widened to 16.
struct BlockCopy {
    size_t q_off;        // bytes from q base
    uint32_t q_len;
    size_t s_lo, s_a;    // exact start, aligned start
    uint32_t s_len;      // aligned length
    size_t z_lo, z_a;
    uint32_t z_len;
    int zrow0;           // first zero row (n_first / 8)
};

__device__ inline BlockCopy block_copy(int e, int n_first, int cnt, int N, int K) {
    const int G = K / 32;
    BlockCopy c;
    const size_t row = (size_t)e * N + n_first;
    c.q_off = row * (size_t)(K / 2);
    c.q_len = (uint32_t)(cnt * (K / 2));
    c.s_lo = row * G * 2;
    const size_t s_hi = (row + cnt) * G * 2;
    c.s_a = c.s_lo & ~(size_t)15;
    c.s_len = (uint32_t)(align_up(s_hi, 16) - c.s_a);
    c.zrow0 = n_first / 8;
    const size_t zr0 = (size_t)e * (N / 8) + n_first / 8;
    const size_t zr1 = (size_t)e * (N / 8) + (n_first + cnt - 1) / 8;
    c.z_lo = zr0 * G * 4;
    c.z_a = c.z_lo & ~(size_t)15;
    c.z_len = (uint32_t)(align_up((zr1 + 1) * G * 4, 16) - c.z_a);
    return c;
}

// One unit of the CTA's work list.
struct StageDesc {
    int e, n0, cnt, r0, ne;
    bool valid;
};

__device__ inline StageDesc next_stage(const StreamArgs &a, long long &f, long long f1, int RS) {
    StageDesc d;
    const int ai = (int)(f / a.rows);
    d.n0 = (int)(f % a.rows);
    long long c = RS;
    if (c > a.rows - d.n0) c = a.rows - d.n0;
    if (c > f1 - f) c = f1 - f;
    d.cnt = (int)c;
    f += c;
    d.e = __ldg(a.active + ai);
    d.valid = d.e >= 0 && d.e < a.E;
    d.r0 = d.ne = 0;
    if (d.valid) {
        d.r0 = __ldg(a.offsets + d.e);
        const int r1 = __ldg(a.offsets + d.e + 1);
        d.ne = r1 - d.r0;
        d.valid = d.r0 >= 0 && r1 <= a.P && d.ne > 0;
    }
    return d;
}

template <int MODE, int S>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_kernel(const StreamArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int RS = kConsumerThreads / S;
    constexpr int nmat = MODE == kGateUp ? 2 : 1;
    const int K = a.K, G = K / 32;
    const StageGeom geom = stage_geom<MODE, S>(K);
    __half *xc = reinterpret_cast<__half *>(smem);
    uint8_t *stages = smem + xcache_bytes(K);
    uint64_t *full = reinterpret_cast<uint64_t *>(stages + (size_t)a.nstages * geom.bytes);
    uint64_t *empty = full + kMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kMaxStages);
    const int NST = a.nstages;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    pdl_wait();
    pdl_trigger();
    __syncthreads();

    int A = __ldg(a.num_active);
    A = A < 0 ? 0 : (A > a.E ? a.E : A);
    const long long Wtot = (long long)A * a.rows;
    const long long f0 = Wtot * blockIdx.x / gridDim.x;
    const long long f1 = Wtot * (blockIdx.x + 1) / gridDim.x;

    // ------------------------------------------------------------ producer
    if (warp == kConsumerWarps) {
        if (lane != 0) return;
        long long f = f0;
        int sidx = 0;
        bool ok = true;
        while (f < f1 && ok) {
            const StageDesc d = next_stage(a, f, f1, RS);
            if (!d.valid) {
                set_error(a.err, MOE_DEVERR_BAD_METADATA);
                continue;
            }
            const int slot = sidx % NST;
            if (sidx >= NST && !mbar_wait_bounded(&empty[slot], ((sidx / NST) - 1) & 1, abort_flag)) {
                set_error(a.err, MOE_DEVERR_WAIT_TIMEOUT);
                *abort_flag = 1;
                ok = false;
                break;
            }
            uint8_t *st = stages + (size_t)slot * geom.bytes;
            BlockCopy bc[nmat];
            uint32_t tx = 0;
#pragma unroll
            for (int b = 0; b < nmat; ++b) {
                bc[b] = block_copy(d.e, d.n0 + b * a.rows, d.cnt, a.N, K);
                tx += bc[b].q_len + bc[b].s_len + bc[b].z_len;
            }
            mbar_arrive_expect_tx(&full[slot], tx);
#pragma unroll
            for (int b = 0; b < nmat; ++b) {
                bulk_g2s(st + b * geom.q_bytes, reinterpret_cast<const uint8_t *>(a.q) + bc[b].q_off,
                         bc[b].q_len, &full[slot]);
                bulk_g2s(st + nmat * geom.q_bytes + b * geom.s_bytes,
                         reinterpret_cast<const uint8_t *>(a.s) + bc[b].s_a, bc[b].s_len, &full[slot]);
                bulk_g2s(st + nmat * (geom.q_bytes + geom.s_bytes) + b * geom.z_bytes,
                         reinterpret_cast<const uint8_t *>(a.z) + bc[b].z_a, bc[b].z_len, &full[slot]);
            }
            ++sidx;
        }
        // never leave while copies into this CTA's shared memory are in flight
        for (int i = sidx - NST < 0 ? 0 : sidx - NST; i < sidx; ++i)
            if (!mbar_wait_bounded(&full[i % NST], (i / NST) & 1, nullptr))
                set_error(a.err, MOE_DEVERR_WAIT_TIMEOUT);
        return;
    }

    // ------------------------------------------------------------ consumers
    const int ct = tid;  // 0 .. kConsumerThreads-1
    const int j = ct / S, ks = ct % S;
    const int cw = warp;
    const int KB = K / 8;  // 16-byte blocks per activation row
    const bool all_tokens = (MODE == kGateUp) && a.T <= kXSlots;

    if (all_tokens) {
        for (int idx = ct; idx < a.T * KB; idx += kConsumerThreads) {
            const int t = idx / KB, b = idx % KB;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.vin + (size_t)t * K) + b);
            reinterpret_cast<uint4 *>(xc + (size_t)t * K)[b] = pair_interleave(v);
        }
        named_barrier(kConsumerBarrier, kConsumerThreads);
    }

    int cached_e = -1, cached_tb = -1;
    bool dead = false;
    long long f = f0;
    int sidx = 0;
    while (f < f1) {
        const StageDesc d = next_stage(a, f, f1, RS);
        if (!d.valid) continue;
        const int slot = sidx % NST;
        if (!dead && !mbar_wait_bounded(&full[slot], (sidx / NST) & 1, abort_flag)) {
            dead = true;
            if (ct == 0) set_error(a.err, MOE_DEVERR_WAIT_TIMEOUT);
            *abort_flag = 1;
        }
        const uint8_t *st = stages + (size_t)slot * geom.bytes;
        const bool row_ok = j < d.cnt;

        for (int tb = 0; tb < d.ne; tb += kXSlots) {
            const int nt = min(kXSlots, d.ne - tb);
            int pid[kXSlots], xs[kXSlots];
#pragma unroll
            for (int tt = 0; tt < kXSlots; ++tt) {
                int p = -1;
                if (tt < nt) {
                    p = __ldg(a.sorted_pair + d.r0 + tb + tt);
                    if (p < 0 || p >= a.P) {
                        if (ct == 0) set_error(a.err, MOE_DEVERR_BAD_METADATA);
                        p = -1;
                    }
                }
                pid[tt] = p;
                xs[tt] = (all_tokens && p >= 0) ? p / a.k : tt;
            }
            if (!all_tokens && (cached_e != d.e || cached_tb != tb)) {
                named_barrier(kConsumerBarrier, kConsumerThreads);
                for (int idx = ct; idx < nt * KB; idx += kConsumerThreads) {
                    const int tt = idx / KB, b = idx % KB;
                    const int p = __ldg(a.sorted_pair + d.r0 + tb + tt);
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (p >= 0 && p < a.P) {
                        const __half *src = MODE == kGateUp ? a.vin + (size_t)(p / a.k) * K
                                                            : a.vin + (size_t)(d.r0 + tb + tt) * K;
                        v = __ldg(reinterpret_cast<const uint4 *>(src) + b);
                    }
                    reinterpret_cast<uint4 *>(xc + (size_t)tt * K)[b] = pair_interleave(v);
                }
                named_barrier(kConsumerBarrier, kConsumerThreads);
                cached_e = d.e;
                cached_tb = tb;
            }

            float acc0[kXSlots], acc1[kXSlots];
#pragma unroll
            for (int tt = 0; tt < kXSlots; ++tt) acc0[tt] = acc1[tt] = 0.f;

            if (row_ok && !dead) {
#pragma unroll
                for (int b = 0; b < nmat; ++b) {
                    const int n_first = d.n0 + b * a.rows;
                    const BlockCopy bc = block_copy(d.e, n_first, d.cnt, a.N, K);
                    const uint8_t *qb = st + b * geom.q_bytes + (size_t)j * (K / 2);
                    const uint8_t *sb = st + nmat * geom.q_bytes + b * geom.s_bytes + (bc.s_lo - bc.s_a) +
                                        (size_t)j * G * 2;
                    const uint8_t *zb = st + nmat * (geom.q_bytes + geom.s_bytes) + b * geom.z_bytes +
                                        (bc.z_lo - bc.z_a) +
                                        (size_t)((n_first + j) / 8 - bc.zrow0) * G * 4;
                    const int zshift = 4 * ((n_first + j) & 7);
                    float accb[kXSlots];
#pragma unroll
                    for (int tt = 0; tt < kXSlots; ++tt) accb[tt] = 0.f;
                    for (int g = ks; g < G; g += S) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(qb + (size_t)g * 16);
                        const float sc = __half2float(*reinterpret_cast<const __half *>(sb + g * 2));
                        const uint32_t zw = *reinterpret_cast<const uint32_t *>(zb + g * 4);
                        const ZeroPoint zp = make_zero_point((zw >> zshift) & 0xFu);
                        __half2 dq[16];
                        dequant_word(w.x, zp, dq + 0);
                        dequant_word(w.y, zp, dq + 4);
                        dequant_word(w.z, zp, dq + 8);
                        dequant_word(w.w, zp, dq + 12);
#pragma unroll
                        for (int tt = 0; tt < kXSlots; ++tt) {
                            if (tt < nt) {
                                const uint4 *xp =
                                    reinterpret_cast<const uint4 *>(xc + (size_t)xs[tt] * K + g * 32);
                                __half2 hs = __float2half2_rn(0.f);
#pragma unroll
                                for (int wd = 0; wd < 4; ++wd) {
                                    const uint4 X = xp[wd];
                                    hs = __hfma2(dq[4 * wd + 0], u32_as_half2(X.x), hs);
                                    hs = __hfma2(dq[4 * wd + 1], u32_as_half2(X.y), hs);
                                    hs = __hfma2(dq[4 * wd + 2], u32_as_half2(X.z), hs);
                                    hs = __hfma2(dq[4 * wd + 3], u32_as_half2(X.w), hs);
                                }
                                const float2 fs = __half22float2(hs);
                                accb[tt] = fmaf(sc, fs.x + fs.y, accb[tt]);
                            }
                        }
                    }
#pragma unroll
                    for (int tt = 0; tt < kXSlots; ++tt) {
                        if (b == 0)
                            acc0[tt] = accb[tt];
                        else
                            acc1[tt] = accb[tt];
                    }
                }
            }

            // finish the dot products across the S lanes of each row
#pragma unroll
            for (int tt = 0; tt < kXSlots; ++tt) {
                if (tt < nt) {
#pragma unroll
                    for (int off = S / 2; off > 0; off >>= 1) {
                        acc0[tt] += __shfl_xor_sync(0xffffffffu, acc0[tt], off);
                        if (MODE == kGateUp) acc1[tt] += __shfl_xor_sync(0xffffffffu, acc1[tt], off);
                    }
                }
            }
            if (row_ok && !dead) {
#pragma unroll
                for (int tt = 0; tt < kXSlots; ++tt) {
                    if (tt < nt && (tt % S) == ks && pid[tt] >= 0) {
                        if (MODE == kGateUp) {
                            const float gv = acc0[tt], uv = acc1[tt];
                            const float hv = gv / (1.0f + __expf(-gv)) * uv;
                            a.h_out[(size_t)(d.r0 + tb + tt) * a.rows + d.n0 + j] = __float2half_rn(hv);
                        } else {
                            a.y_out[(size_t)pid[tt] * a.N + d.n0 + j] = acc0[tt];
                        }
                    }
                }
            }
        }

        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);

        if (MODE == kDown && a.fuse_combine) {
            // rows of this stage are written; count them into their 8-row blocks
            __threadfence();
            named_barrier(kConsumerBarrier, kConsumerThreads);
            const int nb_first = d.n0 / 8, nb_last = (d.n0 + d.cnt - 1) / 8;
            for (int nb = nb_first + cw; nb <= nb_last; nb += kConsumerWarps) {
                const int covered = min(d.n0 + d.cnt, nb * 8 + 8) - max(d.n0, nb * 8);
                unsigned old = 0;
                if (lane == 0 && !dead) old = atomicAdd(a.counters + nb, (unsigned)covered);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (!dead && old + covered == (unsigned)A * 8u) {
                    __threadfence();
                    for (int idx = lane; idx < a.T * 8; idx += 32) {
                        const int t = idx >> 3, n = nb * 8 + (idx & 7);
                        float acc = 0.f;
                        for (int jj = 0; jj < a.k; ++jj) {
                            const int p = t * a.k + jj;
                            acc = fmaf(__ldg(a.topk_w + p), __ldcg(a.y_out + (size_t)p * a.N + n), acc);
                        }
                        a.out[(size_t)t * a.N + n] = __float2half_rn(acc);
                    }
                    __syncwarp();
                    if (lane == 0) atomicExch(a.counters + nb, 0u);
                }
            }
        }
        ++sidx;
    }
}

// out[t][n] = sum_j topk_w[t][j] * y[t*k+j][n], j in order; 8 outputs/thread.
__global__ void combine_kernel(const float *__restrict__ y, const float *__restrict__ topk_w, int T,
                               int k, int H, __half *__restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int HB = H / 8;
    if (idx >= (long long)T * HB) return;
    const int t = (int)(idx / HB), nb = (int)(idx % HB);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int jj = 0; jj < k; ++jj) {
        const int p = t * k + jj;
        const float w = __ldg(topk_w + p);
        const float4 *yp = reinterpret_cast<const float4 *>(y + (size_t)p * H + nb * 8);
        const float4 v0 = __ldcg(yp), v1 = __ldcg(yp + 1);
        acc[0] = fmaf(w, v0.x, acc[0]);
        acc[1] = fmaf(w, v0.y, acc[1]);
        acc[2] = fmaf(w, v0.z, acc[2]);
        acc[3] = fmaf(w, v0.w, acc[3]);
        acc[4] = fmaf(w, v1.x, acc[4]);
        acc[5] = fmaf(w, v1.y, acc[5]);
        acc[6] = fmaf(w, v1.z, acc[6]);
        acc[7] = fmaf(w, v1.w, acc[7]);
    }
    uint4 o;
    __half2 h0 = __floats2half2_rn(acc[0], acc[1]), h1 = __floats2half2_rn(acc[2], acc[3]);
    __half2 h2 = __floats2half2_rn(acc[4], acc[5]), h3 = __floats2half2_rn(acc[6], acc[7]);
    o.x = *reinterpret_cast<uint32_t *>(&h0);
    o.y = *reinterpret_cast<uint32_t *>(&h1);
    o.z = *reinterpret_cast<uint32_t *>(&h2);
    o.w = *reinterpret_cast<uint32_t *>(&h3);
    reinterpret_cast<uint4 *>(out + (size_t)t * H)[nb] = o;
}

cudaError_t launch_combine(const float *y, const float *topk_w, int T, int k, int H, __half *out,
                           cudaStream_t stream) {
    const long long n = (long long)T * (H / 8);
    return launch_pdl(combine_kernel, (unsigned)((n + 255) / 256), 256, 0, stream, y, topk_w, T, k, H, out);
}

// ---------------------------------------------------------------- launchers
template <int MODE, int S>
static cudaError_t launch_stream_t(StreamArgs a, int num_sms, size_t smem_limit, cudaStream_t stream) {
    constexpr int RS = kConsumerThreads / S;
    const StageGeom geom = stage_geom<MODE, S>(a.K);
    const size_t fixed = xcache_bytes(a.K) + 2 * kMaxStages * sizeof(uint64_t) + 16;
    if (fixed + geom.bytes > smem_limit) return cudaErrorInvalidConfiguration;
    int nst = (int)((smem_limit - fixed) / geom.bytes);
    nst = nst > kMaxStages ? kMaxStages : nst;
    a.nstages = nst;
    const size_t smem = fixed + (size_t)nst * geom.bytes;
    static int configured[128];
    cudaError_t e = ensure_smem(stream_kernel<MODE, S>, configured, smem);
    if (e != cudaSuccess) return e;
    const long long amax = a.E < a.P ? a.E : a.P;
    const long long units = (amax * a.rows + RS - 1) / RS;
    const int grid = (int)(units < num_sms ? (units < 1 ? 1 : units) : num_sms);
    return launch_pdl(stream_kernel<MODE, S>, grid, kStreamThreads, smem, stream, a);
}

cudaError_t launch_gate_up_stream(const __half *x, const uint32_t *q, const __half *s,
                                  const uint32_t *z, const int32_t *offsets,
                                  const int32_t *sorted_pair, const int32_t *active,
                                  const int32_t *num_active, int T, int E, int k, int H, int I,
                                  __half *h, uint32_t *err, int num_sms, size_t smem_limit,
                                  cudaStream_t stream) {
    StreamArgs a{};
    a.q = q; a.s = s; a.z = z;
    a.E = E; a.N = 2 * I; a.K = H; a.rows = I;
    a.vin = x; a.T = T; a.k = k; a.P = T * k;
    a.offsets = offsets; a.sorted_pair = sorted_pair; a.active = active; a.num_active = num_active;
    a.h_out = h; a.err = err;
    if (H / 32 >= 32) return launch_stream_t<kGateUp, 16>(a, num_sms, smem_limit, stream);
    return launch_stream_t<kGateUp, 4>(a, num_sms, smem_limit, stream);
}

cudaError_t launch_down_stream(const __half *h, const uint32_t *q, const __half *s, const uint32_t *z,
                               const int32_t *offsets, const int32_t *sorted_pair,
                               const int32_t *active, const int32_t *num_active, const float *topk_w,
                               int T, int E, int k, int H, int I, __half *out, float *y,
                               uint32_t *counters, uint32_t *err, int num_sms, size_t smem_limit,
                               cudaStream_t stream) {
    StreamArgs a{};
    a.q = q; a.s = s; a.z = z;
    a.E = E; a.N = H; a.K = I; a.rows = H;
    a.vin = h; a.T = T; a.k = k; a.P = T * k;
    a.offsets = offsets; a.sorted_pair = sorted_pair; a.active = active; a.num_active = num_active;
    a.y_out = y; a.topk_w = topk_w; a.out = out; a.counters = counters;
    a.fuse_combine = T <= kXSlots;
    a.err = err;
    cudaError_t e;
    if (I / 32 >= 32)
        e = launch_stream_t<kDown, 16>(a, num_sms, smem_limit, stream);
    else
        e = launch_stream_t<kDown, 4>(a, num_sms, smem_limit, stream);
    if (e != cudaSuccess || a.fuse_combine) return e;
    const long long n = (long long)T * (H / 8);
    return launch_pdl(combine_kernel, (unsigned)((n + 255) / 256), 256, 0, stream,
                      (const float *)y, topk_w, T, k, H, out);
}

}  // namespace moe
