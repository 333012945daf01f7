// router.cu -- the router's logits, the step ahead of routing:
//     logits[t][e] = sum over h of x[t][h] * wr[e][h]
// with x fp16 [T][H] and the router matrix wr fp16 [E][H] (the gate of the
// "Sparse MoE layer": a bias-free linear map from the hidden state to one
// score per expert), products of fp16 values exact in fp32, sums in fp32.
//
// Two kernels:
//   router_gemv_kernel  decode batches (T <= 16).  The router matrix (2.6 MB
//       at E = 512, H = 2560) is the only real traffic, so this is a GEMV
//       bound by HBM and by latency: the CTA first stages the batch's x
//       rows in shared memory (one round trip, every thread's loads in
//       flight together), then one warp per expert row requests all of its
//       lane's 16-byte chunks of the row at once and multiplies them by the
//       T activation chunks at the same K offsets.  With `fused`, the last
//       CTA to finish (found by an atomic ticket after a release fence; no
//       CTA ever waits for another) also routes every token and groups the
//       pairs, so logits, top-k and segments come out of one launch.
//   router_tc_kernel    larger batches: a dense contraction on the tcgen05
//       tensor cores.  One CTA per 128-token x 128-expert tile; warp 0 copies
//       the x and router tiles of each 64-wide K block by TMA (128-byte
//       swizzle) into a 4-stage ring, warp 1 issues the MMAs (M = 128
//       tokens, N = 128 experts, fp32 accumulator in tensor memory), warps
//       2-5 read the accumulator and store fp32 logit rows.  Every wait is
//       bounded.
#include "align.cuh"
#include "route.cuh"
#include "tc_common.cuh"

namespace moe {

constexpr int kRgThreads = 256;  // GEMV block: 8 warps, one expert row each
constexpr int kRgMaxT = 16;      // tokens the GEMV path takes
constexpr int kRgChunks = 12;    // 16-byte row chunks a lane requests at once (H <= 3072 in one round)
constexpr size_t kRgStageMax = 96 * 1024;  // x rows staged in shared memory up to this size

// ---------------------------------------------------------------- GEMV
__device__ __forceinline__ float dot8(uint4 w, uint4 x) {
    const __half2 *wh = reinterpret_cast<const __half2 *>(&w);
    const __half2 *xh = reinterpret_cast<const __half2 *>(&x);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 a = __half22float2(wh[i]), b = __half22float2(xh[i]);
        s = fmaf(a.x, b.x, s);
        s = fmaf(a.y, b.y, s);
    }
    return s;
}

// x rows into shared memory, all loads issued before the stores
__device__ __forceinline__ void stage_x(const uint4 *__restrict__ x, int n, uint4 *xs) {
    for (int base = 0; base < n; base += 8 * blockDim.x) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * blockDim.x + threadIdx.x;
            v[u] = i < n ? __ldg(x + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * blockDim.x + threadIdx.x;
            if (i < n) xs[i] = v[u];
        }
    }
}

// x: the staged rows (shared memory) or, past kRgStageMax, global memory
template <int TM>
__device__ __forceinline__ void router_rows(const uint4 *__restrict__ x, const uint4 *__restrict__ wr, int T, int E,
                                            int H8, float *__restrict__ logits) {
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int e = blockIdx.x * wpb + (threadIdx.x >> 5); e < E; e += gridDim.x * wpb) {
        const uint4 *row = wr + (size_t)e * H8;
        float acc[TM];
#pragma unroll
        for (int t = 0; t < TM; ++t) acc[t] = 0.f;
        for (int c0 = 0; c0 < H8; c0 += 32 * kRgChunks) {
            uint4 w[kRgChunks];
#pragma unroll
            for (int u = 0; u < kRgChunks; ++u) {
                const int c = c0 + 32 * u + lane;
                w[u] = c < H8 ? ldg_stream(row + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kRgChunks; ++u) {
                const int c = c0 + 32 * u + lane;
                if (c < H8) {
#pragma unroll
                    for (int t = 0; t < TM; ++t)
                        if (t < T) acc[t] += dot8(w[u], x[(size_t)t * H8 + c]);
                }
            }
        }
        float mine = 0.f;
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            float v = acc[t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == t) mine = v;
        }
        if (lane < T) logits[(size_t)lane * E + e] = mine;
    }
}

struct RouterArgs {
    const uint4 *x, *wr;
    int T, E, k, H8, WS;
    float *logits;
    int32_t *ids;
    float *w;
    int32_t *offsets, *sorted, *active, *num_active;
    uint32_t *ctrl;  // workspace control block (error word, completion ticket)
    int fused;
};

template <int TM>
__global__ void __launch_bounds__(kRgThreads) router_gemv_kernel(const RouterArgs a) {
    extern __shared__ uint4 rg_smem4[];
    __shared__ int s_last;
    pdl_wait();
    pdl_trigger();
    const int nx = a.T * a.H8;
    const bool staged = (size_t)nx * 16 <= kRgStageMax;
    if (staged) {
        stage_x(a.x, nx, rg_smem4);
        __syncthreads();
    }
    router_rows<TM>(staged ? rg_smem4 : a.x, a.wr, a.T, a.E, a.H8, a.logits);
    if (!a.fused) return;
    // release this thread's logits, then take a ticket; the CTA with the
    // last ticket sees every CTA's logits
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(a.ctrl + kCtrlRouterTicket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int P = a.T * a.k;
    int *s_ids = reinterpret_cast<int *>(rg_smem4 + (staged ? nx : 0));  // [P], after the staged x rows
    int *s_align = s_ids + ((P + 31) & ~31);                     // align_block scratch
    uint32_t *s_key = reinterpret_cast<uint32_t *>(s_align + align_smem_ints(a.WS, a.E));  // [warps][E]
    for (int t = warp; t < a.T; t += nwarps)
        route_token_compact<true>(a.logits + (size_t)t * a.E, a.E, a.k, t, a.ids, a.w, s_ids, nullptr,
                                  s_key + (size_t)warp * a.E);
    __syncthreads();
    align_block(s_ids, P, a.E, a.WS, a.offsets, a.sorted, a.active, a.num_active, a.ctrl + kCtrlErrorWord,
                s_align);
    if (threadIdx.x == 0) a.ctrl[kCtrlRouterTicket] = 0;  // ready for the next call on this workspace
}

// shared memory of a GEMV launch: the staged x rows (when they fit the
// staging budget), then, for the fused launch, the routing and grouping
static size_t x_stage_bytes(int T, int H) {
    const size_t b = (size_t)T * H * 2;
    return b <= kRgStageMax ? b : 0;
}

static size_t gemv_smem(int T, int E, int k, int H, bool fused) {
    size_t b = x_stage_bytes(T, H);
    if (fused) {
        const int P = T * k, WS = align_slices(P);
        const int rw = T < kRgThreads / 32 ? T : kRgThreads / 32;
        b += (((size_t)(P + 31) & ~(size_t)31) + align_smem_ints(WS, E) + (size_t)rw * E) * sizeof(int);
    }
    return b;
}

bool router_fusable(int T, int E, int k, int H, size_t smem_limit) {
    return T >= 1 && T <= kRgMaxT && 32 * align_slices(T * k) <= kRgThreads &&
           gemv_smem(T, E, k, H, true) <= smem_limit;
}

static cudaError_t launch_gemv(const RouterArgs &a, int num_sms, cudaStream_t stream) {
    const int wpb = kRgThreads / 32;
    int grid = (a.E + wpb - 1) / wpb;
    if (grid > 4 * num_sms) grid = 4 * num_sms;
    const size_t smem = gemv_smem(a.T, a.E, a.k, 8 * a.H8, a.fused != 0);
    static int configured[5][128];
#define MOE_RG(TM, IDX)                                                                          \
    do {                                                                                         \
        cudaError_t e = ensure_smem(router_gemv_kernel<TM>, configured[IDX], smem);              \
        if (e != cudaSuccess) return e;                                                          \
        return launch_pdl(router_gemv_kernel<TM>, grid, kRgThreads, smem, stream, a);            \
    } while (0)
    if (a.T <= 1) MOE_RG(1, 0);
    if (a.T <= 2) MOE_RG(2, 1);
    if (a.T <= 4) MOE_RG(4, 2);
    if (a.T <= 8) MOE_RG(8, 3);
    MOE_RG(16, 4);
#undef MOE_RG
}

// ---------------------------------------------------------------- tcgen05 GEMM
constexpr int kRtThreads = 192;  // warp 0 copies, warp 1 MMA, warps 2-5 epilogue
constexpr int kRtM = 128;        // tokens per tile (MMA M)
constexpr int kRtN = 128;        // experts per tile (MMA N)
constexpr int kRtKB = 64;        // K per stage: one 128-byte row of fp16
constexpr int kRtStages = 4;
constexpr uint32_t kRtTileBytes = kRtM * kRtKB * 2;  // 16 KB (x tile; the router tile is the same size)
constexpr uint32_t kRtStageBytes = 2 * kRtTileBytes;
constexpr uint32_t kRtTmemCols = kRtN;
static_assert(kRtM == kRtN, "one tile size for both operands");

struct RtCtrl {
    uint64_t full[kRtStages], freeb[kRtStages], acc, drain;
    uint32_t tmem;
    int abort;
};

constexpr size_t kRtSmem = 1024 + (size_t)kRtStages * kRtStageBytes + sizeof(RtCtrl);

__global__ void __launch_bounds__(kRtThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap, int T,
                     int E, int H, float *__restrict__ logits, uint32_t *err) {
    extern __shared__ uint8_t rt_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(rt_smem_raw) + 1023) & ~(uintptr_t)1023);
    RtCtrl *ctl = reinterpret_cast<RtCtrl *>(smem + (size_t)kRtStages * kRtStageBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * kRtM, n0 = blockIdx.y * kRtN;
    const int nkb = (H + kRtKB - 1) / kRtKB;
    if (tid == 0) {
        for (int s = 0; s < kRtStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->freeb[s], 1);
        }
        mbar_init(&ctl->acc, 1);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&ctl->tmem)),
                     "r"(kRtTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    volatile int *abort_flag = &ctl->abort;
    pdl_wait();
    pdl_trigger();
    auto fail = [&]() {
        set_error(err, MOE_DEVERR_WAIT_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kRtStages;
                const uint32_t ph = (uint32_t)(kb / kRtStages) & 1u;
                if (!mbar_wait_bounded(&ctl->freeb[s], ph ^ 1u, abort_flag)) {
                    if (!*abort_flag) fail();
                    break;
                }
                uint8_t *stg = smem + (size_t)s * kRtStageBytes;
                mbar_arrive_expect_tx(&ctl->full[s], kRtStageBytes);
                tma_load_2d(stg, &xmap, kb * kRtKB, m0, &ctl->full[s]);
                tma_load_2d(stg + kRtTileBytes, &wmap, kb * kRtKB, n0, &ctl->full[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc_idesc(kRtM, kRtN);
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kRtStages;
                const uint32_t ph = (uint32_t)(kb / kRtStages) & 1u;
                if (!mbar_wait_bounded(&ctl->full[s], ph, abort_flag)) {
                    if (!*abort_flag) fail();
                    break;
                }
                tc_fence_after();
                // a K step of 16 advances each descriptor's start address by 32 bytes
                const uint64_t ad = tc_desc_sw128(smem_addr(smem + (size_t)s * kRtStageBytes));
                const uint64_t bd = tc_desc_sw128(smem_addr(smem + (size_t)s * kRtStageBytes + kRtTileBytes));
#pragma unroll
                for (int ks = 0; ks < kRtKB / 16; ++ks)
                    tc_mma(tmem, ad + (uint64_t)(ks * 2), bd + (uint64_t)(ks * 2), idesc, (kb | ks) != 0);
                tc_commit(&ctl->freeb[s]);
            }
            tc_commit(&ctl->acc);
            // every MMA issued has completed before tensor memory is released
            tc_commit(&ctl->drain);
            mbar_wait_bounded(&ctl->drain, 0, nullptr);
        }
    } else {
        // lane m of the accumulator holds token m0 + m, column n expert n0 + n
        const int q = warp & 3;  // tensor-memory lane quadrant this warp may read
        const int row = m0 + q * 32 + lane;
        if (__all_sync(0xffffffffu, mbar_wait_bounded(&ctl->acc, 0, abort_flag))) {
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
            float *dst = logits + (size_t)row * E + n0;
            const bool vec = (E & 3) == 0 && n0 + kRtN <= E;
#pragma unroll 1
            for (int c0 = 0; c0 < kRtN; c0 += 16) {
                uint32_t r[16];
                tc_ld16(taddr + (uint32_t)c0, r);
                tc_wait_ld();
                if (row < T) {
                    if (vec) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4 *>(dst + c0 + j) =
                                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (n0 + c0 + j < E) dst[c0 + j] = __uint_as_float(r[j]);
                    }
                }
            }
        } else if (lane == 0 && !*abort_flag) {
            fail();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kRtTmemCols));
    }
}

bool router_tc_supported(int T, int E, int H, size_t smem_limit) {
    return T >= 1 && E >= 1 && H % 8 == 0 && encode_fn() != nullptr && kRtSmem <= smem_limit;
}

static cudaError_t launch_router_tc(const __half *x, const __half *wr, int T, int E, int H, float *logits,
                                   uint32_t *err, cudaStream_t stream) {
    CUtensorMap xmap, wmap;
    cudaError_t e = rows_map(&xmap, x, T, H, kRtKB, kRtM);
    if (e != cudaSuccess) return e;
    e = rows_map(&wmap, wr, E, H, kRtKB, kRtN);
    if (e != cudaSuccess) return e;
    static int configured[128];
    e = ensure_smem(router_tc_kernel, configured, kRtSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((T + kRtM - 1) / kRtM), (unsigned)((E + kRtN - 1) / kRtN));
    return launch_pdl(router_tc_kernel, grid, kRtThreads, kRtSmem, stream, xmap, wmap, T, E, H, logits, err);
}

// ---------------------------------------------------------------- dispatch
// Which kernel computes the logits: the GEMV for T <= 16, the tensor cores above.
int router_path(int T, int E, int H, size_t smem_limit) {
    if (T >= 1 && T <= kRgMaxT) return 1;
    return router_tc_supported(T, E, H, smem_limit) ? 2 : 0;
}

cudaError_t launch_router_logits(const __half *x, const __half *wr, int T, int E, int H, float *logits,
                                 uint32_t *err, int num_sms, size_t smem_limit, cudaStream_t stream) {
    const int path = router_path(T, E, H, smem_limit);
    if (path == 1) {
        RouterArgs a{};
        a.x = reinterpret_cast<const uint4 *>(x);
        a.wr = reinterpret_cast<const uint4 *>(wr);
        a.T = T; a.E = E; a.k = 1; a.H8 = H / 8;
        a.logits = logits;
        a.ctrl = err - kCtrlErrorWord;
        a.fused = 0;
        return launch_gemv(a, num_sms, stream);
    }
    if (path == 2) return launch_router_tc(x, wr, T, E, H, logits, err, stream);
    return cudaErrorInvalidConfiguration;
}

// Logits, routing and grouping in one launch (router_fusable shapes).
// ctrl: the workspace control block; its ticket word must be zero (it is
// left zero).
cudaError_t launch_router_route_align(const __half *x, const __half *wr, int T, int E, int k, int H, float *logits,
                                      int32_t *ids, float *w, int32_t *offsets, int32_t *sorted, int32_t *active,
                                      int32_t *num_active, uint32_t *ctrl, int num_sms, cudaStream_t stream) {
    RouterArgs a{};
    a.x = reinterpret_cast<const uint4 *>(x);
    a.wr = reinterpret_cast<const uint4 *>(wr);
    a.T = T; a.E = E; a.k = k; a.H8 = H / 8; a.WS = align_slices(T * k);
    a.logits = logits; a.ids = ids; a.w = w;
    a.offsets = offsets; a.sorted = sorted; a.active = active; a.num_active = num_active;
    a.ctrl = ctrl;
    a.fused = 1;
    return launch_gemv(a, num_sms, stream);
}

}  // namespace moe
