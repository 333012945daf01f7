// prefill_tc.cu -- steps 3 and 4 for large batches on the 5th-generation
// tensor cores (tcgen05 MMA, accumulators in tensor memory).
//
// With thousands of tokens every expert sees tens to hundreds of rows, so
// the per-expert products of "Sparse MoE layer" (gate/up + SiLU, down) are
// dense contractions: for expert e, D[n][r] = sum_K W_e[n][K] * act[r][K]
// over the weight rows n of two 128-row tiles (the gate and up tiles of the
// same units, or two consecutive down tiles) and the (up to 128) activation
// rows r of a chunk of e's segment: the grouping of "Active grouped decode"
// (active-expert segments with offsets) decides the work list.
//
// One persistent CTA per SM, warp-specialised, all stages in shared memory:
//   warp 0      bulk tensor copies (TMA) of the packed codes of both tiles,
//               one per 64-wide K block, into the codes ring, and an L2
//               prefetch of the copies a few K blocks further on
//   warp 17     bulk tensor copies of the chunk's activation rows in the
//               128-byte-swizzled K-major operand layout into the B ring
//               (step 3 reads a sorted, pair-ordered copy of the x rows made
//               by sorted_rows_kernel; step 4 the h rows, already in sorted
//               order)
//   warps 2-..  dequantise the codes to fp16 ((q - z) * s, per 32-wide
//               group, exact q - z from the binary16 exponent trick) into the
//               A ring in the same layout; step 3 keeps the dequantiser's
//               pair order [k0 k4 k1 k5 k2 k6 k3 k7] (x was permuted alike:
//               the contraction over K does not depend on the order), step 4
//               restores natural order to match h
//   warp 1      one thread issues tcgen05.mma (kind::f16, fp32 accumulate in
//               tensor memory) for each K block and commits to mbarriers;
//               step 3 puts the chunk's rows in the M = 128 slot and gate and
//               up together in one N = 256 operand (4 MMAs per K block), step
//               4 each of its two weight tiles in M = 128 and the chunk in N
//               (8 MMAs per K block)
//   warps 18-21 read the accumulators (tcgen05.ld) and finish: h =
//               silu(gate) * up in fp16 (step 3), or the fp32 per-pair
//               projection y (step 4, summed per token by combine_kernel)
// Each ring is freed by its own readers: the codes ring by the dequantising
// warps as soon as they have converted a stage, the B and A rings by the
// MMAs that read them.  So the refill of the codes (from HBM, the longest
// latency) never waits for the tensor core, and the small codes stages can
// be many.  The accumulators are double-buffered, so copies,
// dequantisation, MMA and the epilogue of consecutive tiles overlap.
// Every wait is bounded.
#include <cuda.h>

#include "align.cuh"
#include "decode_common.cuh"
#include "tc_common.cuh"

namespace moe {

constexpr int kTcThreads = 704;
constexpr int kTcProducerWarp = 0, kTcMmaWarp = 1, kTcDqWarp0 = 2, kTcDqWarps = 16;
constexpr int kTcEpiWarp0 = 18, kTcEpiWarps = 4;
constexpr int kTcM = 128;     // weight rows per tile
constexpr int kTcKB = 64;     // K per stage: one 128-byte row of fp16
constexpr int kTcMaxN = 128;  // activation rows per chunk
// Dequantising warps of each step.  Every thread converts WPT words of one
// tile row per K block (a K block is 8 words of a row); fewer warps with
// more words each spend fewer instructions on the per-stage hand-offs.
#ifndef TC_GU_DQ_WARPS
#define TC_GU_DQ_WARPS 8
#endif
#ifndef TC_DOWN_DQ_WARPS
#define TC_DOWN_DQ_WARPS 8
#endif
// K blocks by which the L2 prefetch of codes and activation rows runs ahead
// of the copies into shared memory (0: no prefetch)
#ifndef TC_L2_AHEAD
#define TC_L2_AHEAD 8
#endif
// shared-memory split: the deepest A ring (up to TC_MAX_A stages) that
// leaves room for TC_B_STAGES activation-row stages and at least
// TC_MIN_C_STAGES codes stages; the codes ring takes the rest
#ifndef TC_MAX_A
#define TC_MAX_A 4
#endif
#ifndef TC_B_STAGES
#define TC_B_STAGES 3
#endif
#ifndef TC_MIN_C_STAGES
#define TC_MIN_C_STAGES 4
#endif
constexpr int kTcMaxCStages = 16;  // codes ring
constexpr int kTcMaxBStages = 8;   // activation-row ring
constexpr int kTcMaxAStages = 4;   // dequantised-tile ring
// the activation rows have their own producer: the last dequantising warp,
// which no step uses for dequantising
constexpr int kTcBProducerWarp = 2 + 16 - 1;
// smaller batches stay on the CUDA-core kernels; above the decode kernels'
// range the tensor-core path is 1.9-2.3x faster than the stream kernels
// (measured on the Qwen4Exp geometry at 16-48 tokens)
#ifndef TC_MIN_T
#define TC_MIN_T 9
#endif
constexpr int kTcMinT = TC_MIN_T;
constexpr uint32_t kTcTmemCols = 512;

static_assert(kTcEpiWarp0 == kTcDqWarp0 + kTcDqWarps && (kTcEpiWarp0 + kTcEpiWarps) * 32 == kTcThreads &&
                  kTcBProducerWarp == kTcDqWarp0 + kTcDqWarps - 1,
              "warp roles cover the CTA");

enum { kTcGateUp = 0, kTcDown = 1 };

// Each work item and each K-block stage covers two 128-row weight tiles:
// the gate and up tiles of the same output units (step 3), or two
// consecutive tiles of the down matrix (step 4).  Tile b of item tile index
// t starts at matrix row b * tc_mat_stride + t * tc_tile_stride.
constexpr int kTcTiles = 2;

template <int MODE>
struct TcDq {
    static constexpr int ntile = kTcTiles;
    static constexpr int warps = MODE == kTcGateUp ? TC_GU_DQ_WARPS : TC_DOWN_DQ_WARPS;
    static constexpr int wpt = ntile * kTcM * 8 / (warps * 32);  // words per thread per K block
    static_assert(warps < kTcDqWarps && (wpt == 2 || wpt == 4 || wpt == 8) &&
                      wpt * warps * 32 == ntile * kTcM * 8,
                  "dequantising threads cover both tiles: 2, 4 or 8 words each");
};

struct TcArgs {
    const __half *s;    // scales [E][N][G]
    const uint32_t *z;  // zeros  [E][N/8][G]
    const __half *vin;  // step 3: x [T][H]; step 4: h [P][I] (sorted rows)
    int E, N, K, rows;  // N: matrix rows per expert (2I or H); rows: output rows (I or H)
    int T, k, P;
    const int32_t *offsets, *sorted_pair, *active, *num_active;
    __half *h_out;      // step 3: [P][I]
    float *y_out;       // step 4: [P][H]
    uint32_t *err;
    int cstages, bstages, astages;  // ring depths: codes, activation rows, A tiles
    int amax;  // slot table capacity: min(E, P)
};

template <int MODE>
struct TcGeom {
    static constexpr int ntile = kTcTiles;
    static constexpr uint32_t a_bytes = ntile * kTcM * kTcKB * 2;  // the two dequantised tiles: the A ring
    static constexpr uint32_t b_bytes = kTcMaxN * kTcKB * 2;      // activation rows: the B ring
    static constexpr uint32_t c_bytes = ntile * kTcM * kTcKB / 2;  // packed codes: the codes ring
    static_assert(a_bytes % 1024 == 0 && b_bytes % 1024 == 0 && c_bytes % 1024 == 0, "stage alignment");
};

// Control block after the rings: mbarriers and the tensor-memory address.
//   c_full/c_free: codes ring (freed by the dequantising warps)
//   b_full/b_free: activation-row ring (freed by the MMAs that read it)
//   a_full/a_free: dequantised A tiles (freed by the MMAs that read them)
//   acc_full/acc_empty: the two accumulator buffers in tensor memory
struct TcCtrl {
    uint64_t c_full[kTcMaxCStages];
    uint64_t c_free[kTcMaxCStages];
    uint64_t b_full[kTcMaxBStages];
    uint64_t b_free[kTcMaxBStages];
    uint64_t a_full[kTcMaxAStages];
    uint64_t a_free[kTcMaxAStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem;
    int abort;
};

__host__ __device__ inline size_t tc_smem_bytes(uint32_t a_bytes, int astages, uint32_t b_bytes, int bstages,
                                                uint32_t c_bytes, int cstages) {
    return 1024 + (size_t)a_bytes * astages + (size_t)b_bytes * bstages + (size_t)c_bytes * cstages + sizeof(TcCtrl);
}

// ---------------------------------------------------------------- work list
// Work items, in order: for each active slot a, for each chunk of up to
// kTcMaxN segment rows, for each 128-row weight tile.  Each CTA builds the
// table of slots (expert, first sorted row, rows, first item) in shared
// memory once; item i of the grid-strided sequence is found by binary
// search over the first-item prefix.
struct TcItem {
    int a, e, lo, ne, tile, chunk;  // slot, expert, first sorted row, segment rows, tile, chunk
};

struct TcTable {
    int *e, *lo, *ne, *pre;  // pre: [A+1] first item of each slot
};

__device__ __forceinline__ TcItem tc_lookup(const TcTable &tb, int A, int tiles, int i) {
    int lo = 0, hi = A;  // pre[lo] <= i < pre[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tb.pre[mid] <= i) lo = mid; else hi = mid;
    }
    TcItem it;
    it.a = lo;
    it.e = tb.e[lo];
    it.lo = tb.lo[lo];
    it.ne = tb.ne[lo];
    const int j = i - tb.pre[lo];
    it.chunk = j / tiles;
    it.tile = j - it.chunk * tiles;
    return it;
}

__host__ __device__ inline size_t tc_table_bytes(int amax) { return ((size_t)5 * amax + 1 + 128) * 4; }

// Row strides of the two tiles of an item: step 3's tile b is matrix b (gate,
// up) at the item's output units; step 4's tiles are consecutive.
template <int MODE>
__device__ __forceinline__ int tc_mat_stride(int rows) { return MODE == kTcGateUp ? rows : kTcM; }
template <int MODE>
__device__ __forceinline__ int tc_tile_stride() { return MODE == kTcGateUp ? kTcM : kTcTiles * kTcM; }
// output unit of row m of tile b of item tile index t
template <int MODE>
__device__ __forceinline__ int tc_unit(int b, int t, int m) {
    return MODE == kTcGateUp ? t * kTcM + m : (kTcTiles * t + b) * kTcM + m;
}

// ---------------------------------------------------------------- kernel
// FMT: kFmtW4A16 (p.s fp16 scales, p.z zero words) or kFmtNvfp4 (p.s the
// E4M3 scale bytes, p.z the per-expert fp32 scales; the A tiles hold
// e2m1 * e4m3 in fp16, exact, and the epilogue applies the expert's scale).
template <int MODE, int FMT>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_kernel(const TcArgs p, const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap bmap) {
    using Gm = TcGeom<MODE>;
    constexpr int ntile = Gm::ntile;
    extern __shared__ uint8_t tc_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~(uintptr_t)1023);
    const int SC = p.cstages, SB = p.bstages, SA = p.astages;
    uint8_t *aring = smem;                              // [SA][a_bytes]
    uint8_t *bring = aring + (size_t)SA * Gm::a_bytes;  // [SB][b_bytes]
    uint8_t *cring = bring + (size_t)SB * Gm::b_bytes;  // [SC][c_bytes]
    TcCtrl *ctl = reinterpret_cast<TcCtrl *>(cring + (size_t)Gm::c_bytes * SC);
    int *tbase = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(ctl) + align_up(sizeof(TcCtrl), 16));
    const TcTable tb{tbase, tbase + p.amax, tbase + 2 * p.amax, tbase + 3 * p.amax};
    int *t_tmp = tbase + 4 * p.amax + 1, *t_scratch = t_tmp + p.amax;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.K / 32;
    const int nkb = (p.K + kTcKB - 1) / kTcKB;
    // item tile indices per chunk: units per item 128 (step 3) or 256 (step 4)
    const int tiles = (p.rows + tc_tile_stride<MODE>() - 1) / tc_tile_stride<MODE>();
    const int mstride = tc_mat_stride<MODE>(p.rows);

    if (tid == 0) {
        for (int s = 0; s < SC; ++s) {
            mbar_init(&ctl->c_full[s], 1);
            mbar_init(&ctl->c_free[s], TcDq<MODE>::warps);
        }
        for (int s = 0; s < SB; ++s) {
            mbar_init(&ctl->b_full[s], 1);
            mbar_init(&ctl->b_free[s], 1);
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(&ctl->a_full[s], TcDq<MODE>::warps);
            mbar_init(&ctl->a_free[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&ctl->acc_full[s], 1);
            mbar_init(&ctl->acc_empty[s], kTcEpiWarps);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&ctl->tmem)),
                     "r"(kTcTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    volatile int *abort_flag = &ctl->abort;
    pdl_wait();
    pdl_trigger();

    int A = *p.num_active;
    A = A < 0 ? 0 : (A > p.amax ? p.amax : A);
    auto fail = [&](uint32_t bits) {
        set_error(p.err, bits);
        *abort_flag = 1;
    };
    // slot table: expert, segment, items (tiles x chunks), then their prefix
    for (int a = tid; a < A; a += kTcThreads) {
        const int e = p.active[a];
        int lo = 0, ne = 0;
        if (e >= 0 && e < p.E) {
            lo = p.offsets[e];
            ne = p.offsets[e + 1] - lo;
        }
        if (ne < 0 || lo < 0 || lo + ne > p.P) ne = 0;
        tb.e[a] = e;
        tb.lo[a] = lo;
        tb.ne[a] = ne;
        tb.pre[a] = tiles * ((ne + kTcMaxN - 1) / kTcMaxN);
        t_tmp[a] = 0;
    }
    __syncthreads();
    const int n_items = block_exclusive_scan2(tb.pre, t_tmp, A, t_scratch).x;
    if (tid == 0) tb.pre[A] = n_items;
    __syncthreads();

    if (warp == kTcProducerWarp || warp == kTcBProducerWarp) {
        // ---- copies of every K block: warp 0 the codes of both tiles (and
        // the L2 prefetch), the B producer the chunk's activation rows; each
        // through its own ring
        const bool codes = warp == kTcProducerWarp;
        const int S = codes ? SC : SB;
        uint64_t *full = codes ? ctl->c_full : ctl->b_full;
        uint64_t *freeb = codes ? ctl->c_free : ctl->b_free;
        int j = 0, s = 0;
        uint32_t ph = 0;  // stage and phase of K block j in the ring
        // L2 prefetch cursor: TC_L2_AHEAD K blocks ahead in this CTA's sequence
        int pf_ii = blockIdx.x, pf_kb = 0;
        TcItem pf_it{};
        if (codes && pf_ii < n_items) pf_it = tc_lookup(tb, A, tiles, pf_ii);
        auto prefetch_next = [&]() {
            if (pf_ii >= n_items) return;
            if (lane == 0) {
#pragma unroll
                for (int b = 0; b < ntile; ++b)
                    tma_prefetch_2d(&qmap, pf_kb * (kTcKB / 8),
                                    pf_it.e * p.N + b * mstride + pf_it.tile * tc_tile_stride<MODE>());
                tma_prefetch_2d(&bmap, pf_kb * kTcKB, pf_it.lo + pf_it.chunk * kTcMaxN);
            }
            if (++pf_kb == nkb) {
                pf_kb = 0;
                pf_ii += gridDim.x;
                if (pf_ii < n_items) pf_it = tc_lookup(tb, A, tiles, pf_ii);
            }
        };
        if (codes)
            for (int d = 0; d < TC_L2_AHEAD; ++d) prefetch_next();
        for (int ii = blockIdx.x; ii < n_items && !__any_sync(0xffffffffu, *abort_flag != 0); ii += gridDim.x) {
            const TcItem it = tc_lookup(tb, A, tiles, ii);
            const int r0 = it.lo + it.chunk * kTcMaxN;
            for (int kb = 0; kb < nkb; ++kb, ++j) {
                if (codes && TC_L2_AHEAD > 0) prefetch_next();
                // the stage is free once its readers are done with its last
                // use (every lane waits; the decision is made warp-uniform)
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&freeb[s], ph ^ 1, abort_flag))) {
                    if (lane == 0 && !*abort_flag) fail(MOE_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                if (lane == 0) {
                    if (codes) {
                        uint8_t *stg = cring + (size_t)Gm::c_bytes * s;
                        mbar_arrive_expect_tx(&full[s], Gm::c_bytes);
#pragma unroll
                        for (int b = 0; b < ntile; ++b) {
                            const int row = it.e * p.N + b * mstride + it.tile * tc_tile_stride<MODE>();
                            tma_load_2d(stg + b * (kTcM * kTcKB / 2), &qmap, kb * (kTcKB / 8), row, &full[s]);
                        }
                    } else {
                        mbar_arrive_expect_tx(&full[s], Gm::b_bytes);
                        tma_load_2d(bring + (size_t)Gm::b_bytes * s, &bmap, kb * kTcKB, r0, &full[s]);
                    }
                }
                __syncwarp();
                if (++s == S) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        if (lane == 0 && *abort_flag) {
            // never leave with a copy in flight: wait for the last issue of each stage
            for (int jj = j > S ? j - S : 0; jj < j; ++jj)
                mbar_wait_bounded(&full[jj % S], (jj / S) & 1, nullptr);
        }
    } else if (warp == kTcMmaWarp) {
        // ---- one thread issues the MMAs
        if (lane == 0) {
            int n_done = 0, s = 0, s2 = 0;
            uint32_t ph = 0, ph2 = 0;  // B ring and A ring positions
            for (int ii = blockIdx.x; ii < n_items && !*abort_flag; ii += gridDim.x, ++n_done) {
                const TcItem it = tc_lookup(tb, A, tiles, ii);
                // Step 3: D[chunk row][weight row] = act . W^T, the chunk's
                // rows the A operand (M = 128; rows past the segment are
                // ignored by the epilogue), gate and up together the B operand
                // (N = 256): one MMA per K step.  Step 4: D[weight row][chunk
                // row] = W . act^T (M = 128 weight rows, N = the chunk padded
                // to 16), which lets its epilogue store fp32 rows coalesced.
                const int nrows = min(kTcMaxN, it.ne - it.chunk * kTcMaxN);
                const uint32_t idesc = MODE == kTcGateUp ? tc_idesc(kTcMaxN, ntile * kTcM)
                                                         : tc_idesc(kTcM, (nrows + 15) & ~15);
                const int as = n_done & 1;
                if (!mbar_wait_bounded(&ctl->acc_empty[as], ((n_done >> 1) & 1) ^ 1, abort_flag)) {
                    if (!*abort_flag) fail(MOE_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                tc_fence_after();
                const uint32_t dacc = tmem + (uint32_t)as * (ntile * kTcM);
                bool broke = false;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(&ctl->a_full[s2], ph2, abort_flag) ||
                        !mbar_wait_bounded(&ctl->b_full[s], ph, abort_flag)) {
                        if (!*abort_flag) fail(MOE_DEVERR_WAIT_TIMEOUT);
                        broke = true;
                        break;
                    }
                    tc_fence_after();
                    // descriptors of the stage's tiles; a K step of 16 advances
                    // the start address by 32 bytes, i.e. the descriptor by 2
                    // (shared addresses are below 2^18, so the 14-bit field
                    // never carries)
                    const uint64_t ad0 = tc_desc_sw128(smem_addr(aring + (size_t)Gm::a_bytes * s2));
                    const uint64_t bd0 = tc_desc_sw128(smem_addr(bring + (size_t)Gm::b_bytes * s));
#pragma unroll
                    for (int ks = 0; ks < kTcKB / 16; ++ks) {
                        if (MODE == kTcGateUp)
                            tc_mma(dacc, bd0 + (uint64_t)(ks * 2), ad0 + (uint64_t)(ks * 2), idesc, (kb | ks) != 0);
                        else
#pragma unroll
                            for (int b = 0; b < ntile; ++b)
                                tc_mma(dacc + b * kTcMaxN, ad0 + (uint64_t)(b * (kTcM * kTcKB * 2 / 16) + ks * 2),
                                       bd0 + (uint64_t)(ks * 2), idesc, (kb | ks) != 0);
                    }
                    tc_commit(&ctl->b_free[s]);
                    tc_commit(&ctl->a_free[s2]);
                    if (++s == SB) {
                        s = 0;
                        ph ^= 1;
                    }
                    if (++s2 == SA) {
                        s2 = 0;
                        ph2 ^= 1;
                    }
                }
                if (broke) break;
                tc_commit(&ctl->acc_full[as]);
            }
            // every MMA this thread issued has completed before tensor memory is released
            tc_commit(&ctl->drain);
            mbar_wait_bounded(&ctl->drain, 0, nullptr);
        }
    } else if (warp >= kTcDqWarp0 && warp < kTcDqWarp0 + kTcDqWarps) {
      constexpr int kDqActive = TcDq<MODE>::warps;
      if (warp < kTcDqWarp0 + kDqActive) {
        // ---- dequantise the codes into the A tiles
        const int t = tid - kTcDqWarp0 * 32;
        // each thread: one row of one tile and WPT words of the K block
        // (half a group, one group or both groups); the threads of a row are
        // adjacent, so a warp reads a contiguous run of codes
        constexpr int WPT = TcDq<MODE>::wpt, NWB = 8 / WPT;
        constexpr int NG = WPT == 8 ? 2 : 1;  // groups per thread per K block
        const int r = t / NWB, wb = t % NWB;
        const int b = r / kTcM, m = r % kTcM;
        const int w0 = wb * WPT, gi = w0 / 4;  // first word, first group within the K block
        int s = 0, s2 = 0;
        uint32_t ph = 0, ph2 = 0;  // codes ring and A ring positions
        // this thread's 16-byte chunks in a 128-byte-swizzled tile: row base
        // and the XOR applied to the chunk index
        const uint32_t rbase = (uint32_t)((m >> 3) * 1024 + (m & 7) * 128), rx = (uint32_t)(m & 7);
        // byte offsets inside a stage: this thread's codes, and its WPT
        // chunks of the A tile ((w0 + wi) ^ rx = (w0 ^ rx) ^ wi: w0 is a
        // multiple of WPT)
        const uint32_t coff = b * (kTcM * kTcKB / 2) + m * (kTcKB / 2) + w0 * 4;
        uint32_t aoff[WPT];
#pragma unroll
        for (int wi = 0; wi < WPT; ++wi)
            aoff[wi] = (uint32_t)(b * (kTcM * kTcKB * 2)) + rbase + ((((uint32_t)w0 ^ rx) ^ (uint32_t)wi) << 4);
        uint32_t tst = 0, ast = 0;  // byte offsets of the current codes stage and A stage
        for (int ii = blockIdx.x; ii < n_items && !__any_sync(0xffffffffu, *abort_flag != 0); ii += gridDim.x) {
            const TcItem it = tc_lookup(tb, A, tiles, ii);
            const int unit = tc_unit<MODE>(b, it.tile, m);
            const bool row_ok = unit < p.rows;
            const int n = b * mstride + it.tile * tc_tile_stride<MODE>() + m;  // row of the expert's matrix
            const __half *sp = p.s + ((size_t)it.e * p.N + n) * G + gi;
            const uint32_t *zp = p.z + ((size_t)it.e * (p.N / 8) + n / 8) * G + gi;
            const uint32_t zsh = 4u * (n & 7);
            // groups this thread may read: group 2 kb + gi + j of K block kb
            const int glim = row_ok ? G - gi : 0;
            // scale and zero word of this thread's group(s), fetched three K
            // blocks ahead
            uint32_t f0[2 * NG], f1[2 * NG], f2[2 * NG];
            auto fetch = [&](int kb, uint32_t (&f)[2 * NG]) {
#pragma unroll
                for (int j = 0; j < NG; ++j) {
                    const bool ok = 2 * kb + j < glim;
                    f[2 * j] = ok ? (uint32_t)__half_as_ushort(__ldg(sp + 2 * kb + j)) : 0u;
                    f[2 * j + 1] = (ok && FMT != kFmtNvfp4) ? __ldg(zp + 2 * kb + j) : 0u;
                }
            };
            fetch(0, f0);
            fetch(1, f1);
            fetch(2, f2);
            for (int kb = 0; kb < nkb; ++kb) {
                uint32_t fc[2 * NG];
#pragma unroll
                for (int i = 0; i < 2 * NG; ++i) {
                    fc[i] = f0[i];
                    f0[i] = f1[i];
                    f1[i] = f2[i];
                }
                fetch(kb + 3, f2);
                // the codes of this K block have landed; the A stage is free
                // once the MMAs of its last use are done
                const bool w_ok =
                    (mbar_test(&ctl->c_full[s], ph) || mbar_wait_bounded(&ctl->c_full[s], ph, abort_flag)) &&
                    (mbar_test(&ctl->a_free[s2], ph2 ^ 1) || mbar_wait_bounded(&ctl->a_free[s2], ph2 ^ 1, abort_flag));
                if (!__all_sync(0xffffffffu, w_ok)) {
                    if (lane == 0 && !*abort_flag) fail(MOE_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                const uint8_t *codes = cring + tst + coff;
                uint8_t *At = aring + ast;
                ZeroPoint zpt[NG];
                __half2 sv[NG], sv2[NG];  // NVFP4: the scales of the group's two 16-element blocks
#pragma unroll
                for (int j = 0; j < NG; ++j) {
                    if (FMT == kFmtNvfp4) {
                        const __half2 s2 = __half2(
                            __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(fc[2 * j] & 0xFFFFu), __NV_E4M3));
                        sv[j] = __low2half2(s2);
                        sv2[j] = __high2half2(s2);
                    } else {
                        zpt[j] = make_zero_point((fc[2 * j + 1] >> zsh) & 0xFu);
                        sv[j] = __half2half2(__ushort_as_half((unsigned short)(fc[2 * j] & 0xFFFFu)));
                    }
                }
                uint32_t cw[WPT];
                if (WPT == 2) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(codes);
                    cw[0] = v.x; cw[1 % WPT] = v.y;
                } else {
#pragma unroll
                    for (int c4 = 0; c4 < WPT / 4; ++c4) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(codes + 16 * c4);
                        cw[(4 * c4) % WPT] = v.x; cw[(4 * c4 + 1) % WPT] = v.y;
                        cw[(4 * c4 + 2) % WPT] = v.z; cw[(4 * c4 + 3) % WPT] = v.w;
                    }
                }
#pragma unroll
                for (int wi = 0; wi < WPT; ++wi) {
                    const int j = wi / 4 < NG ? wi / 4 : 0;  // group of word wi
                    __half2 d[4];
                    __half2 scl = sv[j];
                    if (FMT == kFmtNvfp4) {
                        e2m1_word(cw[wi], d);
                        if (((w0 + wi) & 3) >= 2) scl = sv2[j];  // words 2-3 of a group: its second block
                    } else {
                        dequant_word(cw[wi], zpt[j], d);
                    }
                    uint32_t u[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __half2 v2 = __hmul2(d[i], scl);
                        u[i] = *reinterpret_cast<const uint32_t *>(&v2);
                    }
                    uint4 o;
                    if (MODE == kTcGateUp) {
                        o = make_uint4(u[0], u[1], u[2], u[3]);  // pair order, like the sorted x copy
                    } else {
                        // natural order: (k0,k1) (k2,k3) (k4,k5) (k6,k7)
                        o.x = __byte_perm(u[0], u[1], 0x5410);
                        o.y = __byte_perm(u[2], u[3], 0x5410);
                        o.z = __byte_perm(u[0], u[1], 0x7632);
                        o.w = __byte_perm(u[2], u[3], 0x7632);
                    }
                    *reinterpret_cast<uint4 *>(At + aoff[wi]) = o;
                }
                fence_proxy_async();  // operands written by this thread -> tensor core reads
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&ctl->c_free[s]);  // the warp's codes are read
                    mbar_arrive(&ctl->a_full[s2]);
                }
                tst += Gm::c_bytes;
                if (++s == SC) {
                    s = 0;
                    tst = 0;
                    ph ^= 1;
                }
                ast += Gm::a_bytes;
                if (++s2 == SA) {
                    s2 = 0;
                    ast = 0;
                    ph2 ^= 1;
                }
            }
        }
      }
    } else {
        // ---- epilogue: accumulators -> h (step 3) or y (step 4)
        const int q = warp & 3;  // tensor-memory lane quadrant of this warp
        const int m = q * 32 + lane;
        int n_done = 0;
        for (int ii = blockIdx.x; ii < n_items && !__any_sync(0xffffffffu, *abort_flag != 0); ii += gridDim.x, ++n_done) {
            const TcItem it = tc_lookup(tb, A, tiles, ii);
            const int nrows = min(kTcMaxN, it.ne - it.chunk * kTcMaxN);
            const int as = n_done & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&ctl->acc_full[as], (n_done >> 1) & 1, abort_flag))) {
                if (lane == 0 && !*abort_flag) fail(MOE_DEVERR_WAIT_TIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t dacc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)as * (ntile * kTcM);
            const int r0 = it.lo + it.chunk * kTcMaxN;
            const float escale = FMT == kFmtNvfp4 ? __ldg(reinterpret_cast<const float *>(p.z) + it.e) : 1.f;
            const int u0 = it.tile * kTcM;  // first output unit of the tile
            if (MODE == kTcGateUp) {
                // lane m holds chunk row m (one token-expert pair), column n
                // weight row n (gate 0..127, up 128..255): each thread
                // finishes one pair's outputs, 16 at a time, in 32-byte
                // stores.  Units come in runs of 16 that are wholly valid or
                // wholly past the last row (rows is a multiple of 32), so the
                // bound is warp-uniform.
                const bool row_ok = m < nrows;
                for (int c0 = 0; c0 < kTcM && u0 + c0 < p.rows; c0 += 16) {
                    uint32_t g[16], u[16];
                    tc_ld16(dacc + c0, g);
                    tc_ld16(dacc + kTcM + c0, u);
                    tc_wait_ld();
                    if (row_ok) {
                        uint32_t hv[8];
#pragma unroll
                        for (int c = 0; c < 16; c += 2) {
                            float o[2];
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const float gv = __uint_as_float(g[c + i]) * escale,
                                            uv = __uint_as_float(u[c + i]) * escale;
                                o[i] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                            }
                            const __half2 h2 = __floats2half2_rn(o[0], o[1]);
                            hv[c / 2] = *reinterpret_cast<const uint32_t *>(&h2);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(p.h_out + (size_t)(r0 + m) * p.rows + u0 + c0);
                        dst[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                        dst[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
                    }
                }
            } else {
                // lane m holds weight row m of tile b, column c chunk row c:
                // for each column the warp stores 32 consecutive fp32 outputs
                // of one pair (pair ids: lane l holds rows l + 32i)
                int prs[4] = {-1, -1, -1, -1};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (lane + 32 * i < nrows) prs[i] = __ldg(p.sorted_pair + r0 + lane + 32 * i);
                for (int b = 0; b < ntile; ++b)
                for (int c0 = 0; c0 < nrows; c0 += 16) {
                    const int unit = tc_unit<MODE>(b, it.tile, m);
                    uint32_t g[16];
                    tc_ld16(dacc + b * kTcMaxN + c0, g);
                    tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        // every lane takes part in the shuffle; only valid rows store
                        const int col = c0 + c, q4 = col >> 5;
                        const int v = q4 == 0 ? prs[0] : (q4 == 1 ? prs[1] : (q4 == 2 ? prs[2] : prs[3]));
                        const int pr = __shfl_sync(0xffffffffu, v, col & 31);
                        if (unit < p.rows && col < nrows && pr >= 0 && pr < p.P)
                            p.y_out[(size_t)pr * p.rows + unit] = __uint_as_float(g[c]) * escale;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->acc_empty[as]);
        }
    }

    // ---- teardown: every role has finished; release tensor memory
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols));
    }
}

// ---------------------------------------------------------------- host side
namespace {

// 2-D map over the packed codes viewed as [E*N rows][K/8 words], box of
// 8 words x 128 rows (one 64-wide K block of one tile); reads beyond the
// tensor return zeros.
cudaError_t codes_map(CUtensorMap *map, const uint32_t *q, int E, int N, int K) {
    EncodeTiled fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)E * N};
    const cuuint64_t strides[1] = {(cuuint64_t)K / 2};
    const cuuint32_t box[2] = {kTcKB / 8, kTcM};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t *>(q), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int MODE, int FMT>
cudaError_t launch_tc(const TcArgs &a0, const uint32_t *q, const __half *brows, long long nbrows, int num_sms,
                      size_t smem_limit, cudaStream_t stream) {
    using Gm = TcGeom<MODE>;
    TcArgs a = a0;
    a.amax = a.E < a.P ? a.E : a.P;
    // the deepest A ring (up to TC_MAX_A) that leaves room for the B ring
    // and a codes ring of at least TC_MIN_C_STAGES; the codes ring takes the rest
    const size_t base = tc_smem_bytes(0, 0, 0, 0, 0, 0) + 16 + tc_table_bytes(a.amax);
    const int sb_want = TC_B_STAGES < kTcMaxBStages ? TC_B_STAGES : kTcMaxBStages;
    a.astages = 0;
    for (int sa = TC_MAX_A < kTcMaxAStages ? TC_MAX_A : kTcMaxAStages; sa >= 2 && a.astages == 0; --sa)
        for (int sb = sb_want; sb >= 2; --sb)
            if (base + (size_t)sa * Gm::a_bytes + (size_t)sb * Gm::b_bytes + TC_MIN_C_STAGES * (size_t)Gm::c_bytes <=
                smem_limit) {
                a.astages = sa;
                a.bstages = sb;
                break;
            }
    if (a.astages == 0) return cudaErrorInvalidConfiguration;
    const size_t fixed = base + (size_t)a.astages * Gm::a_bytes + (size_t)a.bstages * Gm::b_bytes;
    const int SC = (int)((smem_limit - fixed) / Gm::c_bytes);
    a.cstages = SC > kTcMaxCStages ? kTcMaxCStages : SC;
    const size_t smem = fixed + (size_t)Gm::c_bytes * a.cstages;
    CUtensorMap map, bmap;
    cudaError_t e = codes_map(&map, q, a.E, a.N, a.K);
    if (e != cudaSuccess) return e;
    e = rows_map(&bmap, brows, nbrows, a.K, kTcKB, kTcMaxN);
    if (e != cudaSuccess) return e;
    static int configured[128];
    e = ensure_smem(tc_kernel<MODE, FMT>, configured, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(tc_kernel<MODE, FMT>, num_sms, kTcThreads, smem, stream, a, map, bmap);
}

// xs[r] = x[token of sorted row r], each 8-element block in the
// dequantiser's pair order (rows of invalid pairs: zeros).  Step 3 then
// reads the activation rows of a chunk as one contiguous tile.  One warp per
// row: the row's pair id is read once, then up to 8 loads per lane are in
// flight before the stores.
__global__ void sorted_rows_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ sorted_pair, int k,
                                   int P, int H8, uint4 *__restrict__ xs) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
    const int nwarps = gridDim.x * wpb;
    for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < P; r += nwarps) {
        const int pr = __ldg(sorted_pair + r);
        const bool ok = pr >= 0 && pr < P;
        const uint4 *src = x + (size_t)(ok ? pr / k : 0) * H8;
        uint4 *dst = xs + (size_t)r * H8;
        for (int c0 = 0; c0 < H8; c0 += 32 * 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = c0 + 32 * u + lane;
                v[u] = (ok && c < H8) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = c0 + 32 * u + lane;
                if (c < H8) dst[c] = pair_interleave(v[u]);
            }
        }
    }
}

}  // namespace

// Shapes the tensor-core path takes: fp16 activations with K a multiple of
// 32 (groups) and enough rows per expert on average to fill MMA granules.
bool tc_supported(int T, int E, int k, int H, int I, size_t smem_limit) {
    const int amax = E < T * k ? E : T * k;
    // a chunk's activation box may reach past the last sorted row (P < 128):
    // those rows lie outside the tensor map and are read as zeros
    return T >= kTcMinT && H % 32 == 0 && I % 32 == 0 && encode_fn() != nullptr &&
           tc_smem_bytes(TcGeom<kTcGateUp>::a_bytes, 2, TcGeom<kTcGateUp>::b_bytes, 2, TcGeom<kTcGateUp>::c_bytes,
                         TC_MIN_C_STAGES) + 16 + tc_table_bytes(amax) <=
               smem_limit;
}

template <int FMT>
static cudaError_t launch_gate_up_tc_f(const __half *x, const uint32_t *q, const __half *s, const uint32_t *z,
                              const int32_t *offsets, const int32_t *sorted_pair, const int32_t *active,
                              const int32_t *num_active, int T, int E, int k, int H, int I, __half *h, __half *xperm,
                              uint32_t *err, int num_sms, size_t smem_limit, cudaStream_t stream) {
    TcArgs a{};
    a.s = s; a.z = z; a.vin = x;
    a.E = E; a.N = 2 * I; a.K = H; a.rows = I;
    a.T = T; a.k = k; a.P = T * k;
    a.offsets = offsets; a.sorted_pair = sorted_pair; a.active = active; a.num_active = num_active;
    a.h_out = h; a.err = err;
    // the sorted, pair-ordered x rows, in the scratch the caller provides (P*H halves)
    cudaError_t e = launch_pdl(sorted_rows_kernel, num_sms * 8, 256, 0, stream, reinterpret_cast<const uint4 *>(x),
                               sorted_pair, k, T * k, H / 8, reinterpret_cast<uint4 *>(xperm));
    if (e != cudaSuccess) return e;
    return launch_tc<kTcGateUp, FMT>(a, q, xperm, (long long)T * k, num_sms, smem_limit, stream);
}

cudaError_t launch_gate_up_tc(const __half *x, const uint32_t *q, const __half *s, const uint32_t *z,
                              const int32_t *offsets, const int32_t *sorted_pair, const int32_t *active,
                              const int32_t *num_active, int T, int E, int k, int H, int I, __half *h, __half *xperm,
                              uint32_t *err, int num_sms, size_t smem_limit, cudaStream_t stream) {
    return launch_gate_up_tc_f<kFmtW4A16>(x, q, s, z, offsets, sorted_pair, active, num_active, T, E, k, H, I, h,
                                          xperm, err, num_sms, smem_limit, stream);
}

// NVFP4 weights: s the E4M3 scale bytes, gs the per-expert scales
cudaError_t launch_gate_up_tc_nvfp4(const __half *x, const uint32_t *q, const uint8_t *s, const float *gs,
                                    const int32_t *offsets, const int32_t *sorted_pair, const int32_t *active,
                                    const int32_t *num_active, int T, int E, int k, int H, int I, __half *h,
                                    __half *xperm, uint32_t *err, int num_sms, size_t smem_limit,
                                    cudaStream_t stream) {
    return launch_gate_up_tc_f<kFmtNvfp4>(x, q, reinterpret_cast<const __half *>(s),
                                          reinterpret_cast<const uint32_t *>(gs), offsets, sorted_pair, active,
                                          num_active, T, E, k, H, I, h, xperm, err, num_sms, smem_limit, stream);
}

cudaError_t launch_combine(const float *y, const float *topk_w, int T, int k, int H, __half *out,
                           cudaStream_t stream);

template <int FMT>
static cudaError_t launch_down_tc_f(const __half *h, const uint32_t *q, const __half *s, const uint32_t *z,
                           const int32_t *offsets, const int32_t *sorted_pair, const int32_t *active,
                           const int32_t *num_active, const float *topk_w, int T, int E, int k, int H, int I,
                           __half *out, float *y, uint32_t *err, int num_sms, size_t smem_limit,
                           cudaStream_t stream) {
    TcArgs a{};
    a.s = s; a.z = z; a.vin = h;
    a.E = E; a.N = H; a.K = I; a.rows = H;
    a.T = T; a.k = k; a.P = T * k;
    a.offsets = offsets; a.sorted_pair = sorted_pair; a.active = active; a.num_active = num_active;
    a.y_out = y; a.err = err;
    cudaError_t e = launch_tc<kTcDown, FMT>(a, q, h, (long long)T * k, num_sms, smem_limit, stream);
    if (e != cudaSuccess) return e;
    return launch_combine(y, topk_w, T, k, H, out, stream);
}

cudaError_t launch_down_tc(const __half *h, const uint32_t *q, const __half *s, const uint32_t *z,
                           const int32_t *offsets, const int32_t *sorted_pair, const int32_t *active,
                           const int32_t *num_active, const float *topk_w, int T, int E, int k, int H, int I,
                           __half *out, float *y, uint32_t *err, int num_sms, size_t smem_limit,
                           cudaStream_t stream) {
    return launch_down_tc_f<kFmtW4A16>(h, q, s, z, offsets, sorted_pair, active, num_active, topk_w, T, E, k, H, I,
                                       out, y, err, num_sms, smem_limit, stream);
}

cudaError_t launch_down_tc_nvfp4(const __half *h, const uint32_t *q, const uint8_t *s, const float *gs,
                                 const int32_t *offsets, const int32_t *sorted_pair, const int32_t *active,
                                 const int32_t *num_active, const float *topk_w, int T, int E, int k, int H, int I,
                                 __half *out, float *y, uint32_t *err, int num_sms, size_t smem_limit,
                                 cudaStream_t stream) {
    return launch_down_tc_f<kFmtNvfp4>(h, q, reinterpret_cast<const __half *>(s),
                                       reinterpret_cast<const uint32_t *>(gs), offsets, sorted_pair, active,
                                       num_active, topk_w, T, E, k, H, I, out, y, err, num_sms, smem_limit, stream);
}

}  // namespace moe
