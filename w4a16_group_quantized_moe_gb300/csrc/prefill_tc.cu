// prefill_tc.cu -- steps 3 and 4 for large batches on the 5th-generation
// tensor cores (tcgen05 MMA, accumulators in tensor memory).
//
// With thousands of tokens every expert sees tens to hundreds of rows, so
// the per-expert products of "Sparse MoE layer" (gate/up + SiLU, down) are
// dense contractions: for expert e, D[n][r] = sum_K W_e[n][K] * act[r][K]
// over the weight rows n of a 128-row tile and the (up to 128) activation
// rows r of a chunk of e's segment.  The weight is the MMA's A operand
// (M = 128 rows), the gathered activation rows its B operand (N = the chunk,
// padded to 16): the grouping of "Active grouped decode" (active-expert
// segments with offsets) decides the work list, and no expert is padded
// beyond one 16-row MMA granule.
//
// One persistent CTA per SM, warp-specialised, all stages in shared memory:
//   warp 0      bulk tensor copies (TMA) per 64-wide K block, into a ring
//               of copy stages: the packed codes of the tile(s), and the
//               chunk's activation rows in the 128-byte-swizzled K-major
//               operand layout, one copy (step 3 reads a sorted,
//               pair-ordered copy of the x rows made by sorted_rows_kernel;
//               step 4 the h rows, already in sorted order)
//   warps 2-17  dequantise the codes to fp16 ((q - z) * s, per 32-wide
//               group, exact q - z from the binary16 exponent trick) into the
//               same layout; step 3 keeps the dequantiser's pair order
//               [k0 k4 k1 k5 k2 k6 k3 k7] (x was permuted alike: the
//               contraction over K does not depend on the order), step 4
//               restores natural order to match h
//   warp 1      one thread issues tcgen05.mma (kind::f16, fp32 accumulate in
//               tensor memory) for each K block and commits to mbarriers
//   warps 18-21 read the accumulators (tcgen05.ld) and finish: h =
//               silu(gate) * up in fp16 (step 3), or the fp32 per-pair
//               projection y (step 4, summed per token by combine_kernel)
// The copy ring is as deep as shared memory allows (it covers the HBM
// latency of the codes), the dequantised tiles have their own two-stage
// ring, and the accumulators are double-buffered, so copies,
// dequantisation, MMA and the epilogue of consecutive tiles overlap.
// Every wait is bounded.
#include <cuda.h>

#include "align.cuh"

namespace moe {

constexpr int kTcThreads = 704;
constexpr int kTcProducerWarp = 0, kTcMmaWarp = 1, kTcDqWarp0 = 2, kTcDqWarps = 16;
constexpr int kTcEpiWarp0 = 18, kTcEpiWarps = 4;
constexpr int kTcM = 128;     // weight rows per tile
constexpr int kTcKB = 64;     // K per stage: one 128-byte row of fp16
constexpr int kTcMaxN = 128;  // activation rows per chunk
// dequantising warps of step 4 (128 rows per tile: 8 warps, 4 words per
// thread, measured faster than 16 warps with 2 words)
#ifndef TC_DOWN_DQ_WARPS
#define TC_DOWN_DQ_WARPS 8
#endif
constexpr int kTcMaxStages = 8;   // copy ring
constexpr int kTcMaxAStages = 4;  // dequantised-tile ring
constexpr int kTcMinT = 64;   // smaller batches stay on the CUDA-core stream kernels
constexpr uint32_t kTcTmemCols = 512;

static_assert(kTcEpiWarp0 == kTcDqWarp0 + kTcDqWarps && (kTcEpiWarp0 + kTcEpiWarps) * 32 == kTcThreads,
              "warp roles cover the CTA");

enum { kTcGateUp = 0, kTcDown = 1 };

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
    int nstages, astages;
    int amax;  // slot table capacity: min(E, P)
};

template <int MODE>
struct TcGeom {
    static constexpr int nmat = MODE == kTcGateUp ? 2 : 1;
    static constexpr uint32_t a_bytes = nmat * kTcM * kTcKB * 2;  // dequantised tile(s): the A ring
    static constexpr uint32_t b_bytes = kTcMaxN * kTcKB * 2;      // activation rows   } the copy
    static constexpr uint32_t c_bytes = nmat * kTcM * kTcKB / 2;  // packed codes      } ring
    static constexpr uint32_t t_bytes = b_bytes + c_bytes;        // multiples of 1024
};

// Control block after the rings: mbarriers and the tensor-memory address.
//   t_full/t_free: copy ring (codes and activation rows of a K block)
//   a_full/a_free: dequantised A tiles (astages stages)
//   acc_full/acc_empty: the two accumulator buffers in tensor memory
struct TcCtrl {
    uint64_t t_full[kTcMaxStages];
    uint64_t t_free[kTcMaxStages];
    uint64_t a_full[kTcMaxAStages];
    uint64_t a_free[kTcMaxAStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem;
    int abort;
};

__host__ __device__ inline size_t tc_smem_bytes(uint32_t a_bytes, int astages, uint32_t t_bytes, int nstages) {
    return 1024 + (size_t)a_bytes * astages + (size_t)t_bytes * nstages + sizeof(TcCtrl);
}

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {
    // shared-memory matrix descriptor: K-major, 128-byte swizzle; start
    // address >> 4, leading offset unused (1), stride offset 1024 B between
    // 8-row groups, descriptor version 1, layout type 2 (128-byte swizzle)
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24
__device__ __forceinline__ uint32_t tc_idesc(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

// byte offset of 16-byte chunk c (K elements 8c..8c+7) of row r in a
// 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
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

// ---------------------------------------------------------------- kernel
template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_kernel(const TcArgs p, const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap bmap) {
    using Gm = TcGeom<MODE>;
    constexpr int nmat = Gm::nmat;
    extern __shared__ uint8_t tc_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~(uintptr_t)1023);
    const int S = p.nstages, SA = p.astages;
    uint8_t *aring = smem;                             // [SA][a_bytes]
    uint8_t *tring = smem + (size_t)SA * Gm::a_bytes;  // [S][b_bytes + c_bytes]
    TcCtrl *ctl = reinterpret_cast<TcCtrl *>(tring + (size_t)Gm::t_bytes * S);
    int *tbase = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(ctl) + align_up(sizeof(TcCtrl), 16));
    const TcTable tb{tbase, tbase + p.amax, tbase + 2 * p.amax, tbase + 3 * p.amax};
    int *t_tmp = tbase + 4 * p.amax + 1, *t_scratch = t_tmp + p.amax;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.K / 32;
    const int nkb = (p.K + kTcKB - 1) / kTcKB;
    const int tiles = (p.rows + kTcM - 1) / kTcM;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl->t_full[s], 1);
            mbar_init(&ctl->t_free[s], 1);
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(&ctl->a_full[s], MODE == kTcGateUp ? kTcDqWarps : TC_DOWN_DQ_WARPS);
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

    if (warp == kTcProducerWarp) {
        // ---- codes and activation rows of every K block, through the copy ring
        int j = 0, s = 0;
        uint32_t ph = 0;  // stage and phase of K block j in the copy ring
        for (int ii = blockIdx.x; ii < n_items && !__any_sync(0xffffffffu, *abort_flag != 0); ii += gridDim.x) {
            const TcItem it = tc_lookup(tb, A, tiles, ii);
            const int r0 = it.lo + it.chunk * kTcMaxN;
            for (int kb = 0; kb < nkb; ++kb, ++j) {
                // the stage is free once the MMAs of its last use are done
                // (every lane waits; the decision is made warp-uniform)
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&ctl->t_free[s], ph ^ 1, abort_flag))) {
                    if (lane == 0 && !*abort_flag) fail(MOE_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                if (lane == 0) {
                    uint8_t *stg = tring + (size_t)Gm::t_bytes * s;
                    mbar_arrive_expect_tx(&ctl->t_full[s], Gm::t_bytes);
#pragma unroll
                    for (int b = 0; b < nmat; ++b) {
                        const int row = it.e * p.N + b * p.rows + it.tile * kTcM;
                        tma_load_2d(stg + Gm::b_bytes + b * (kTcM * kTcKB / 2), &qmap, kb * (kTcKB / 8), row,
                                    &ctl->t_full[s]);
                    }
                    tma_load_2d(stg, &bmap, kb * kTcKB, r0, &ctl->t_full[s]);
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
                mbar_wait_bounded(&ctl->t_full[jj % S], (jj / S) & 1, nullptr);
        }
    } else if (warp == kTcMmaWarp) {
        // ---- one thread issues the MMAs
        if (lane == 0) {
            int n_done = 0, s = 0, s2 = 0;
            uint32_t ph = 0, ph2 = 0;  // copy ring and A ring positions
            for (int ii = blockIdx.x; ii < n_items && !*abort_flag; ii += gridDim.x, ++n_done) {
                const TcItem it = tc_lookup(tb, A, tiles, ii);
                const int nrows = min(kTcMaxN, it.ne - it.chunk * kTcMaxN);
                const uint32_t idesc = tc_idesc((nrows + 15) & ~15);
                const int as = n_done & 1;
                if (!mbar_wait_bounded(&ctl->acc_empty[as], ((n_done >> 1) & 1) ^ 1, abort_flag)) {
                    if (!*abort_flag) fail(MOE_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                tc_fence_after();
                const uint32_t dacc = tmem + (uint32_t)as * (nmat * kTcMaxN);
                bool broke = false;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(&ctl->a_full[s2], ph2, abort_flag) ||
                        !mbar_wait_bounded(&ctl->t_full[s], ph, abort_flag)) {
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
                    const uint64_t bd0 = tc_desc_sw128(smem_addr(tring + (size_t)Gm::t_bytes * s));
#pragma unroll
                    for (int ks = 0; ks < kTcKB / 16; ++ks) {
#pragma unroll
                        for (int b = 0; b < nmat; ++b)
                            tc_mma(dacc + b * kTcMaxN, ad0 + (uint64_t)(b * (kTcM * kTcKB * 2 / 16) + ks * 2),
                                   bd0 + (uint64_t)(ks * 2), idesc, (kb | ks) != 0);
                    }
                    tc_commit(&ctl->t_free[s]);
                    tc_commit(&ctl->a_free[s2]);
                    if (++s == S) {
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
      constexpr int kDqActive = MODE == kTcGateUp ? kTcDqWarps : TC_DOWN_DQ_WARPS;
      if (warp < kTcDqWarp0 + kDqActive) {
        // ---- dequantise the codes into the A tile(s)
        const int t = tid - kTcDqWarp0 * 32;  // 0..511
        // each thread: one row of the tile(s) and WPT words (one group) of
        // the K block; the threads of a row are adjacent, so a warp reads a
        // contiguous run of codes.  Step 3: 2 threads per row of 256 (matrix
        // b = r / 128), 4 words each; step 4: 4 threads per row of 128, 2
        // words each.
        constexpr int WPT = nmat * kTcM * 8 / (kDqActive * 32), NWB = 8 / WPT;
        const int r = t / NWB, wb = t % NWB;
        const int b = r / kTcM, m = r % kTcM;
        const int w0 = wb * WPT, gi = w0 / 4;  // first word, group within the K block
        int s = 0, s2 = 0;
        uint32_t ph = 0, ph2 = 0;  // copy ring and A ring positions
        // this thread's 16-byte chunks in a 128-byte-swizzled tile: row base
        // and the XOR applied to the chunk index
        const uint32_t rbase = (uint32_t)((m >> 3) * 1024 + (m & 7) * 128), rx = (uint32_t)(m & 7);
        // byte offsets inside a stage: this thread's codes, and its WPT
        // chunks of the A tile ((w0 + wi) ^ rx = (w0 ^ rx) ^ wi: w0 is a
        // multiple of WPT)
        const uint32_t coff = Gm::b_bytes + b * (kTcM * kTcKB / 2) + m * (kTcKB / 2) + w0 * 4;
        uint32_t aoff[WPT];
#pragma unroll
        for (int wi = 0; wi < WPT; ++wi)
            aoff[wi] = (uint32_t)(b * (kTcM * kTcKB * 2)) + rbase + ((((uint32_t)w0 ^ rx) ^ (uint32_t)wi) << 4);
        uint32_t tst = 0, ast = 0;  // byte offsets of the current copy stage and A stage
        for (int ii = blockIdx.x; ii < n_items && !__any_sync(0xffffffffu, *abort_flag != 0); ii += gridDim.x) {
            const TcItem it = tc_lookup(tb, A, tiles, ii);
            const int unit = it.tile * kTcM + m;
            const bool row_ok = unit < p.rows;
            const int n = b * p.rows + unit;
            const __half *sp = p.s + ((size_t)it.e * p.N + n) * G + gi;
            const uint32_t *zp = p.z + ((size_t)it.e * (p.N / 8) + n / 8) * G + gi;
            const uint32_t zsh = 4u * (n & 7);
            // scale and zero word of this thread's group, fetched three K
            // blocks ahead
            uint32_t f0[2] = {0, 0}, f1[2] = {0, 0}, f2[2] = {0, 0};
            // K blocks whose group this thread has (g = 2 kb + gi < G)
            const int kb_lim = row_ok ? min(nkb, (G - gi + 1) / 2) : 0;
            auto fetch = [&](int kb, uint32_t (&f)[2]) {
                f[0] = f[1] = 0;
                if (kb >= kb_lim) return;
                f[0] = (uint32_t)__half_as_ushort(__ldg(sp + 2 * kb));
                f[1] = __ldg(zp + 2 * kb);
            };
            fetch(0, f0);
            fetch(1, f1);
            fetch(2, f2);
            for (int kb = 0; kb < nkb; ++kb) {
                const uint32_t sc = f0[0], zc = f0[1];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    f0[i] = f1[i];
                    f1[i] = f2[i];
                }
                fetch(kb + 3, f2);
                // the codes of this K block have landed; the A stage is free
                // once the MMAs of its last use are done
                const bool w_ok =
                    (mbar_test(&ctl->t_full[s], ph) || mbar_wait_bounded(&ctl->t_full[s], ph, abort_flag)) &&
                    (mbar_test(&ctl->a_free[s2], ph2 ^ 1) || mbar_wait_bounded(&ctl->a_free[s2], ph2 ^ 1, abort_flag));
                if (!__all_sync(0xffffffffu, w_ok)) {
                    if (lane == 0 && !*abort_flag) fail(MOE_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                const uint8_t *codes = tring + tst + coff;
                uint8_t *At = aring + ast;
                const ZeroPoint zpt = make_zero_point((zc >> zsh) & 0xFu);
                const __half2 sv = __half2half2(__ushort_as_half((unsigned short)(sc & 0xFFFFu)));
                uint32_t cw[WPT];
                if (WPT == 4) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(codes);
                    cw[0] = v.x; cw[1] = v.y; cw[2 % WPT] = v.z; cw[3 % WPT] = v.w;
                } else {
                    const uint2 v = *reinterpret_cast<const uint2 *>(codes);
                    cw[0] = v.x; cw[1] = v.y;
                }
#pragma unroll
                for (int wi = 0; wi < WPT; ++wi) {
                    __half2 d[4];
                    dequant_word(cw[wi], zpt, d);
                    uint32_t u[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __half2 v2 = __hmul2(d[i], sv);
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
                if (lane == 0) mbar_arrive(&ctl->a_full[s2]);
                tst += Gm::t_bytes;
                if (++s == S) {
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
            const uint32_t dacc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)as * (nmat * kTcMaxN);
            const int unit = it.tile * kTcM + m;
            const int r0 = it.lo + it.chunk * kTcMaxN;
            // step 4: pair ids of the chunk's rows, lane l holding rows l + 32i
            int prs[4] = {-1, -1, -1, -1};
            if (MODE == kTcDown) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (lane + 32 * i < nrows) prs[i] = __ldg(p.sorted_pair + r0 + lane + 32 * i);
            }
            for (int c0 = 0; c0 < nrows; c0 += 16) {
                uint32_t g[16];
                tc_ld16(dacc + c0, g);
                if (MODE == kTcGateUp) {
                    uint32_t u[16];
                    tc_ld16(dacc + kTcMaxN + c0, u);
                    tc_wait_ld();
                    if (unit < p.rows) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            if (c0 + c < nrows) {
                                const float gv = __uint_as_float(g[c]), uv = __uint_as_float(u[c]);
                                const float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                                p.h_out[(size_t)(r0 + c0 + c) * p.rows + unit] = __float2half_rn(hv);
                            }
                        }
                    }
                } else {
                    tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        // every lane takes part in the shuffle; only valid rows store
                        const int col = c0 + c, q4 = col >> 5;
                        const int v = q4 == 0 ? prs[0] : (q4 == 1 ? prs[1] : (q4 == 2 ? prs[2] : prs[3]));
                        const int pr = __shfl_sync(0xffffffffu, v, col & 31);
                        if (unit < p.rows && col < nrows && pr >= 0 && pr < p.P)
                            p.y_out[(size_t)pr * p.rows + unit] = __uint_as_float(g[c]);
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

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
    }
    return fn;
}

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

// 2-D map over fp16 activation rows [rows][K] with the 128-byte swizzle;
// box of 64 elements x box_rows rows.
cudaError_t rows_map(CUtensorMap *map, const __half *base, long long rows, int K, int box_rows) {
    EncodeTiled fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {kTcKB, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int MODE>
cudaError_t launch_tc(const TcArgs &a0, const uint32_t *q, const __half *brows, long long nbrows, int num_sms,
                      size_t smem_limit, cudaStream_t stream) {
    using Gm = TcGeom<MODE>;
    TcArgs a = a0;
    a.amax = a.E < a.P ? a.E : a.P;
    // the deepest A ring (up to 4) that leaves at least 4 copy stages
    const size_t base = tc_smem_bytes(0, 0, 0, 0) + 16 + tc_table_bytes(a.amax);
    a.astages = 0;
    for (int sa = kTcMaxAStages; sa >= 2; --sa)
        if (base + (size_t)sa * Gm::a_bytes + 4 * (size_t)Gm::t_bytes <= smem_limit) {
            a.astages = sa;
            break;
        }
    if (a.astages == 0) return cudaErrorInvalidConfiguration;
    const size_t fixed = base + (size_t)a.astages * Gm::a_bytes;
    const int S = (int)((smem_limit - fixed) / Gm::t_bytes);
    a.nstages = S > kTcMaxStages ? kTcMaxStages : S;
    const size_t smem = fixed + (size_t)Gm::t_bytes * a.nstages;
    CUtensorMap map, bmap;
    cudaError_t e = codes_map(&map, q, a.E, a.N, a.K);
    if (e != cudaSuccess) return e;
    e = rows_map(&bmap, brows, nbrows, a.K, kTcMaxN);
    if (e != cudaSuccess) return e;
    static int configured[128];
    e = ensure_smem(tc_kernel<MODE>, configured, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(tc_kernel<MODE>, num_sms, kTcThreads, smem, stream, a, map, bmap);
}

// xs[r] = x[token of sorted row r], each 8-element block in the
// dequantiser's pair order (rows of invalid pairs: zeros).  Step 3 then
// reads the activation rows of a chunk as one contiguous tile.
__global__ void sorted_rows_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ sorted_pair, int k,
                                   int P, int H8, uint4 *__restrict__ xs) {
    pdl_wait();
    pdl_trigger();
    const long long n = (long long)P * H8;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(i / H8), c = (int)(i - (long long)r * H8);
        const int pr = __ldg(sorted_pair + r);
        xs[i] = (pr >= 0 && pr < P) ? pair_interleave(__ldg(x + (size_t)(pr / k) * H8 + c)) : make_uint4(0, 0, 0, 0);
    }
}

}  // namespace

// Shapes the tensor-core path takes: fp16 activations with K a multiple of
// 32 (groups) and enough rows per expert on average to fill MMA granules.
bool tc_supported(int T, int E, int k, int H, int I, size_t smem_limit) {
    const int amax = E < T * k ? E : T * k;
    return T >= kTcMinT && H % 32 == 0 && I % 32 == 0 && encode_fn() != nullptr &&
           tc_smem_bytes(TcGeom<kTcGateUp>::a_bytes, 2, TcGeom<kTcGateUp>::t_bytes, 4) + 16 + tc_table_bytes(amax) <=
               smem_limit;
}

cudaError_t launch_gate_up_tc(const __half *x, const uint32_t *q, const __half *s, const uint32_t *z,
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
    return launch_tc<kTcGateUp>(a, q, xperm, (long long)T * k, num_sms, smem_limit, stream);
}

cudaError_t launch_combine(const float *y, const float *topk_w, int T, int k, int H, __half *out,
                           cudaStream_t stream);

cudaError_t launch_down_tc(const __half *h, const uint32_t *q, const __half *s, const uint32_t *z,
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
    cudaError_t e = launch_tc<kTcDown>(a, q, h, (long long)T * k, num_sms, smem_limit, stream);
    if (e != cudaSuccess) return e;
    return launch_combine(y, topk_w, T, k, H, out, stream);
}

}  // namespace moe
