// decode_common.cuh -- the pieces of the decode weight stream shared by the
// per-step decode kernels (decode_gemv.cu) and the one-launch decode layer
// (decode_layer.cu): the per-warp task buffer and the bulk-copy ranges of a
// task, the activation cache layout, and the dequantise-and-accumulate loop.
#pragma once
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

// Weight formats of the expert matrices:
//   kFmtW4A16: AWQ-style uint4 codes, uint4 zero points and fp16 scales per
//              32 elements along K; w = (q - z) * s
//   kFmtNvfp4: E2M1 codes, an FP8 E4M3 scale per 16 elements along K (the
//              two scales of a 32-element group sit where the fp16 group
//              scale sits in the W4A16 layout: the same bytes per row) and
//              an fp32 scale per expert matrix (passed where the W4A16 zero
//              words are); w = e2m1(q) * e4m3(s) * scale[e]
enum { kFmtW4A16 = 0, kFmtNvfp4 = 1 };

// The eight E2M1 codes of one 32-bit word (code j in bits 4j..4j+3) as four
// fp16 pairs in dequant_word's pairing: d[0] = (c0, c4), d[1] = (c1, c5),
// d[2] = (c2, c6), d[3] = (c3, c7).  Each pair is gathered into one byte
// (low nibble first) and converted by the CUDA fp4 intrinsic.
__device__ __forceinline__ void e2m1_word(uint32_t w, __half2 *d) {
    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;  // c0 c2 c4 c6 / c1 c3 c5 c7
    const uint32_t L = lo | (lo >> 12), Hh = hi | (hi >> 12);            // bytes (c0 c4) (c2 c6), (c1 c5) (c3 c7)
    const __half2_raw r0 = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)(L & 0xFFu), __NV_E2M1);
    const __half2_raw r1 = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)(Hh & 0xFFu), __NV_E2M1);
    const __half2_raw r2 = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((L >> 8) & 0xFFu), __NV_E2M1);
    const __half2_raw r3 = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((Hh >> 8) & 0xFFu), __NV_E2M1);
    d[0] = __half2(r0);
    d[1] = __half2(r1);
    d[2] = __half2(r2);
    d[3] = __half2(r3);
}

// The two E4M3 scales of a 32-element group (the low byte covers its first
// 16 elements) as floats.
__device__ __forceinline__ float2 e4m3_pair(uint16_t v) {
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
    return __half22float2(__half2(r));
}

constexpr int kDecPass = 4;   // activation rows per compute pass
constexpr int kGPI = 2;       // groups per lane worked on together

enum { kDecGateUp = 0, kDecDown = 1 };

// Per-warp buffer for a task of RT rows in each of nmat matrices: codes,
// then scales, then zero words of every matrix; scale and zero copies are
// widened to 16-byte boundaries, hence the slack.
struct WarpGeom {
    uint32_t q_bytes, s_bytes, z_bytes, bytes;
};

__host__ __device__ inline WarpGeom warp_geom(int RT, int nmat, int K) {
    const int G = K / 32;
    WarpGeom g;
    g.q_bytes = (uint32_t)(RT * K / 2);
    g.s_bytes = (uint32_t)align_up((size_t)RT * G * 2 + 32, 16);
    // a task starts on a multiple of min(RT, 8) rows, so it spans
    // ceil(RT / 8) zero-word rows
    g.z_bytes = (uint32_t)align_up((size_t)((RT + 7) / 8) * G * 4 + 32, 16);
    g.bytes = (uint32_t)align_up((size_t)nmat * (g.q_bytes + g.s_bytes + g.z_bytes), 128);
    return g;
}


// Byte ranges (from the tensor bases) of one matrix block of a task: rows
// [n_first, n_first + cnt) of expert e; scale and zero ranges widened to
// 16-byte boundaries (the tensors' sizes are multiples of 16 bytes).
struct WarpCopy {
    size_t q_off;
    uint32_t q_len;
    uint32_t s_skip;   // bytes from the copied scale range's start to the first row
    size_t s_a;
    uint32_t s_len;
    uint32_t z_skip;
    size_t z_a;
    uint32_t z_len;
};

__device__ __forceinline__ WarpCopy warp_copy(int e, int n_first, int cnt, int N, int K) {
    const int G = K / 32;
    WarpCopy c;
    const size_t row = (size_t)e * N + n_first;
    c.q_off = row * (size_t)(K / 2);
    c.q_len = (uint32_t)(cnt * (K / 2));
    const size_t s_lo = row * G * 2, s_hi = (row + cnt) * G * 2;
    c.s_a = s_lo & ~(size_t)15;
    c.s_skip = (uint32_t)(s_lo - c.s_a);
    c.s_len = (uint32_t)(align_up(s_hi, 16) - c.s_a);
    const size_t zr0 = (size_t)e * (N / 8) + n_first / 8;
    const size_t zr1 = (size_t)e * (N / 8) + (n_first + cnt - 1) / 8;
    const size_t z_lo = zr0 * G * 4;
    c.z_a = z_lo & ~(size_t)15;
    c.z_skip = (uint32_t)(z_lo - c.z_a);
    c.z_len = (uint32_t)(align_up((zr1 + 1) * G * 4, 16) - c.z_a);
    return c;
}

// shared activation cache: slot s, 8-element block kb = 4*g + wd stored at
// ((s*4 + wd)*G + g)*16 bytes (consecutive groups -> consecutive banks)
__device__ __forceinline__ uint32_t dec_xoff(int slot, int kb, int G) {
    return (uint32_t)(((slot * 4 + (kb & 3)) * G + (kb >> 2)) * 16);
}

__device__ __forceinline__ uint32_t dec_word(const uint4 &w, int i) {
    return i == 0 ? w.x : (i == 1 ? w.y : (i == 2 ? w.z : w.w));
}

// Sizes the compute loop needs: matrix rows per expert N, reduction length
// K, row units per expert, pairs P and top-k.
struct TaskDims {
    int N, K, rows, P, k;
};

template <int MODE, int L, int RU>
struct DecTraits {
    static constexpr int nmat = MODE == kDecGateUp ? 2 : 1;
    static constexpr int UPW = 32 / L;  // row units per warp step
    static constexpr int RT = UPW * RU; // row units per task
};

// The task a warp works on: RT row units of expert e from unit0, and the
// token pass tb (activation rows r0+tb .. r0+tb+3 of the segment).
struct Cursor {
    int e, unit0, cnt, r0, ne, tb;
};

// Dequantise the warp's buffered task and accumulate against NT activation
// rows.  GT = groups per row when known at compile time (0: read from a.K).
// The kGPI groups of a step are worked on together, each product sum in up
// to four independent fp16 chains.
//
// Activation rows: step 3 reads token p / k of pair p from cache slot p / k
// (s_tok[r], when given, holds that token for sorted row r);
// step 4 reads sorted row r from cache slot r - slot_base or, when vin is
// given, straight from vin[r][K] in global memory.
template <int MODE, int L, int RU, int GT, int NT, int FMT = kFmtW4A16>
__device__ __forceinline__ void dec_compute(const uint8_t *wb, const WarpGeom &wg,
                                            float (&acc)[RU][DecTraits<MODE, L, RU>::nmat][kDecPass],
                                            const Cursor &c, const int *s_pairs, const uint8_t *xcb,
                                            int slot_base, const __half *vin, const TaskDims &a,
                                            int lane, const int *s_tok = nullptr, float gsc = 1.f) {
    using Tr = DecTraits<MODE, L, RU>;
    constexpr int nmat = Tr::nmat;
    // independent chains per product sum; with NVFP4 the two chains are the
    // group's two 16-element blocks, each with its own scale
    constexpr int CH = FMT == kFmtNvfp4 ? 2 : (NT == 1 ? 4 : (NT == 2 ? 2 : 1));
    const int G = GT ? GT : a.K / 32;
    const int K = 32 * G;
    const int GL = (G + L - 1) / L;  // groups per lane (compile time when GT != 0)
    const int ks = lane % L, us = lane / L;
    const uint8_t *xb[NT];  // this lane's first block of each activation row
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int r = c.r0 + c.tb + t;
        int slot;
        if (MODE == kDecGateUp) {
            if (s_tok) {
                slot = s_tok[r];
            } else {
                const int p = s_pairs[r];
                slot = (p >= 0 && p < a.P) ? p / a.k : 0;
            }
        } else {
            slot = r - slot_base;
        }
        xb[t] = xcb + (size_t)slot * 4 * G * 16 + ks * 16;
    }
    uint32_t soff[nmat], zoff[nmat];
    int nfirst[nmat];
#pragma unroll
    for (int b = 0; b < nmat; ++b) {
        nfirst[b] = c.unit0 + b * a.rows;
        // the copies' 16-byte widening: only the low four bits of the byte
        // offsets matter, so 32-bit products (wrapping) give them exactly
        const uint32_t row = (uint32_t)c.e * (uint32_t)a.N + (uint32_t)nfirst[b];
        const uint32_t zrow = (uint32_t)c.e * (uint32_t)(a.N / 8) + (uint32_t)(nfirst[b] / 8);
        soff[b] = nmat * wg.q_bytes + b * wg.s_bytes + ((row * (uint32_t)G * 2u) & 15u);
        zoff[b] = nmat * (wg.q_bytes + wg.s_bytes) + b * wg.z_bytes + ((zrow * (uint32_t)G * 4u) & 15u);
    }
#pragma unroll
    for (int ru = 0; ru < RU; ++ru) {
        const int lr = us + ru * Tr::UPW;  // row within the task
        if (lr >= c.cnt) continue;
        const uint8_t *qp[nmat], *sp[nmat], *zp[nmat];
        uint32_t zsh[nmat];
#pragma unroll
        for (int b = 0; b < nmat; ++b) {
            const int n = nfirst[b] + lr;
            qp[b] = wb + b * wg.q_bytes + lr * (K / 2) + ks * 16;
            sp[b] = wb + soff[b] + (lr * G + ks) * 2;
            zp[b] = wb + zoff[b] + ((n / 8 - nfirst[b] / 8) * G + ks) * 4;
            zsh[b] = 4 * (n & 7);
        }
#pragma unroll
        for (int m0 = 0; m0 < GL; m0 += kGPI) {
            uint4 w[nmat][kGPI];
            float sc[nmat][kGPI], sc2[nmat][kGPI];  // NVFP4: the scales of the two blocks
            ZeroPoint zq[nmat][kGPI];
            bool gok[kGPI];
#pragma unroll
            for (int i = 0; i < kGPI; ++i) {
                const int m = m0 + i;
                // with G a multiple of L (and GT known) this folds to a constant
                gok[i] = (GT && GT % L == 0) ? m < GL : ks + L * m < G;
#pragma unroll
                for (int b = 0; b < nmat; ++b) {
                    if (gok[i]) {
                        w[b][i] = *reinterpret_cast<const uint4 *>(qp[b] + L * 16 * m);
                        if (FMT == kFmtNvfp4) {
                            const float2 s2 = e4m3_pair(*reinterpret_cast<const uint16_t *>(sp[b] + L * 2 * m));
                            sc[b][i] = s2.x * gsc;
                            sc2[b][i] = s2.y * gsc;
                        } else {
                            sc[b][i] = __half2float(*reinterpret_cast<const __half *>(sp[b] + L * 2 * m));
                            zq[b][i] = make_zero_point(
                                (*reinterpret_cast<const uint32_t *>(zp[b] + L * 4 * m) >> zsh[b]) & 0xFu);
                        }
                    } else {
                        // groups past G: zero codes, zero point 0, scale 0
                        w[b][i] = make_uint4(0, 0, 0, 0);
                        sc[b][i] = sc2[b][i] = 0.f;
                        if (FMT != kFmtNvfp4) zq[b][i] = make_zero_point(0u);
                    }
                }
            }
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
                    const int m = m0 + i;
                    __half2 dq[nmat][4];
#pragma unroll
                    for (int b = 0; b < nmat; ++b) {
                        if (FMT == kFmtNvfp4)
                            e2m1_word(dec_word(w[b][i], wd), dq[b]);
                        else
                            dequant_word(dec_word(w[b][i], wd), zq[b][i], dq[b]);
                    }
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        // activations of groups past G read as zero so sums stay finite
                        uint4 X = make_uint4(0, 0, 0, 0);
                        if (gok[i]) {
                            if (MODE == kDecGateUp || vin == nullptr) {
                                X = *reinterpret_cast<const uint4 *>(xb[t] + (wd * G + L * m) * 16);
                            } else {
                                const int g = ks + L * m;
                                X = pair_interleave(__ldg(reinterpret_cast<const uint4 *>(
                                    vin + (size_t)(c.r0 + c.tb + t) * K + g * 32 + wd * 8)));
                            }
                        }
#pragma unroll
                        for (int b = 0; b < nmat; ++b) {
                            __half2 &h = hs[i][b][t][FMT == kFmtNvfp4 ? wd / 2 : wd % CH];
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
                        if (FMT == kFmtNvfp4) {
                            const float2 f0 = __half22float2(hs[i][b][t][0]), f1 = __half22float2(hs[i][b][t][1]);
                            acc[ru][b][t] = fmaf(sc[b][i], f0.x + f0.y, fmaf(sc2[b][i], f1.x + f1.y, acc[ru][b][t]));
                        } else {
                            __half2 s2 = hs[i][b][t][0];
#pragma unroll
                            for (int ch = 1; ch < CH; ++ch) s2 = __hadd2(s2, hs[i][b][t][ch]);
                            const float2 f = __half22float2(s2);
                            acc[ru][b][t] = fmaf(sc[b][i], f.x + f.y, acc[ru][b][t]);
                        }
                    }
        }
    }
}


// Cooperative copy of n activation rows (starting at src) into cache slots
// 0..n-1, pair-interleaved; every thread issues its loads before any store.
__device__ __forceinline__ void dec_stage_rows(const __half *src, int n, int K, int G, uint8_t *xcb,
                                               int tid, int nthreads) {
    const int KB = K / 8, nx = n * KB;
    for (int base = 0; base < nx; base += 16 * nthreads) {
        uint4 v[16];  // up to 16 loads in flight per thread: one round trip for most batches
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int i = base + tid + c * nthreads;
            v[c] = i < nx ? __ldg(reinterpret_cast<const uint4 *>(src) + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int i = base + tid + c * nthreads;
            if (i < nx) *reinterpret_cast<uint4 *>(xcb + dec_xoff(i / KB, i % KB, G)) = pair_interleave(v[c]);
        }
    }
}

}  // namespace moe
