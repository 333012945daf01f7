// awq_import.cu -- repack of AWQ checkpoint layers into the layer's layout.
//
// The public AWQ "GEMM" packing of a linear layer with input size K and
// output size N stores
//     qweight u32 [K][N/8]     nibble i of word [kk][c] = code of column 8c + ORDER[i]
//     qzeros  u32 [K/32][N/8]  nibble i of word [g][c]  = zero of column 8c + ORDER[i]
//     scales  f16 [K/32][N]
//     ORDER = (0, 2, 4, 6, 1, 3, 5, 7)
// while the layer reads W[N][K] with codes along K in natural nibble order,
// scales [N][K/32] and zeros packed along N (moe_w4a16.h).  So the codes
// are a transpose at 4-bit granularity, the scales a 16-bit transpose, and
// each zero word only a permutation of its own nibbles (output row
// r = 8b + j holds the nibble of column j, which sits in slot
// (j >> 1) | ((j & 1) << 2) of the AWQ word).
//
// One CTA per tile of 256 K rows x 64 output columns of one expert.  Each
// thread loads 8 code words: the same 8 columns (one AWQ word) on 8
// consecutive K rows; as a matrix of nibbles (row = K row, column = word
// slot) that is an 8x8 block, and its transpose is 8 words of the layer's
// layout (word s = the 8 K codes of the column in slot s).  The transpose is
// three rounds of masked shift/xor swaps between word pairs (blocks of 4,
// 8 and 16 bits), about nine instructions per word, all in registers.  The
// words go through a padded shared-memory tile so that each output row's
// 128 contiguous bytes are written by one warp; scales (a 16-bit transpose)
// take the same route, and each zero word is a nibble permutation of one
// AWQ word.  Loads and stores move whole 32-byte sectors: the kernel is a
// copy bound by HBM.
#include "common.cuh"

namespace moe {

constexpr int kAwqThreads = 256;
constexpr int kAwqKT = 256;  // K rows per tile (32 output words per row)
constexpr int kAwqNT = 64;   // output columns per tile (8 AWQ words per K row)

// slot of column j (0..7) in an AWQ word: the inverse of ORDER
__device__ __forceinline__ int awq_slot(int j) { return (j >> 1) | ((j & 1) << 2); }

struct AwqArgs {
    const uint32_t *aq, *az;
    const uint16_t *as;
    int K, N, Ndst, row0;
    uint32_t *q, *z;
    uint16_t *s;
};

// Transposes the 8x8 nibble matrix held in a[0..7] (a[i] nibble s ->
// a[s] nibble i): swaps of 4-bit blocks between words i, i+1, of 8-bit
// blocks between i, i+2, of 16-bit blocks between i, i+4.
__device__ __forceinline__ void transpose_nibbles(uint32_t (&a)[8]) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const uint32_t x = ((a[i] >> 4) ^ a[i + 1]) & 0x0F0F0F0Fu;
        a[i + 1] ^= x;
        a[i] ^= x << 4;
    }
#pragma unroll
    for (int i = 0; i < 8; i += (i & 1) ? 3 : 1) {  // 0, 1, 4, 5
        const uint32_t x = ((a[i] >> 8) ^ a[i + 2]) & 0x00FF00FFu;
        a[i + 2] ^= x;
        a[i] ^= x << 8;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t x = ((a[i] >> 16) ^ a[i + 4]) & 0x0000FFFFu;
        a[i + 4] ^= x;
        a[i] ^= x << 16;
    }
}

__global__ void __launch_bounds__(kAwqThreads) awq_import_kernel(const AwqArgs a) {
    __shared__ uint32_t t_out[kAwqNT][kAwqKT / 8 + 1];  // [output row][output word], padded
    __shared__ uint16_t t_scales[kAwqKT / 32][kAwqNT];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x;
    const int e = blockIdx.z;
    const int k0 = blockIdx.x * kAwqKT, n0 = blockIdx.y * kAwqNT;
    const int W = a.N / 8, G = a.K / 32;
    const int c0 = n0 / 8, g0 = k0 / 32;
    const uint32_t *aq = a.aq + (size_t)e * a.K * W;
    // codes: thread = (AWQ word cw of the tile, 8 K rows from 8 * kq)
    {
        const int cw = tid & 7, kq = tid >> 3;
        const int kr = k0 + 8 * kq;
        uint32_t v[8];
        const bool ok = kr < a.K && c0 + cw < W;  // K is a multiple of 8: all 8 rows or none
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = ok ? __ldg(aq + (size_t)(kr + i) * W + c0 + cw) : 0u;
        transpose_nibbles(v);
        // word s now holds the 8 codes of column 8 cw + ORDER[s]
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
            const int j = (sl & 3) * 2 + (sl >> 2);  // ORDER[sl]
            t_out[8 * cw + j][kq] = v[sl];
        }
    }
    // scales: 8 groups x 64 columns
#pragma unroll
    for (int i = 0; i < (kAwqKT / 32) * kAwqNT / kAwqThreads; ++i) {
        const int idx = tid + i * kAwqThreads;
        const int gi = idx / kAwqNT, n = idx % kAwqNT;
        const bool ok = g0 + gi < G && n0 + n < a.N;
        t_scales[gi][n] = ok ? __ldg(a.as + ((size_t)e * G + g0 + gi) * a.N + n0 + n) : (uint16_t)0;
    }
    // zeros: one word per (column word, group), a permutation of its nibbles
    if (tid < (kAwqNT / 8) * (kAwqKT / 32)) {
        const int c = tid / (kAwqKT / 32), gi = tid % (kAwqKT / 32);
        if (c0 + c < W && g0 + gi < G) {
            const uint32_t v = __ldg(a.az + ((size_t)e * G + g0 + gi) * W + c0 + c);
            uint32_t o = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) o |= ((v >> (4 * awq_slot(j))) & 0xFu) << (4 * j);
            a.z[((size_t)e * (a.Ndst / 8) + (a.row0 + n0) / 8 + c) * G + g0 + gi] = o;
        }
    }
    __syncthreads();
    // codes out: one warp per output row, lane = word of the row (128 bytes)
    {
        const size_t KW = (size_t)a.K / 8;
        const int lane = tid & 31;
        const int kw = k0 / 8 + lane;
        for (int n = tid >> 5; n < kAwqNT; n += kAwqThreads / 32)
            if (n0 + n < a.N && kw < (int)KW)
                a.q[((size_t)e * a.Ndst + a.row0 + n0 + n) * KW + kw] = t_out[n][lane];
    }
    // scales out: 8 consecutive groups of each row
#pragma unroll
    for (int i = 0; i < (kAwqKT / 32) * kAwqNT / kAwqThreads; ++i) {
        const int idx = tid + i * kAwqThreads;
        const int n = idx / (kAwqKT / 32), gi = idx % (kAwqKT / 32);
        if (g0 + gi < G && n0 + n < a.N)
            a.s[((size_t)e * a.Ndst + a.row0 + n0 + n) * G + g0 + gi] = t_scales[gi][n];
    }
}

cudaError_t launch_awq_import(const uint32_t *aq, const uint32_t *az, const uint16_t *as, int E, int K, int N,
                              uint32_t *q, uint16_t *s, uint32_t *z, int Ndst, int row0, cudaStream_t stream) {
    AwqArgs a{aq, az, as, K, N, Ndst, row0, q, z, s};
    const dim3 grid((unsigned)((K + kAwqKT - 1) / kAwqKT), (unsigned)((N + kAwqNT - 1) / kAwqNT), (unsigned)E);
    return launch_pdl(awq_import_kernel, grid, kAwqThreads, 0, stream, a);
}

}  // namespace moe
