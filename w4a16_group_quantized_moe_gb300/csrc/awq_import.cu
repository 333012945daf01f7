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
// One CTA per tile of 256 K rows x 64 output columns of one expert: it reads
// the tile's 8 KB of codes (each K row's 32 contiguous bytes), the 8 groups
// of scales and zeros, into shared memory, then writes each of the 64 output
// rows' 128 contiguous bytes of codes (two 16-byte stores per thread), the
// rows' scales and the 8 zero words.  Both sides move whole 32-byte sectors:
// the kernel is a copy bound by HBM.
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

__global__ void __launch_bounds__(kAwqThreads) awq_import_kernel(const AwqArgs a) {
    __shared__ uint32_t t_codes[kAwqKT][kAwqNT / 8];
    __shared__ uint16_t t_scales[kAwqKT / 32][kAwqNT];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x;
    const int e = blockIdx.z;
    const int k0 = blockIdx.x * kAwqKT, n0 = blockIdx.y * kAwqNT;
    const int W = a.N / 8, G = a.K / 32;
    const int c0 = n0 / 8, g0 = k0 / 32;
    const uint32_t *aq = a.aq + (size_t)e * a.K * W;
    // codes: 8 words per K row, 4 rows per warp instruction
#pragma unroll
    for (int i = 0; i < kAwqKT * (kAwqNT / 8) / kAwqThreads; ++i) {
        const int idx = tid + i * kAwqThreads;
        const int kr = idx >> 3, c = idx & 7;
        const bool ok = k0 + kr < a.K && c0 + c < W;
        t_codes[kr][c] = ok ? __ldg(aq + (size_t)(k0 + kr) * W + c0 + c) : 0u;
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
    // codes out: thread = (column n, quarter qq of the tile's 32 words per row)
    {
        const int n = tid & (kAwqNT - 1), qq = tid >> 6;
        const int sl = awq_slot(n & 7), cw = n >> 3;
        const size_t KW = (size_t)a.K / 8;
        const int kw0 = k0 / 8 + qq * 8;  // first output word of this thread
        if (n0 + n < a.N && kw0 < (int)KW) {
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t v = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) v |= ((t_codes[(qq * 8 + i) * 8 + j][cw] >> (4 * sl)) & 0xFu) << (4 * j);
                o[i] = v;
            }
            uint4 *dst = reinterpret_cast<uint4 *>(a.q + ((size_t)e * a.Ndst + a.row0 + n0 + n) * KW + kw0);
            // K is a multiple of 32, so the words left in a row come in fours
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            if (kw0 + 4 < (int)KW) dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
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
