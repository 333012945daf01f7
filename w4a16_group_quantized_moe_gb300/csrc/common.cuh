// common.cuh -- device helpers shared by the libmoe_w4a16 kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_w4a16.h"

namespace moe {

// ---------------------------------------------------------------- workspace
// Control block at the start of the workspace.
constexpr size_t kCtrlBytes = 256;
constexpr int kCtrlErrorWord = 0;     // u32: MOE_DEVERR_* bits
// Diagnostic words of the control block (zero in a zero-filled workspace,
// which selects the defaults); see MOE_CTRL_* in moe_w4a16.h.
constexpr int kCtrlWaitPolls = MOE_CTRL_WAIT_POLLS;  // u32: polls before a cross-CTA wait gives up
constexpr int kCtrlWaitExtra = MOE_CTRL_WAIT_EXTRA;  // u32: added to every cross-CTA wait target
constexpr int kCtrlTimeline = MOE_CTRL_TIMELINE;     // u64 (words 4-5): timeline buffer address
constexpr int kCtrlRouterTicket = 8;  // u32: CTAs of the fused router launch that have finished (0 between calls)

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace regions after the control block (all 256-byte aligned).
struct WorkspaceLayout {
    size_t counters;   // u32 [H/8]: arrivals per 8-row output block (down, decode)
    size_t y;          // f32 [P][H]: per-pair down projection
    size_t total;
};

__host__ __device__ inline WorkspaceLayout workspace_layout(int T, int k, int H) {
    WorkspaceLayout L;
    L.counters = kCtrlBytes;
    L.y = L.counters + align_up((size_t)(H / 8) * 4, 256);
    L.total = L.y + align_up((size_t)T * k * H * 4, 256);
    return L;
}

__device__ inline void set_error(uint32_t *err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

// ---------------------------------------------------------------- PTX wrappers
__device__ inline uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ inline void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ inline void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ inline void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Waits (suspended, not spinning) for the phase of `parity` to complete, for
// at most about kSuspendHintNs; returns whether it completed.
constexpr uint32_t kSuspendHintNs = 1000000;

__device__ inline bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Non-blocking test of a barrier phase (one instruction when already done).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on a barrier phase.  Gives up after about a second (far
// beyond any legitimate wait here) and returns false so the caller can flag
// the error and leave instead of hanging the GPU.  `abort_flag` (shared)
// lets one thread's failure release every other waiter of the CTA.
constexpr uint32_t kWaitTries = 1024;

__device__ inline bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                         volatile int *abort_flag) {
    for (uint32_t it = 0; it < kWaitTries; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag && *abort_flag) return false;
    }
    return false;
}

// Orders this thread's earlier generic-proxy accesses to shared memory
// before its later async-proxy (bulk copy) accesses.
__device__ inline void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ inline void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 16-byte read of data used once (packed weights): read-only path, not kept
// in L1.
__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Acquire load (gpu scope) of a counter written by other CTAs.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Nanoseconds of the GPU's global timer (for the optional phase timeline).
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One warp-level MMA, D = A.B + C: A 16x16 fp16 (row), B 16x8 fp16 (col),
// C and D 16x8 fp32.  Fragment of lane l (group g = l / 4, t = l % 4):
// a[0] = A[g][2t..2t+1], a[1] = A[g+8][2t..2t+1], a[2] = A[g][2t+8..2t+9],
// a[3] = A[g+8][2t+8..2t+9]; b[0] = B[2t..2t+1][g], b[1] = B[2t+8..2t+9][g];
// c[0..1] = C[g][2t..2t+1], c[2..3] = C[g+8][2t..2t+1].
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Named barrier for a subset of the CTA's warps (id 0 is __syncthreads).
__device__ inline void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Arrival at a named barrier without waiting (the producer side of a
// producer/consumer hand-off: the consumers bar.sync on the same id).
__device__ inline void named_barrier_arrive(int id, int threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- dependent launch
// Programmatic dependent launch: every kernel of the library is launched
// with programmatic stream serialisation, so it can be scheduled while its
// predecessor on the stream is still running.  Protocol, for every kernel:
// nothing before pdl_wait() reads global memory (only barrier set-up runs
// there); pdl_wait() returns once the predecessor grid has completed and its
// writes are visible; pdl_trigger() right after lets the successor start its
// own set-up.  So every kernel still sees all earlier work on the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Raises a kernel's dynamic shared-memory limit once per device and size.
template <typename K>
inline cudaError_t ensure_smem(K kernel, int *configured /* [128] */, size_t smem) {
    if (smem <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    if (configured[dev] >= (int)smem) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) configured[dev] = (int)smem;
    return e;
}

// ---------------------------------------------------------------- int4 dequant
// Codes of one 32-bit word (8 codes, code j in bits 4j..4j+3) minus the zero
// point, as four fp16 pairs, straight from the binary16 format: 0x6400 is
// 1024.0 and binary16 values in [1024, 2048) are spaced exactly 1 apart, so
// OR-ing a 4-bit field into the low mantissa bits gives exactly 1024 + code,
// and a field sitting at bits 4..7 gives exactly 1024 + 16*code.  Subtracting
// (1024 + z), or scaling by 1/16 and subtracting (64 + z) in one fused
// multiply-add, leaves code - z exactly (a small integer).  Two codes per
// instruction, with no integer-to-float conversion.
//
// Output pairing: d[0] = (c0, c4), d[1] = (c1, c5), d[2] = (c2, c6),
// d[3] = (c3, c7) (low half first).  Activations are staged in the matching
// order [a0 a4 a1 a5 a2 a6 a3 a7] per block of eight.
struct ZeroPoint {
    __half2 z1024;    // (1024 + z, 1024 + z)
    __half2 neg_z64;  // (-(64 + z), -(64 + z))
};

__device__ inline ZeroPoint make_zero_point(uint32_t z) {
    ZeroPoint zp;
    uint32_t bits = (0x6400u | z) * 0x00010001u;
    zp.z1024 = *reinterpret_cast<__half2 *>(&bits);
    zp.neg_z64 = __hsub2(__float2half2_rn(960.0f), zp.z1024);
    return zp;
}

// (a & mask) | 0x64006400 as one three-input logic instruction.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or_6400(uint32_t a) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "n"(MASK), "n"(0x64006400u));
    return r;
}

__device__ inline void dequant_word(uint32_t w, const ZeroPoint &zp, __half2 *d) {
    const uint32_t lo = and_or_6400<0x000F000Fu>(w);
    const uint32_t hi = and_or_6400<0x00F000F0u>(w);
    const uint32_t w8 = w >> 8;
    const uint32_t lo2 = and_or_6400<0x000F000Fu>(w8);
    const uint32_t hi2 = and_or_6400<0x00F000F0u>(w8);
    const __half2 sixteenth = __float2half2_rn(0.0625f);
    d[0] = __hsub2(*reinterpret_cast<const __half2 *>(&lo), zp.z1024);
    d[1] = __hfma2(*reinterpret_cast<const __half2 *>(&hi), sixteenth, zp.neg_z64);
    d[2] = __hsub2(*reinterpret_cast<const __half2 *>(&lo2), zp.z1024);
    d[3] = __hfma2(*reinterpret_cast<const __half2 *>(&hi2), sixteenth, zp.neg_z64);
}

// Reorders eight fp16 values [a0..a7] (one uint4) into the pairing used by
// dequant_word: [a0 a4 a1 a5 a2 a6 a3 a7].
__device__ inline uint4 pair_interleave(uint4 v) {
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    return o;
}

__device__ inline __half2 u32_as_half2(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }

}  // namespace moe
