// noalloc.cu -- step 4 for callers that cannot allocate device memory.
//
// Some callers of this library are not allowed to call cudaMalloc: an
// inference engine that plans all of its device memory before it starts
// serving and forbids allocation afterwards, a plugin loaded into a host
// application that owns every allocator, or a latency-critical loop where an
// allocation could synchronise the device.  They still need somewhere for
// the per-pair fp32 projections and the block counters that the down/combine
// step keeps in its workspace.  This file gives them a fixed scratch array
// that lives in the library itself: every GPU that loads the library holds
// it, at its full size, until the process exits.
#include <mutex>

#include "common.cuh"

#define MOE_EXPORT extern "C" __attribute__((visibility("default")))

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;

// The scratch.  In host code this name is only a stand-in for the device
// array, never an address a kernel could use; the real device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[128];  // per device, looked up once

// Device address of the scratch on the current device.  The first call on a
// device performs the lookup (with that device current).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace moe

MOE_EXPORT int moe_w4a16_down_combine_noalloc(const uint16_t *h, const uint32_t *w2_q,
                                              const uint16_t *w2_s, const uint32_t *w2_z,
                                              int group_size, const int32_t *expert_offsets,
                                              const int32_t *sorted_pair,
                                              const int32_t *active_experts,
                                              const int32_t *num_active, const float *topk_w, int T,
                                              int E, int k, int H, int I, uint16_t *out,
                                              void *stream) {
    const size_t need = moe_workspace_bytes(T, E, k, H, I);
    if (need == 0)  // sizes rejected: let the regular call report which error, before any launch
        return moe_w4a16_down_combine(h, w2_q, w2_s, w2_z, group_size, expert_offsets, sorted_pair,
                                      active_experts, num_active, topk_w, T, E, k, H, I, out, nullptr,
                                      0, stream);
    if (need > moe::kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (moe::scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    // the control block and the block counters must start at zero; the
    // per-pair projections are fully rewritten by every call
    const size_t zero_bytes = moe::workspace_layout(T, k, H).y;
    if (T > 0 && cudaMemsetAsync(scratch, 0, zero_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return moe_w4a16_down_combine(h, w2_q, w2_s, w2_z, group_size, expert_offsets, sorted_pair,
                                  active_experts, num_active, topk_w, T, E, k, H, I, out, scratch,
                                  moe::kNoAllocScratchBytes, stream);
}
