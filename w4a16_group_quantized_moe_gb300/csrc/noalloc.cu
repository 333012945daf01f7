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
int check_down_combine_args(const uint16_t *, const uint32_t *, const uint16_t *, const uint32_t *, int,
                            const int32_t *, const int32_t *, const int32_t *, const int32_t *,
                            const float *, int, int, int, int, int, const uint16_t *);
namespace {

constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;

// The scratch.  In host code this name is only a stand-in for the device
// array, never an address a kernel could use; the real device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[128];  // per device: the last address looked up

// Device address of the scratch on the current device.  Outside stream
// capture the address is looked up again on every call (cheap), so a device
// reset that reloads the module never leaves a stale pointer behind; during
// capture (where the lookup could count as a capture-unsafe call) the address
// of the last call on this device is reused, so the first call on a device
// must come before any capture.
cudaError_t scratch_address(cudaStream_t stream, void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    } else if (g_scratch_addr[dev] == nullptr) {
        return cudaErrorStreamCaptureUnsupported;
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
    // every argument check first: a rejected call launches nothing and
    // leaves the shared scratch as it was
    const int st = moe::check_down_combine_args(h, w2_q, w2_s, w2_z, group_size, expert_offsets,
                                                sorted_pair, active_experts, num_active, topk_w, T, E, k,
                                                H, I, out);
    if (st != MOE_OK) return st;
    if (moe_workspace_bytes(T, E, k, H, I) > moe::kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *scratch = nullptr;
    if (moe::scratch_address(s, &scratch) != cudaSuccess) return MOE_ERR_CUDA;
    // the control block and the block counters must start at zero; the
    // per-pair projections are fully rewritten by every call
    const size_t zero_bytes = moe::workspace_layout(T, k, H).y;
    if (cudaMemsetAsync(scratch, 0, zero_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    return moe_w4a16_down_combine(h, w2_q, w2_s, w2_z, group_size, expert_offsets, sorted_pair,
                                  active_experts, num_active, topk_w, T, E, k, H, I, out, scratch,
                                  moe::kNoAllocScratchBytes, stream);
}
