// capi.cu -- the extern "C" boundary of libmoe_w4a16 (declared, with the
// meaning, layout, ownership and error behaviour of every argument, in
// include/moe_w4a16.h).  Host code only: argument validation, cached device
// attributes, and kernel dispatch.
#include <mutex>

#include "common.cuh"
#include "dispatch_table.cuh"

#define MOE_EXPORT extern "C" __attribute__((visibility("default")))

namespace moe {
cudaError_t launch_route(const float *, int, int, int, int32_t *, float *, cudaStream_t);
cudaError_t launch_align(const int32_t *, int, int, int32_t *, int32_t *, int32_t *, int32_t *,
                         uint32_t *, size_t, cudaStream_t);
cudaError_t launch_gate_up_stream(const __half *, const uint32_t *, const __half *, const uint32_t *,
                                  const int32_t *, const int32_t *, const int32_t *, const int32_t *,
                                  int, int, int, int, int, __half *, uint32_t *, int, size_t,
                                  cudaStream_t);
cudaError_t launch_down_stream(const __half *, const uint32_t *, const __half *, const uint32_t *,
                               const int32_t *, const int32_t *, const int32_t *, const int32_t *,
                               const float *, int, int, int, int, int, __half *, float *, uint32_t *,
                               uint32_t *, int, size_t, cudaStream_t);

bool decode_supported(int, int, int, int, int, size_t);
bool route_align_fusable(int, int, int, size_t);
cudaError_t launch_route_align(const float *, int, int, int, int32_t *, float *, int32_t *, int32_t *,
                               int32_t *, int32_t *, uint32_t *, cudaStream_t);
cudaError_t launch_gate_up_decode(const __half *, const uint32_t *, const __half *, const uint32_t *,
                                  const int32_t *, const int32_t *, const int32_t *, const int32_t *,
                                  int, int, int, int, int, __half *, uint32_t *, int, size_t,
                                  cudaStream_t);
cudaError_t launch_down_decode(const __half *, const uint32_t *, const __half *, const uint32_t *,
                               const int32_t *, const int32_t *, const int32_t *, const int32_t *,
                               const float *, int, int, int, int, int, __half *, float *, uint32_t *,
                               uint32_t *, int, size_t, cudaStream_t);

bool tc_supported(int, int, int, int, int, size_t);
cudaError_t launch_gate_up_tc(const __half *, const uint32_t *, const __half *, const uint32_t *,
                              const int32_t *, const int32_t *, const int32_t *, const int32_t *, int, int,
                              int, int, int, __half *, __half *, uint32_t *, int, size_t, cudaStream_t);
cudaError_t launch_down_tc(const __half *, const uint32_t *, const __half *, const uint32_t *,
                           const int32_t *, const int32_t *, const int32_t *, const int32_t *, const float *,
                           int, int, int, int, int, __half *, float *, uint32_t *, int, size_t, cudaStream_t);
bool layer_fusable(int, int, int, int, int, int, size_t);
cudaError_t launch_decode_layer(const float *, const __half *, const uint32_t *, const __half *,
                                const uint32_t *, const uint32_t *, const __half *, const uint32_t *,
                                int, int, int, int, int, int32_t *, float *, __half *, __half *,
                                float *, uint32_t *, uint32_t *, uint32_t *, uint32_t *, int, size_t,
                                cudaStream_t);

cudaError_t launch_gate_up_decode_nvfp4(const __half *, const uint32_t *, const uint8_t *, const float *,
                                        const int32_t *, const int32_t *, const int32_t *, const int32_t *, int,
                                        int, int, int, int, __half *, uint32_t *, int, size_t, cudaStream_t);
cudaError_t launch_down_decode_nvfp4(const __half *, const uint32_t *, const uint8_t *, const float *,
                                     const int32_t *, const int32_t *, const int32_t *, const int32_t *,
                                     const float *, int, int, int, int, int, __half *, float *, uint32_t *,
                                     uint32_t *, int, size_t, cudaStream_t);
cudaError_t launch_gate_up_tc_nvfp4(const __half *, const uint32_t *, const uint8_t *, const float *,
                                    const int32_t *, const int32_t *, const int32_t *, const int32_t *, int, int,
                                    int, int, int, __half *, __half *, uint32_t *, int, size_t, cudaStream_t);
cudaError_t launch_down_tc_nvfp4(const __half *, const uint32_t *, const uint8_t *, const float *,
                                 const int32_t *, const int32_t *, const int32_t *, const int32_t *, const float *,
                                 int, int, int, int, int, __half *, float *, uint32_t *, int, size_t, cudaStream_t);
cudaError_t launch_layer_floor(int, int, int, int, int, int, size_t, cudaStream_t);
cudaError_t launch_decode_layer_nvfp4(const float *, const __half *, const uint32_t *, const uint8_t *,
                                      const float *, const uint32_t *, const uint8_t *, const float *, int, int,
                                      int, int, int, int32_t *, float *, __half *, __half *, float *, uint32_t *,
                                      uint32_t *, uint32_t *, uint32_t *, int, size_t, cudaStream_t);

bool router_fusable(int, int, int, int, size_t);
int router_path(int, int, int, size_t);
cudaError_t launch_router_logits(const __half *, const __half *, int, int, int, float *, uint32_t *, int, size_t,
                                 cudaStream_t);
cudaError_t launch_router_route_align(const __half *, const __half *, int, int, int, int, float *, int32_t *,
                                      float *, int32_t *, int32_t *, int32_t *, int32_t *, uint32_t *, int,
                                      cudaStream_t);
cudaError_t launch_awq_import(const uint32_t *, const uint32_t *, const uint16_t *, int, int, int, uint32_t *,
                              uint16_t *, uint32_t *, int, int, cudaStream_t);

namespace {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr long long kMaxPairs = 1LL << 24;
constexpr int kMaxDim = 1 << 16;

struct DeviceInfo {
    int sms = 0;
    size_t smem_optin = 0;
};

std::mutex g_mu;
DeviceInfo g_info[128];

// SM count and opt-in shared memory of the current device, queried once.
cudaError_t device_info(DeviceInfo *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_info[dev].sms == 0) {
        int sms = 0, smem = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        g_info[dev].sms = sms;
        g_info[dev].smem_optin = (size_t)smem;
    }
    *out = g_info[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sizes shared by every call.  H or I <= 0 means "not used by this call".
int check_sizes(int T, int E, int k, int H, int I) {
    if (T < 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (H != -1 && (H <= 0 || H % 32)) return MOE_ERR_INVALID_ARG;
    if (I != -1 && (I <= 0 || I % 32)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxE || k > kMaxK || (long long)T * k > kMaxPairs) return MOE_ERR_UNSUPPORTED;
    if (H > kMaxDim || I > kMaxDim) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int check_group(int group_size) {
    if (group_size <= 0) return MOE_ERR_INVALID_ARG;
    return group_size == 32 ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

template <typename... Ps>
bool all_aligned(const Ps *...ps) {
    bool ok = true;
    ((ok = ok && ps != nullptr && aligned16(ps)), ...);
    return ok;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool path_value_ok(int path) {
    return path == MOE_PATH_AUTO || path == MOE_PATH_DECODE || path == MOE_PATH_TENSOR_CORE ||
           path == MOE_PATH_STREAM;
}

bool path_supported(int path, int T, int E, int k, int H, int I, size_t smem) {
    switch (path) {
        case MOE_PATH_DECODE: return decode_supported(T, E, k, H, I, smem);
        case MOE_PATH_TENSOR_CORE: return tc_supported(T, E, k, H, I, smem);
        case MOE_PATH_STREAM: return true;
        default: return false;
    }
}

// The kernels of the step calls for a shape: the per-shape table's measured
// choice where it has one (and the path can take the shape), else by shape
// alone: the latency-first decode kernels up to 16 tokens while their
// shared-memory layout fits (at 9 and 10 tokens on the Qwen4Exp geometry
// 123 and 137 us through the step calls, against 216 and 231 us on the
// tensor cores), then the tensor cores, the stream kernels only where
// neither fits.  A forced path the shape cannot take is
// MOE_ERR_UNSUPPORTED.
constexpr int kRuleDecodeMaxT = 16;

// NVFP4 weights: the decode kernels by the same rule, else the tensor cores
// (no stream kernels for this format); MOE_PATH_NONE if neither fits.
int nvfp4_path(int T, int E, int k, int H, int I, size_t smem) {
    if (T <= kRuleDecodeMaxT && decode_supported(T, E, k, H, I, smem)) return MOE_PATH_DECODE;
    if (tc_supported(T, E, k, H, I, smem)) return MOE_PATH_TENSOR_CORE;
    return MOE_PATH_NONE;
}
int resolve_path(int *path, int T, int E, int k, int H, int I, size_t smem) {
    if (*path != MOE_PATH_AUTO) {
        if (!path_value_ok(*path)) return MOE_ERR_INVALID_ARG;
        return path_supported(*path, T, E, k, H, I, smem) ? MOE_OK : MOE_ERR_UNSUPPORTED;
    }
    const int tp = tuned_path(T, E, k, H, I);
    if (tp != MOE_PATH_AUTO && path_supported(tp, T, E, k, H, I, smem))
        *path = tp;
    else if (T <= kRuleDecodeMaxT && decode_supported(T, E, k, H, I, smem))
        *path = MOE_PATH_DECODE;
    else if (tc_supported(T, E, k, H, I, smem))
        *path = MOE_PATH_TENSOR_CORE;
    else
        *path = MOE_PATH_STREAM;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_EXPORT int moe_abi_version(void) { return 1; }

MOE_EXPORT const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported size or option";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_DEVICE_FLAG: return "device kernel flagged invalid data";
        default: return "unknown status";
    }
}

MOE_EXPORT size_t moe_workspace_bytes(int T, int E, int k, int H, int I) {
    if (check_sizes(T, E, k, H, I) != MOE_OK) return 0;
    return workspace_layout(T, k, H).total;
}

MOE_EXPORT int moe_get_device_error(void *workspace, size_t ws_bytes, uint32_t *flag_out,
                                    void *stream) {
    if (!workspace || !flag_out || ws_bytes < kCtrlBytes || !aligned16(workspace))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && v) {
        e = cudaMemsetAsync(workspace, 0, sizeof(v), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    *flag_out = v;
    return v ? MOE_ERR_DEVICE_FLAG : MOE_OK;
}

MOE_EXPORT int moe_step_kernel_path(int T, int E, int k, int H, int I) {
    if (check_sizes(T, E, k, H, I) != MOE_OK) return MOE_PATH_NONE;
    if (T == 0) return MOE_PATH_NONE;
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess) return MOE_PATH_NONE;
    int path = MOE_PATH_AUTO;
    return resolve_path(&path, T, E, k, H, I, di.smem_optin) == MOE_OK ? path : MOE_PATH_NONE;
}

MOE_EXPORT int moe_topk_route(const float *logits, int T, int E, int k, int32_t *topk_ids,
                              float *topk_w, void *stream) {
    int st = check_sizes(T, E, k, -1, -1);
    if (st != MOE_OK) return st;
    if (!all_aligned(logits, topk_ids, topk_w)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    return cuda_status(launch_route(logits, T, E, k, topk_ids, topk_w, static_cast<cudaStream_t>(stream)));
}

MOE_EXPORT int moe_align_offsets(const int32_t *topk_ids, int T, int E, int k,
                                 int32_t *expert_offsets, int32_t *sorted_pair,
                                 int32_t *active_experts, int32_t *num_active, void *workspace,
                                 size_t ws_bytes, void *stream) {
    int st = check_sizes(T, E, k, -1, -1);
    if (st != MOE_OK) return st;
    if (!all_aligned(expert_offsets, active_experts, num_active)) return MOE_ERR_INVALID_ARG;
    // with no pairs the id and pair buffers are empty and may be NULL
    if (T > 0 && !all_aligned(topk_ids, sorted_pair)) return MOE_ERR_INVALID_ARG;
    if (workspace && (ws_bytes < kCtrlBytes || !aligned16(workspace))) return MOE_ERR_WORKSPACE;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    // T == 0 still defines the outputs: empty segments, no active experts
    return cuda_status(launch_align(topk_ids, T * k, E, expert_offsets, sorted_pair, active_experts,
                                    num_active, static_cast<uint32_t *>(workspace), di.smem_optin,
                                    static_cast<cudaStream_t>(stream)));
}

MOE_EXPORT int moe_topk_route_align(const float *logits, int T, int E, int k, int32_t *topk_ids,
                                    float *topk_w, int32_t *expert_offsets, int32_t *sorted_pair,
                                    int32_t *active_experts, int32_t *num_active, void *workspace,
                                    size_t ws_bytes, void *stream) {
    int st = check_sizes(T, E, k, -1, -1);
    if (st != MOE_OK) return st;
    if (!all_aligned(expert_offsets, active_experts, num_active)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && !all_aligned(logits, topk_ids, topk_w, sorted_pair)) return MOE_ERR_INVALID_ARG;
    if (workspace && (ws_bytes < kCtrlBytes || !aligned16(workspace))) return MOE_ERR_WORKSPACE;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t *err = static_cast<uint32_t *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > 0 && route_align_fusable(T, E, k, di.smem_optin))
        return cuda_status(launch_route_align(logits, T, E, k, topk_ids, topk_w, expert_offsets,
                                              sorted_pair, active_experts, num_active, err, s));
    if (T > 0) {
        e = launch_route(logits, T, E, k, topk_ids, topk_w, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    return cuda_status(launch_align(topk_ids, T * k, E, expert_offsets, sorted_pair, active_experts,
                                    num_active, err, di.smem_optin, s));
}

MOE_EXPORT int moe_w4a16_gate_up_silu_ex(const uint16_t *x, const uint32_t *w13_q,
                                         const uint16_t *w13_s, const uint32_t *w13_z, int group_size,
                                         const int32_t *expert_offsets, const int32_t *sorted_pair,
                                         const int32_t *active_experts, const int32_t *num_active,
                                         int T, int E, int k, int H, int I, uint16_t *h,
                                         void *workspace, size_t ws_bytes, int path, void *stream) {
    int st = check_sizes(T, E, k, H, I);
    if (st != MOE_OK) return st;
    if ((st = check_group(group_size)) != MOE_OK) return st;
    if (!all_aligned(x, w13_q, w13_s, w13_z, expert_offsets, sorted_pair, active_experts,
                     num_active, h) || !path_value_ok(path))
        return MOE_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < moe_workspace_bytes(T, E, k, H, I))
        return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t *err = static_cast<uint32_t *>(workspace) + kCtrlErrorWord;
    if ((st = resolve_path(&path, T, E, k, H, I, di.smem_optin)) != MOE_OK) return st;
    if (path == MOE_PATH_DECODE)
        return cuda_status(launch_gate_up_decode(
            reinterpret_cast<const __half *>(x), w13_q, reinterpret_cast<const __half *>(w13_s), w13_z,
            expert_offsets, sorted_pair, active_experts, num_active, T, E, k, H, I,
            reinterpret_cast<__half *>(h), err, di.sms, di.smem_optin, static_cast<cudaStream_t>(stream)));
    if (path == MOE_PATH_TENSOR_CORE)
        return cuda_status(launch_gate_up_tc(
            reinterpret_cast<const __half *>(x), w13_q, reinterpret_cast<const __half *>(w13_s), w13_z,
            expert_offsets, sorted_pair, active_experts, num_active, T, E, k, H, I,
            reinterpret_cast<__half *>(h),
            // scratch for the sorted x rows: the per-pair y area, unused until step 4
            reinterpret_cast<__half *>(static_cast<uint8_t *>(workspace) + workspace_layout(T, k, H).y), err,
            di.sms, di.smem_optin, static_cast<cudaStream_t>(stream)));
    e = launch_gate_up_stream(reinterpret_cast<const __half *>(x), w13_q,
                              reinterpret_cast<const __half *>(w13_s), w13_z, expert_offsets,
                              sorted_pair, active_experts, num_active, T, E, k, H, I,
                              reinterpret_cast<__half *>(h), err, di.sms, di.smem_optin,
                              static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

MOE_EXPORT int moe_w4a16_gate_up_silu(const uint16_t *x, const uint32_t *w13_q,
                                      const uint16_t *w13_s, const uint32_t *w13_z, int group_size,
                                      const int32_t *expert_offsets, const int32_t *sorted_pair,
                                      const int32_t *active_experts, const int32_t *num_active,
                                      int T, int E, int k, int H, int I, uint16_t *h,
                                      void *workspace, size_t ws_bytes, void *stream) {
    return moe_w4a16_gate_up_silu_ex(x, w13_q, w13_s, w13_z, group_size, expert_offsets, sorted_pair,
                                     active_experts, num_active, T, E, k, H, I, h, workspace, ws_bytes,
                                     MOE_PATH_AUTO, stream);
}

namespace moe {
// Every argument check of moe_w4a16_down_combine except the workspace's
// (shared with the allocation-free variant, which must reject a call before
// it touches its scratch).
int check_down_combine_args(const uint16_t *h, const uint32_t *w2_q, const uint16_t *w2_s,
                            const uint32_t *w2_z, int group_size, const int32_t *expert_offsets,
                            const int32_t *sorted_pair, const int32_t *active_experts,
                            const int32_t *num_active, const float *topk_w, int T, int E, int k, int H,
                            int I, const uint16_t *out) {
    int st = check_sizes(T, E, k, H, I);
    if (st != MOE_OK) return st;
    if ((st = check_group(group_size)) != MOE_OK) return st;
    if (!all_aligned(h, w2_q, w2_s, w2_z, expert_offsets, sorted_pair, active_experts, num_active,
                     topk_w, out))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}
}  // namespace moe

MOE_EXPORT int moe_w4a16_down_combine_ex(const uint16_t *h, const uint32_t *w2_q, const uint16_t *w2_s,
                                         const uint32_t *w2_z, int group_size,
                                         const int32_t *expert_offsets, const int32_t *sorted_pair,
                                         const int32_t *active_experts, const int32_t *num_active,
                                         const float *topk_w, int T, int E, int k, int H, int I,
                                         uint16_t *out, void *workspace, size_t ws_bytes, int path,
                                         void *stream) {
    int st = check_down_combine_args(h, w2_q, w2_s, w2_z, group_size, expert_offsets, sorted_pair,
                                     active_experts, num_active, topk_w, T, E, k, H, I, out);
    if (st != MOE_OK) return st;
    if (!path_value_ok(path)) return MOE_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < moe_workspace_bytes(T, E, k, H, I))
        return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    const WorkspaceLayout L = workspace_layout(T, k, H);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws) + kCtrlErrorWord;
    if ((st = resolve_path(&path, T, E, k, H, I, di.smem_optin)) != MOE_OK) return st;
    if (path == MOE_PATH_DECODE)
        return cuda_status(launch_down_decode(
            reinterpret_cast<const __half *>(h), w2_q, reinterpret_cast<const __half *>(w2_s), w2_z,
            expert_offsets, sorted_pair, active_experts, num_active, topk_w, T, E, k, H, I,
            reinterpret_cast<__half *>(out), reinterpret_cast<float *>(ws + L.y),
            reinterpret_cast<uint32_t *>(ws + L.counters), err, di.sms, di.smem_optin,
            static_cast<cudaStream_t>(stream)));
    if (path == MOE_PATH_TENSOR_CORE)
        return cuda_status(launch_down_tc(
            reinterpret_cast<const __half *>(h), w2_q, reinterpret_cast<const __half *>(w2_s), w2_z,
            expert_offsets, sorted_pair, active_experts, num_active, topk_w, T, E, k, H, I,
            reinterpret_cast<__half *>(out), reinterpret_cast<float *>(ws + L.y), err, di.sms, di.smem_optin,
            static_cast<cudaStream_t>(stream)));
    e = launch_down_stream(reinterpret_cast<const __half *>(h), w2_q,
                           reinterpret_cast<const __half *>(w2_s), w2_z, expert_offsets, sorted_pair,
                           active_experts, num_active, topk_w, T, E, k, H, I,
                           reinterpret_cast<__half *>(out), reinterpret_cast<float *>(ws + L.y),
                           reinterpret_cast<uint32_t *>(ws + L.counters), err, di.sms,
                           di.smem_optin, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

MOE_EXPORT int moe_w4a16_down_combine(const uint16_t *h, const uint32_t *w2_q, const uint16_t *w2_s,
                                      const uint32_t *w2_z, int group_size,
                                      const int32_t *expert_offsets, const int32_t *sorted_pair,
                                      const int32_t *active_experts, const int32_t *num_active,
                                      const float *topk_w, int T, int E, int k, int H, int I,
                                      uint16_t *out, void *workspace, size_t ws_bytes,
                                      void *stream) {
    return moe_w4a16_down_combine_ex(h, w2_q, w2_s, w2_z, group_size, expert_offsets, sorted_pair,
                                     active_experts, num_active, topk_w, T, E, k, H, I, out, workspace,
                                     ws_bytes, MOE_PATH_AUTO, stream);
}

namespace moe {
namespace {

// The layer call's workspace: the workspace of steps 3 and 4 (control
// words, block counters, per-pair y), then the grouping outputs, h, and the
// per-expert and exit counters of the one-launch decode layer.
struct LayerWorkspace {
    size_t offsets, sorted, active, num_active, h, done, exitctr, total;
};

LayerWorkspace layer_workspace(int T, int E, int k, int H, int I) {
    LayerWorkspace L;
    const size_t P = (size_t)T * k;
    L.offsets = workspace_layout(T, k, H).total;
    L.sorted = L.offsets + align_up((size_t)(E + 1) * 4, 256);
    L.active = L.sorted + align_up(P * 4, 256);
    L.num_active = L.active + align_up((size_t)E * 4, 256);
    L.h = L.num_active + 256;
    L.done = L.h + align_up(P * I * 2, 256);
    L.exitctr = L.done + align_up(P * 4, 256);
    L.total = L.exitctr + 256;
    return L;
}

}  // namespace
}  // namespace moe

MOE_EXPORT size_t moe_layer_workspace_bytes(int T, int E, int k, int H, int I) {
    if (check_sizes(T, E, k, H, I) != MOE_OK) return 0;
    return layer_workspace(T, E, k, H, I).total;
}

MOE_EXPORT int moe_decode_layer_floor(int T, int E, int k, int H, int I, void *stream) {
    int st = check_sizes(T, E, k, H, I);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess) return MOE_ERR_CUDA;
    if (!layer_fusable(T, E, k, H, I, di.sms, di.smem_optin)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(launch_layer_floor(T, E, k, H, I, di.sms, di.smem_optin, static_cast<cudaStream_t>(stream)));
}

MOE_EXPORT int moe_w4a16_moe_layer(const float *logits, const uint16_t *x, const uint32_t *w13_q,
                                   const uint16_t *w13_s, const uint32_t *w13_z, const uint32_t *w2_q,
                                   const uint16_t *w2_s, const uint32_t *w2_z, int group_size, int T,
                                   int E, int k, int H, int I, int32_t *topk_ids, float *topk_w,
                                   uint16_t *out, void *workspace, size_t ws_bytes, void *stream) {
    int st = check_sizes(T, E, k, H, I);
    if (st != MOE_OK) return st;
    if ((st = check_group(group_size)) != MOE_OK) return st;
    if (!all_aligned(w13_q, w13_s, w13_z, w2_q, w2_s, w2_z)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && !all_aligned(logits, x, topk_ids, topk_w, out)) return MOE_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < moe_layer_workspace_bytes(T, E, k, H, I))
        return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const WorkspaceLayout W = workspace_layout(T, k, H);
    const LayerWorkspace L = layer_workspace(T, E, k, H, I);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws) + kCtrlErrorWord;
    if (layer_fusable(T, E, k, H, I, di.sms, di.smem_optin))
        return cuda_status(launch_decode_layer(
            logits, reinterpret_cast<const __half *>(x), w13_q, reinterpret_cast<const __half *>(w13_s),
            w13_z, w2_q, reinterpret_cast<const __half *>(w2_s), w2_z, T, E, k, H, I, topk_ids, topk_w,
            reinterpret_cast<__half *>(out), reinterpret_cast<__half *>(ws + L.h),
            reinterpret_cast<float *>(ws + W.y), reinterpret_cast<uint32_t *>(ws + W.counters),
            reinterpret_cast<uint32_t *>(ws + L.done), reinterpret_cast<uint32_t *>(ws + L.exitctr), err,
            di.sms, di.smem_optin, s));
    // the four steps as separate launches
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    int32_t *sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
    int32_t *active = reinterpret_cast<int32_t *>(ws + L.active);
    int32_t *num_active = reinterpret_cast<int32_t *>(ws + L.num_active);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h);
    // routing and grouping as two launches: ahead of the decode step kernels
    // this measured 10-12 us faster than the one-launch route+align (9-16
    // tokens on the Qwen4Exp geometry), and the same ahead of the tensor cores
    if ((st = moe_topk_route(logits, T, E, k, topk_ids, topk_w, stream)) != MOE_OK) return st;
    if ((st = moe_align_offsets(topk_ids, T, E, k, offsets, sorted, active, num_active, workspace, ws_bytes,
                                stream)) != MOE_OK)
        return st;
    if ((st = moe_w4a16_gate_up_silu(x, w13_q, w13_s, w13_z, group_size, offsets, sorted, active,
                                     num_active, T, E, k, H, I, h, workspace, ws_bytes, stream)) != MOE_OK)
        return st;
    return moe_w4a16_down_combine(h, w2_q, w2_s, w2_z, group_size, offsets, sorted, active, num_active,
                                  topk_w, T, E, k, H, I, out, workspace, ws_bytes, stream);
}


// ---------------------------------------------------------------- NVFP4 weights
MOE_EXPORT int moe_nvfp4_gate_up_silu(const uint16_t *x, const uint32_t *w13_codes, const uint8_t *w13_bscale,
                                      const float *w13_gscale, const int32_t *expert_offsets,
                                      const int32_t *sorted_pair, const int32_t *active_experts,
                                      const int32_t *num_active, int T, int E, int k, int H, int I, uint16_t *h,
                                      void *workspace, size_t ws_bytes, void *stream) {
    int st = check_sizes(T, E, k, H, I);
    if (st != MOE_OK) return st;
    if (!all_aligned(x, w13_codes, w13_bscale, w13_gscale, expert_offsets, sorted_pair, active_experts,
                     num_active, h))
        return MOE_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < moe_workspace_bytes(T, E, k, H, I))
        return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t *err = static_cast<uint32_t *>(workspace) + kCtrlErrorWord;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int path = nvfp4_path(T, E, k, H, I, di.smem_optin);
    if (path == MOE_PATH_DECODE)
        return cuda_status(launch_gate_up_decode_nvfp4(
            reinterpret_cast<const __half *>(x), w13_codes, w13_bscale, w13_gscale, expert_offsets, sorted_pair,
            active_experts, num_active, T, E, k, H, I, reinterpret_cast<__half *>(h), err, di.sms, di.smem_optin, s));
    if (path == MOE_PATH_TENSOR_CORE)
        return cuda_status(launch_gate_up_tc_nvfp4(
            reinterpret_cast<const __half *>(x), w13_codes, w13_bscale, w13_gscale, expert_offsets, sorted_pair,
            active_experts, num_active, T, E, k, H, I, reinterpret_cast<__half *>(h),
            reinterpret_cast<__half *>(static_cast<uint8_t *>(workspace) + workspace_layout(T, k, H).y), err,
            di.sms, di.smem_optin, s));
    return MOE_ERR_UNSUPPORTED;  // the staged stream kernels read W4A16 weights only
}

MOE_EXPORT int moe_nvfp4_down_combine(const uint16_t *h, const uint32_t *w2_codes, const uint8_t *w2_bscale,
                                      const float *w2_gscale, const int32_t *expert_offsets,
                                      const int32_t *sorted_pair, const int32_t *active_experts,
                                      const int32_t *num_active, const float *topk_w, int T, int E, int k, int H,
                                      int I, uint16_t *out, void *workspace, size_t ws_bytes, void *stream) {
    int st = check_sizes(T, E, k, H, I);
    if (st != MOE_OK) return st;
    if (!all_aligned(h, w2_codes, w2_bscale, w2_gscale, expert_offsets, sorted_pair, active_experts, num_active,
                     topk_w, out))
        return MOE_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < moe_workspace_bytes(T, E, k, H, I))
        return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    const WorkspaceLayout L = workspace_layout(T, k, H);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws) + kCtrlErrorWord;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int path = nvfp4_path(T, E, k, H, I, di.smem_optin);
    if (path == MOE_PATH_DECODE)
        return cuda_status(launch_down_decode_nvfp4(
            reinterpret_cast<const __half *>(h), w2_codes, w2_bscale, w2_gscale, expert_offsets, sorted_pair,
            active_experts, num_active, topk_w, T, E, k, H, I, reinterpret_cast<__half *>(out),
            reinterpret_cast<float *>(ws + L.y), reinterpret_cast<uint32_t *>(ws + L.counters), err, di.sms,
            di.smem_optin, s));
    if (path == MOE_PATH_TENSOR_CORE)
        return cuda_status(launch_down_tc_nvfp4(
            reinterpret_cast<const __half *>(h), w2_codes, w2_bscale, w2_gscale, expert_offsets, sorted_pair,
            active_experts, num_active, topk_w, T, E, k, H, I, reinterpret_cast<__half *>(out),
            reinterpret_cast<float *>(ws + L.y), err, di.sms, di.smem_optin, s));
    return MOE_ERR_UNSUPPORTED;
}

MOE_EXPORT int moe_nvfp4_moe_layer(const float *logits, const uint16_t *x, const uint32_t *w13_codes,
                                   const uint8_t *w13_bscale, const float *w13_gscale, const uint32_t *w2_codes,
                                   const uint8_t *w2_bscale, const float *w2_gscale, int T, int E, int k, int H,
                                   int I, int32_t *topk_ids, float *topk_w, uint16_t *out, void *workspace,
                                   size_t ws_bytes, void *stream) {
    int st = check_sizes(T, E, k, H, I);
    if (st != MOE_OK) return st;
    if (!all_aligned(w13_codes, w13_bscale, w13_gscale, w2_codes, w2_bscale, w2_gscale)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && !all_aligned(logits, x, topk_ids, topk_w, out)) return MOE_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < moe_layer_workspace_bytes(T, E, k, H, I))
        return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const WorkspaceLayout W = workspace_layout(T, k, H);
    const LayerWorkspace L = layer_workspace(T, E, k, H, I);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws) + kCtrlErrorWord;
    if (layer_fusable(T, E, k, H, I, di.sms, di.smem_optin))
        return cuda_status(launch_decode_layer_nvfp4(
            logits, reinterpret_cast<const __half *>(x), w13_codes, w13_bscale, w13_gscale, w2_codes, w2_bscale,
            w2_gscale, T, E, k, H, I, topk_ids, topk_w, reinterpret_cast<__half *>(out),
            reinterpret_cast<__half *>(ws + L.h), reinterpret_cast<float *>(ws + W.y),
            reinterpret_cast<uint32_t *>(ws + W.counters), reinterpret_cast<uint32_t *>(ws + L.done),
            reinterpret_cast<uint32_t *>(ws + L.exitctr), err, di.sms, di.smem_optin, s));
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    int32_t *sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
    int32_t *active = reinterpret_cast<int32_t *>(ws + L.active);
    int32_t *num_active = reinterpret_cast<int32_t *>(ws + L.num_active);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h);
    if (nvfp4_path(T, E, k, H, I, di.smem_optin) == MOE_PATH_NONE)
        return MOE_ERR_UNSUPPORTED;  // checked before anything is launched
    if ((st = moe_topk_route(logits, T, E, k, topk_ids, topk_w, stream)) != MOE_OK) return st;
    if ((st = moe_align_offsets(topk_ids, T, E, k, offsets, sorted, active, num_active, workspace, ws_bytes,
                                stream)) != MOE_OK)
        return st;
    if ((st = moe_nvfp4_gate_up_silu(x, w13_codes, w13_bscale, w13_gscale, offsets, sorted, active, num_active, T,
                                     E, k, H, I, h, workspace, ws_bytes, stream)) != MOE_OK)
        return st;
    return moe_nvfp4_down_combine(h, w2_codes, w2_bscale, w2_gscale, offsets, sorted, active, num_active, topk_w,
                                  T, E, k, H, I, out, workspace, ws_bytes, stream);
}


// ---------------------------------------------------------------- router logits
MOE_EXPORT int moe_router_logits(const uint16_t *x, const uint16_t *w_router, int T, int E, int H, float *logits,
                                 void *workspace, size_t ws_bytes, void *stream) {
    int st = check_sizes(T, E, 1, H, -1);
    if (st != MOE_OK) return st;
    if (!all_aligned(w_router)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && !all_aligned(x, logits)) return MOE_ERR_INVALID_ARG;
    if (workspace && (ws_bytes < kCtrlBytes || !aligned16(workspace))) return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (router_path(T, E, H, di.smem_optin) == 0) return MOE_ERR_UNSUPPORTED;
    uint32_t *err = workspace ? static_cast<uint32_t *>(workspace) + kCtrlErrorWord : nullptr;
    return cuda_status(launch_router_logits(reinterpret_cast<const __half *>(x),
                                            reinterpret_cast<const __half *>(w_router), T, E, H, logits, err,
                                            di.sms, di.smem_optin, static_cast<cudaStream_t>(stream)));
}

MOE_EXPORT int moe_router_route_align(const uint16_t *x, const uint16_t *w_router, int T, int E, int k, int H,
                                      float *logits, int32_t *topk_ids, float *topk_w, int32_t *expert_offsets,
                                      int32_t *sorted_pair, int32_t *active_experts, int32_t *num_active,
                                      void *workspace, size_t ws_bytes, void *stream) {
    int st = check_sizes(T, E, k, H, -1);
    if (st != MOE_OK) return st;
    if (!all_aligned(w_router, expert_offsets, active_experts, num_active)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && !all_aligned(x, logits, topk_ids, topk_w, sorted_pair)) return MOE_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < kCtrlBytes || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > 0 && router_fusable(T, E, k, H, di.smem_optin))
        return cuda_status(launch_router_route_align(
            reinterpret_cast<const __half *>(x), reinterpret_cast<const __half *>(w_router), T, E, k, H, logits,
            topk_ids, topk_w, expert_offsets, sorted_pair, active_experts, num_active,
            static_cast<uint32_t *>(workspace), di.sms, s));
    if (T > 0 && router_path(T, E, H, di.smem_optin) == 0) return MOE_ERR_UNSUPPORTED;
    if ((st = moe_router_logits(x, w_router, T, E, H, logits, workspace, ws_bytes, stream)) != MOE_OK) return st;
    return moe_topk_route_align(logits, T, E, k, topk_ids, topk_w, expert_offsets, sorted_pair, active_experts,
                                num_active, workspace, ws_bytes, stream);
}

// ---------------------------------------------------------------- AWQ import
MOE_EXPORT int moe_awq_import(const uint32_t *awq_qweight, const uint32_t *awq_qzeros,
                              const uint16_t *awq_scales, int E, int K, int N, int group_size,
                              uint32_t *qweight, uint16_t *scales, uint32_t *qzeros, int N_dst, int row0,
                              void *stream) {
    if (E <= 0 || K <= 0 || N <= 0 || K % 32 || N % 8 || N_dst <= 0 || N_dst % 8 || row0 < 0 || row0 % 8 ||
        (long long)row0 + N > N_dst)
        return MOE_ERR_INVALID_ARG;
    int st = check_group(group_size);
    if (st != MOE_OK) return st;
    if (E > kMaxE || K > kMaxDim || N_dst > 2 * kMaxDim) return MOE_ERR_UNSUPPORTED;
    if (!all_aligned(awq_qweight, awq_qzeros, awq_scales, qweight, scales, qzeros)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_awq_import(awq_qweight, awq_qzeros, awq_scales, E, K, N, qweight, scales, qzeros,
                                         N_dst, row0, static_cast<cudaStream_t>(stream)));
}
