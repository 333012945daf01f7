// decode_gemv.cu -- the decode step kernels (decode_gemv.cuh) for W4A16 g32
// weights: the launchers the C entry points call.
#include "decode_gemv.cuh"

namespace moe {

bool decode_supported(int T, int E, int k, int H, int I, size_t smem_limit) {
    return decode_supported_impl(T, E, k, H, I, smem_limit);
}

cudaError_t launch_gate_up_decode(const __half *x, const uint32_t *q, const __half *s, const uint32_t *z,
                                  const int32_t *offsets, const int32_t *sorted_pair,
                                  const int32_t *active, const int32_t *num_active, int T, int E, int k,
                                  int H, int I, __half *h, uint32_t *err, int num_sms, size_t smem_limit,
                                  cudaStream_t stream) {
    return launch_gate_up_decode_f<kFmtW4A16>(x, q, s, z, offsets, sorted_pair, active, num_active, T, E, k, H, I,
                                              h, err, num_sms, smem_limit, stream);
}

cudaError_t launch_down_decode(const __half *h, const uint32_t *q, const __half *s, const uint32_t *z,
                               const int32_t *offsets, const int32_t *sorted_pair, const int32_t *active,
                               const int32_t *num_active, const float *topk_w, int T, int E, int k, int H,
                               int I, __half *out, float *y, uint32_t *counters, uint32_t *err,
                               int num_sms, size_t smem_limit, cudaStream_t stream) {
    return launch_down_decode_f<kFmtW4A16>(h, q, s, z, offsets, sorted_pair, active, num_active, topk_w, T, E, k,
                                           H, I, out, y, counters, err, num_sms, smem_limit, stream);
}

}  // namespace moe
