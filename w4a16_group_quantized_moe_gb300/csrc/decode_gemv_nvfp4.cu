// decode_gemv_nvfp4.cu -- the decode step kernels (decode_gemv.cuh) for
// NVFP4 weights (E2M1 codes, E4M3 scales per 16 elements, fp32 scale per
// expert matrix): the launchers the NVFP4 C entry points call.  q holds the
// codes, s the E4M3 scale bytes and z the per-expert scales (as float).
#include "decode_gemv.cuh"

namespace moe {

cudaError_t launch_gate_up_decode_nvfp4(const __half *x, const uint32_t *q, const uint8_t *s, const float *gs,
                                        const int32_t *offsets, const int32_t *sorted_pair,
                                        const int32_t *active, const int32_t *num_active, int T, int E, int k,
                                        int H, int I, __half *h, uint32_t *err, int num_sms, size_t smem_limit,
                                        cudaStream_t stream) {
    return launch_gate_up_decode_f<kFmtNvfp4>(x, q, reinterpret_cast<const __half *>(s),
                                              reinterpret_cast<const uint32_t *>(gs), offsets, sorted_pair, active,
                                              num_active, T, E, k, H, I, h, err, num_sms, smem_limit, stream);
}

cudaError_t launch_down_decode_nvfp4(const __half *h, const uint32_t *q, const uint8_t *s, const float *gs,
                                     const int32_t *offsets, const int32_t *sorted_pair, const int32_t *active,
                                     const int32_t *num_active, const float *topk_w, int T, int E, int k, int H,
                                     int I, __half *out, float *y, uint32_t *counters, uint32_t *err,
                                     int num_sms, size_t smem_limit, cudaStream_t stream) {
    return launch_down_decode_f<kFmtNvfp4>(h, q, reinterpret_cast<const __half *>(s),
                                           reinterpret_cast<const uint32_t *>(gs), offsets, sorted_pair, active,
                                           num_active, topk_w, T, E, k, H, I, out, y, counters, err, num_sms,
                                           smem_limit, stream);
}

}  // namespace moe
