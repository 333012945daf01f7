// decode_layer_nvfp4_b.cu -- instantiations of the one-launch decode layer
// kernel (decode_layer.cuh) for NVFP4 weights: the narrower lane splits.
#include "decode_layer.cuh"

namespace moe {

template cudaError_t launch_layer_t<4, 0, 4, 0, kFmtNvfp4>(const LayerArgs &, const LayerPlan &, int, cudaStream_t);
template cudaError_t launch_layer_t<4, 0, 1, 0, kFmtNvfp4>(const LayerArgs &, const LayerPlan &, int, cudaStream_t);
template cudaError_t launch_layer_t<1, 0, 4, 0, kFmtNvfp4>(const LayerArgs &, const LayerPlan &, int, cudaStream_t);
template cudaError_t launch_layer_t<1, 0, 1, 0, kFmtNvfp4>(const LayerArgs &, const LayerPlan &, int, cudaStream_t);

}  // namespace moe
