// decode_layer_nvfp4_a.cu -- instantiations of the one-launch decode layer
// kernel (decode_layer.cuh) for NVFP4 weights: the specified geometries and
// the widest generic lane split.
#include "decode_layer.cuh"

namespace moe {

template cudaError_t launch_layer_t<16, 80, 4, 20, kFmtNvfp4>(const LayerArgs &, const LayerPlan &, int, cudaStream_t);
template cudaError_t launch_layer_t<16, 80, 1, 5, kFmtNvfp4>(const LayerArgs &, const LayerPlan &, int, cudaStream_t);
template cudaError_t launch_layer_t<16, 0, 4, 0, kFmtNvfp4>(const LayerArgs &, const LayerPlan &, int, cudaStream_t);
template cudaError_t launch_layer_t<16, 0, 1, 0, kFmtNvfp4>(const LayerArgs &, const LayerPlan &, int, cudaStream_t);

}  // namespace moe
