// decode_layer_gen4.cu -- instantiations of the one-launch decode layer kernel
// (decode_layer.cuh), compiled apart from the others to keep builds parallel.
#include "decode_layer.cuh"

namespace moe {

template cudaError_t launch_layer_t<4, 0, 4, 0, kFmtW4A16>(const LayerArgs &, const LayerPlan &, int, cudaStream_t);
template cudaError_t launch_layer_t<4, 0, 1, 0, kFmtW4A16>(const LayerArgs &, const LayerPlan &, int, cudaStream_t);

}  // namespace moe
