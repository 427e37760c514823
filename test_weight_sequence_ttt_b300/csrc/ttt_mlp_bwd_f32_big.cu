// ttt_mlp_bwd_f32_big.cu -- instantiations of the TTT-MLP backward kernels (ttt_mlp_bwd.cuh)
// for fp32 inputs, mini-batch sizes 8, 16 and the two-CTA cluster kernel.
#include "ttt_mlp_bwd.cuh"

namespace ttt {
namespace mlpb {

template cudaError_t launch_mb<float, 8>(const MlpBwdParams &, int, cudaStream_t);
template cudaError_t launch_mb<float, 16>(const MlpBwdParams &, int, cudaStream_t);
template cudaError_t launch_cluster<float>(const MlpBwdParams &, int, cudaStream_t);

}  // namespace mlpb
}  // namespace ttt
