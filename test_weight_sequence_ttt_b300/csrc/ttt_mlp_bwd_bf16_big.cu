// ttt_mlp_bwd_bf16_big.cu -- instantiations of the TTT-MLP backward kernels (ttt_mlp_bwd.cuh)
// for bf16 inputs, mini-batch sizes 8, 16 and the two-CTA cluster kernel.
#include "ttt_mlp_bwd.cuh"

namespace ttt {
namespace mlpb {

template cudaError_t launch_mb<__nv_bfloat16, 8>(const MlpBwdParams &, int, cudaStream_t);
template cudaError_t launch_mb<__nv_bfloat16, 16>(const MlpBwdParams &, int, cudaStream_t);
template cudaError_t launch_cluster<__nv_bfloat16>(const MlpBwdParams &, int, cudaStream_t);

}  // namespace mlpb
}  // namespace ttt
