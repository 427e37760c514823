// ttt_mlp_bwd_bf16_small.cu -- instantiations of the TTT-MLP backward kernels (ttt_mlp_bwd.cuh)
// for bf16 inputs, mini-batch sizes 1, 2, 4.
#include "ttt_mlp_bwd.cuh"

namespace ttt {
namespace mlpb {

template cudaError_t launch_mb<__nv_bfloat16, 1>(const MlpBwdParams &, int, cudaStream_t);
template cudaError_t launch_mb<__nv_bfloat16, 2>(const MlpBwdParams &, int, cudaStream_t);
template cudaError_t launch_mb<__nv_bfloat16, 4>(const MlpBwdParams &, int, cudaStream_t);

}  // namespace mlpb
}  // namespace ttt
