// ttt_mlp_bwd.cu -- dispatch of the TTT-MLP backward kernels (ttt_mlp_bwd.cuh),
// whose instantiations live in ttt_mlp_bwd_{f32,bf16}_{small,big}.cu.
#include "ttt_mlp_bwd.cuh"

namespace ttt {
namespace mlpb {

extern template cudaError_t launch_mb<float, 1>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_mb<float, 2>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_mb<float, 4>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_mb<float, 8>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_mb<float, 16>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_cluster<float>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_mb<__nv_bfloat16, 1>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_mb<__nv_bfloat16, 2>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_mb<__nv_bfloat16, 4>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_mb<__nv_bfloat16, 8>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_mb<__nv_bfloat16, 16>(const MlpBwdParams &, int, cudaStream_t);
extern template cudaError_t launch_cluster<__nv_bfloat16>(const MlpBwdParams &, int, cudaStream_t);

template <typename IO>
cudaError_t launch_io(const MlpBwdParams &p, int chains, cudaStream_t s)
{
    if (cluster_ok(p.d, p.hidden, p.mb)) return launch_cluster<IO>(p, chains, s);
    switch (p.mb) {
    case 1: return launch_mb<IO, 1>(p, chains, s);
    case 2: return launch_mb<IO, 2>(p, chains, s);
    case 4: return launch_mb<IO, 4>(p, chains, s);
    case 8: return launch_mb<IO, 8>(p, chains, s);
    default: return launch_mb<IO, 16>(p, chains, s);
    }
}

}  // namespace mlpb


bool mlp_bwd_supported(int io, int d, int hidden, int mb)
{
    using namespace mlpb;
    const bool pow2 = mb == 1 || mb == 2 || mb == 4 || mb == 8 || mb == 16;
    return (io == TTT_F32 || io == TTT_BF16) && d >= 4 && d <= 32 * kMaxPer && d % 4 == 0 && hidden >= 4 &&
           hidden % 4 == 0 && pow2 && sizeof(float) * mlp_bwd_smem_floats(d, hidden, mb) <= 227 * 1024;
}

size_t mlp_bwd_workspace_bytes(int B, int H, int T, int d, int hidden, int mb)
{
    // per chain: every mini-batch's starting state, dW1 and dW2, every mini-batch's key side
    const size_t hd = (size_t)hidden * d, n = (size_t)(T / mb);
    return (size_t)B * H * (n * (2 * hd + hidden + d) + 2 * hd + n * mlpb::mlp_bwd_saved_floats(d, hidden, mb)) *
           sizeof(float);
}

cudaError_t launch_mlp_bwd(const MlpBwdParams &p, int io, int chains, cudaStream_t s)
{
    return io == TTT_F32 ? mlpb::launch_io<float>(p, chains, s) : mlpb::launch_io<__nv_bfloat16>(p, chains, s);
}

}  // namespace ttt
