// ttt_internal.h -- launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ttt.h"

namespace ttt {

// Chain-level parameters shared by the TTT-Linear kernels (device pointers).
struct LinearParams {
    int H, T, d, mb;
    float eps;
    const void *Q, *K, *V;
    const float *eta;
    const float *W0, *c0;
    long long w0_bstride, c0_bstride;
    const float *ln_g, *ln_b;
    void *Z;
    float *W_out, *c_out, *loss, *inner_loss;
    int *status;
};

struct MlpParams {
    int H, T, d, hidden, mb;
    float eps;
    const void *Q, *K, *V;
    const float *eta;
    const float *W1, *c1, *W2, *c2;
    long long w_bstride, c1_bstride, c2_bstride;
    const float *ln_g, *ln_b;
    void *Z;
    float *W1_out, *c1_out, *W2_out, *c2_out, *loss, *inner_loss;
    int *status;
};

// fp32 FFMA kernels (io f32 or bf16), any d <= 128, mb <= 64, mb*d <= 4096.
bool linear_f32_supported(int io, int d, int mb);
cudaError_t launch_linear_f32(const LinearParams &p, int io, int chains, cudaStream_t s);
bool mlp_f32_supported(int io, int d, int hidden, int mb);
cudaError_t launch_mlp_f32(const MlpParams &p, int io, int chains, cudaStream_t s);

// Tensor-core kernel (io bf16, d in {64,128}, mb in {1,2,4,8,16}).
bool linear_tc_supported(int io, int d, int mb);
// Returns cudaSuccess or the failing error; tensor maps are built inside.
cudaError_t launch_linear_tc(const LinearParams &p, int chains, cudaStream_t s);

}  // namespace ttt
