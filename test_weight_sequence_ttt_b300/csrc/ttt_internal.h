// ttt_internal.h -- launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ttt.h"

namespace ttt {

// Raise kernel Kern's dynamic shared-memory limit to `bytes` on the current
// device unless an earlier call already did (the attribute lasts for the
// process), so the per-call cost is one cudaGetDevice.
template <auto Kern>
cudaError_t ensure_smem(int bytes)
{
    static std::atomic<int> done[64];  // per device: the largest limit set so far
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) {
        int cur = done[dev].load(std::memory_order_relaxed);
        while (cur < bytes && !done[dev].compare_exchange_weak(cur, bytes, std::memory_order_acq_rel)) {
        }
    }
    return e;
}

// Chain-level parameters shared by the TTT-Linear kernels (device pointers).
struct LinearParams {
    int H, T, d, mb;
    int z_f32;   // Z element type: 1 = fp32, 0 = bf16
    int prefix;  // 1: z_t with the in-batch prefix W_t; 0: with the anchor W_{i-1}
    int q_is_k;  // 1: the queries are the keys (no query tile is loaded)
    int t_commit;  // tokens [0, t_commit) are committed; a partial last mini-batch after them is not
    int drop_step;  // fault-hook builds only: the loader skips this super-step (-1: none)
    int eta_gate;   // 1: eta holds gate logits, eta_t = eta_base * sigmoid(logit)
    float eta_base;
    float eps;
    const void *Q, *K, *V;
    const float *eta;
    const float *W0, *c0;
    long long w0_bstride, c0_bstride;
    const float *ln_g, *ln_b;
    void *Z;
    float *W_out, *c_out, *loss, *inner_loss;
    int *status;
    unsigned long long *trace;  // phase timestamps (TTT_TRACE builds only), else NULL
};

struct MlpParams {
    int H, T, d, hidden, mb;
    int z_f32;
    int prefix;  // as for LinearParams
    int q_is_k;
    int t_commit;
    int drop_step;
    int eta_gate;
    float eta_base;
    float eps;
    const void *Q, *K, *V;
    const float *eta;
    const float *W1, *c1, *W2, *c2;
    long long w_bstride, c1_bstride, c2_bstride;
    const float *ln_g, *ln_b;
    void *Z;
    float *W1_out, *c1_out, *W2_out, *c2_out, *loss, *inner_loss;
    int *status;
    unsigned long long *trace;  // phase timestamps (TTT_TRACE builds only), else NULL
};

// Gradients of the TTT-Linear inner loop (prefix rule, T a multiple of mb).
struct LinearBwdParams {
    int H, T, d, mb;
    int tf32;  // 1: contractions on the tensor cores with tf32 operands (d = 64, mb = 16)
    int eta_gate;
    float eta_base;
    float eps;
    const void *Q, *K, *V, *dZ;  // io element type
    const float *eta;
    const float *W0, *c0;
    long long w0_bstride, c0_bstride;
    const float *ln_g, *ln_b;
    const float *dW_n, *dc_n;  // seeds on the final state, or NULL
    float *dQ, *dK, *dV, *deta, *dW0, *dc0, *dln_g, *dln_b;
    float *ws;  // T/mb anchors (W, c) per chain
    int *status;
};

// Gradients of the TTT-MLP inner loop (prefix rule, T a multiple of mb).
struct MlpBwdParams {
    int H, T, d, hidden, mb;
    int eta_gate;
    float eta_base;
    float eps;
    const void *Q, *K, *V, *dZ;  // io element type
    const float *eta;
    const float *W1, *c1, *W2, *c2;
    long long w_bstride, c1_bstride, c2_bstride;
    const float *ln_g, *ln_b;
    const float *dW1_n, *dc1_n, *dW2_n, *dc2_n;  // seeds on the final state, or NULL
    float *dQ, *dK, *dV, *deta, *dW1, *dc1, *dW2, *dc2, *dln_g, *dln_b;
    float *ws;  // T/mb starting states (W1, c1, W2, c2) and dW1, dW2 per chain
    int *status;
};

// Phase-timestamp hook for performance diagnosis. Compiled in only with
// -DTTT_TRACE; records clock64() of CTA 0 at role phase boundaries for steps
// [kTraceFirst, kTraceFirst + kTraceSteps) into trace[(step - first) * 16 + slot].
constexpr int kTraceFirst = 16, kTraceSteps = 32, kTraceSlots = 16;
#ifdef TTT_TRACE
#define TTT_TRACE_AT(p, step, slot)                                                                   \
    do {                                                                                              \
        if ((p).trace && blockIdx.x == 0 && (threadIdx.x & 31) == 0 && (step) >= kTraceFirst &&       \
            (step) < kTraceFirst + kTraceSteps)                                                       \
            (p).trace[((step)-kTraceFirst) * kTraceSlots + (slot)] = clock64();                       \
    } while (0)
#else
#define TTT_TRACE_AT(p, step, slot) \
    do {                            \
    } while (0)
#endif

// fp32 FFMA kernels (io f32 or bf16), any d <= 128, mb <= 64, mb*d <= 4096.
bool linear_f32_supported(int io, int d, int mb);
cudaError_t launch_linear_f32(const LinearParams &p, int io, int chains, cudaStream_t s);
bool mlp_f32_supported(int io, int d, int hidden, int mb);
cudaError_t launch_mlp_f32(const MlpParams &p, int io, int chains, cudaStream_t s);

// Tensor-core TTT-MLP kernel (io bf16, d = 64, hidden = 256, mb = 16).
bool mlp_tc_supported(int io, int d, int hidden, int mb);
cudaError_t launch_mlp_tc(const MlpParams &p, int chains, cudaStream_t s);
// Chains on two-CTA clusters (hidden units split): 0 never, 1 when
// 2 * chains <= SMs (default), 2 always. A mode outside 0..2 only reads it.
int mlp_cluster_mode(int mode);

// fp32 FFMA backward kernel (io f32 or bf16), d <= 128, mb <= 64.
bool linear_bwd_supported(int io, int d, int mb);
size_t linear_bwd_workspace_bytes(int B, int H, int T, int d, int mb);
// Device address of the library's static backward scratch on the current device.
cudaError_t linear_bwd_noalloc_scratch(void **ptr);
cudaError_t launch_linear_bwd(const LinearBwdParams &p, int io, int chains, cudaStream_t s);

// fp32 FFMA TTT-MLP backward kernel (io f32 or bf16), mb in {1, 2, 4, 8, 16}.
bool mlp_bwd_supported(int io, int d, int hidden, int mb);
size_t mlp_bwd_workspace_bytes(int B, int H, int T, int d, int hidden, int mb);
cudaError_t launch_mlp_bwd(const MlpBwdParams &p, int io, int chains, cudaStream_t s);

// Tensor-core kernel (io bf16, d in {64,128}, mb a power of two up to 1024).
bool linear_tc_supported(int io, int d, int mb);
// Returns cudaSuccess or the failing error; tensor maps are built inside.
cudaError_t launch_linear_tc(const LinearParams &p, int chains, cudaStream_t s);
// When d = 64, b = 16 runs as one chain per two-CTA cluster: 0 never, 1 when
// 2 * chains <= SMs (default), 2 always. A mode outside 0..2 only reads it.
int linear_cluster_mode(int mode);

}  // namespace ttt
