// ttt_linear_f32.cu -- TTT-Linear inner loop in plain fp32 (FFMA), any d <= 128.
//
// One CTA per (sequence, head) chain; W (fp32, padded rows) and the current
// mini-batch live in shared memory. Each mini-batch follows the matrix form of
// the mini-batch rule (Eq. 5 of the "End-to-End Test-Time Training for Long
// Context" review, section 2.3) with the in-batch prefix output of Eq. 5 of the
// "TTT layer" section of the Test-Time Training survey page:
//   Y  = K W^T + c                       (f_res of every key at W_{i-1})
//   G  = d l_t / d y_t through x + LN(y) (Eq. 4 loss, residual LN form)
//   A  = causal (eta_s / b)(q_t.k_s + 1)
//   Yq = Q W^T + c - A G                 (= W_t q_t + c_t)
//   Z  = Q + LN(Yq),  W -= (1/b) G^T diag(eta) K,  c -= (1/b) G^T eta
// This kernel is the precise (fp32-operand) path; the bf16 tensor-core kernel
// is the fast path for d in {64, 128}.
#include <cuda_bf16.h>

#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename IO>
__device__ __forceinline__ float ld_io(const IO *p);
template <>
__device__ __forceinline__ float ld_io<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float ld_io<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

template <typename IO>
__device__ __forceinline__ void st_io(IO *p, float v);
template <>
__device__ __forceinline__ void st_io<float>(float *p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_io<__nv_bfloat16>(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void set_status(int *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

template <typename IO, typename ZT>
__global__ void __launch_bounds__(kThreads) linear_f32_kernel(LinearParams p)
{
    extern __shared__ float sm[];
    const int d = p.d, b = p.mb, T = p.T, dp = d + 1;
    float *W = sm;              // [d][dp]  W[j][i], row j = output feature
    float *c = W + d * dp;      // [d]
    float *Kt = c + d;          // [b][d]
    float *Qt = Kt + b * d;     // [b][d]
    float *G = Qt + b * d;      // [b][d]   d l_s / d y_s
    float *Yq = G + b * d;      // [b][d]   f_res(k) then f_res(q) pre-LN
    float *A = Yq + b * d;      // [b][b]
    float *et = A + b * b;      // [b]

    const int chain = blockIdx.x;
    const int bi = chain / p.H, hi = chain % p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *W0 = p.W0 + bi * p.w0_bstride + (long long)hi * d * d;
    const float *c0 = p.c0 + bi * p.c0_bstride + (long long)hi * d;
    const float *lg = p.ln_g + (long long)hi * d;
    const float *lb = p.ln_b + (long long)hi * d;
    const size_t tok0 = (size_t)chain * T;
    const IO *Qg = static_cast<const IO *>(p.Q) + tok0 * d;
    const IO *Kg = static_cast<const IO *>(p.K) + tok0 * d;
    const IO *Vg = static_cast<const IO *>(p.V) + tok0 * d;
    ZT *Zg = static_cast<ZT *>(p.Z) + tok0 * d;
    const float *eg = p.eta + tok0;
    const float inv_b = 1.0f / (float)b, inv_d = 1.0f / (float)d;

    for (int idx = tid; idx < d * d; idx += kThreads) W[(idx / d) * dp + idx % d] = W0[idx];
    for (int j = tid; j < d; j += kThreads) c[j] = c0[j];

    for (int t0 = 0; t0 < T; t0 += b) {
        // nb < b only for a partial last mini-batch: its rows past T are zero
        // (eta 0: no gradient), its outputs are stored, its update is not applied.
        const int nb = T - t0 < b ? T - t0 : b;
        __syncthreads();
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const size_t g = (size_t)t0 * d + idx;
            Kt[idx] = idx < nb * d ? ld_io<IO>(Kg + g) : 0.f;
            Qt[idx] = idx < nb * d ? ld_io<IO>(Qg + g) : 0.f;
        }
        for (int s = tid; s < b; s += kThreads) {
            const float e = s < nb ? eg[t0 + s] : 0.f;  // eta, or the gate logit
            et[s] = s >= nb ? 0.f : p.eta_gate ? p.eta_base / (1.f + __expf(-e)) : e;
        }
        __syncthreads();
        // Y = K W^T + c  (keys at the anchor W_{i-1})
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int s = idx / d, j = idx - s * d;
            const float *w = W + j * dp, *k = Kt + s * d;
            float acc = c[j];
            for (int i = 0; i < d; ++i) acc = fmaf(w[i], k[i], acc);
            Yq[idx] = acc;
        }
        __syncthreads();
        // LN forward/backward per key row: G = d||k + LN(y) - v||^2 / dy
        for (int s = warp; s < b; s += kWarps) {
            const float *y = Yq + s * d;
            float mu = 0.f;
            for (int j = lane; j < d; j += 32) mu += y[j];
            mu = warp_sum(mu) * inv_d;
            float var = 0.f;
            for (int j = lane; j < d; j += 32) var += (y[j] - mu) * (y[j] - mu);
            var = warp_sum(var) * inv_d;
            const float rstd = rsqrtf(var + p.eps);
            float l = 0.f, m1 = 0.f, m2 = 0.f;
            for (int j = lane; j < d; j += 32) {
                const float yh = (y[j] - mu) * rstd;
                const float e = Kt[s * d + j] + lg[j] * yh + lb[j] - (s < nb ? ld_io<IO>(Vg + (size_t)(t0 + s) * d + j) : 0.f);
                const float dh = 2.f * e * lg[j];
                l += e * e;
                m1 += dh;
                m2 += dh * yh;
            }
            l = warp_sum(l);
            m1 = warp_sum(m1) * inv_d;
            m2 = warp_sum(m2) * inv_d;
            for (int j = lane; j < d; j += 32) {
                const float yh = (y[j] - mu) * rstd;
                const float e = Kt[s * d + j] + lg[j] * yh + lb[j] - (s < nb ? ld_io<IO>(Vg + (size_t)(t0 + s) * d + j) : 0.f);
                const float dh = 2.f * e * lg[j];
                G[s * d + j] = rstd * (dh - m1 - yh * m2);
            }
            if (lane == 0 && p.inner_loss && s < nb) p.inner_loss[tok0 + t0 + s] = l;
        }
        // A[t][s] = (eta_s / b)(q_t . k_s + 1), s <= t
        for (int idx = tid; idx < b * b; idx += kThreads) {
            const int t = idx / b, s = idx - t * b;
            float v = 0.f;
            if (p.prefix && s <= t) {  // the anchor rule sees no update of the batch
                const float *q = Qt + t * d, *k = Kt + s * d;
                float acc = 1.f;
                for (int i = 0; i < d; ++i) acc = fmaf(q[i], k[i], acc);
                v = et[s] * inv_b * acc;
            }
            A[idx] = v;
        }
        __syncthreads();
        // Yq = Q W^T + c - A G
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int t = idx / d, j = idx - t * d;
            const float *w = W + j * dp, *q = Qt + t * d;
            float acc = c[j];
            for (int i = 0; i < d; ++i) acc = fmaf(w[i], q[i], acc);
            for (int s = 0; s <= t; ++s) acc = fmaf(-A[t * b + s], G[s * d + j], acc);
            Yq[idx] = acc;
        }
        __syncthreads();
        // Z = Q + LN(Yq), L_t = ||z_t - v_t||^2
        for (int t = warp; t < nb; t += kWarps) {
            const float *y = Yq + t * d;
            float mu = 0.f;
            for (int j = lane; j < d; j += 32) mu += y[j];
            mu = warp_sum(mu) * inv_d;
            float var = 0.f;
            for (int j = lane; j < d; j += 32) var += (y[j] - mu) * (y[j] - mu);
            var = warp_sum(var) * inv_d;
            const float rstd = rsqrtf(var + p.eps);
            float L = 0.f;
            for (int j = lane; j < d; j += 32) {
                const float z = Qt[t * d + j] + lg[j] * (y[j] - mu) * rstd + lb[j];
                st_io<ZT>(Zg + (size_t)(t0 + t) * d + j, z);
                const float v = ld_io<IO>(Vg + (size_t)(t0 + t) * d + j);
                L += (z - v) * (z - v);
            }
            L = warp_sum(L);
            if (lane == 0 && p.loss) p.loss[tok0 + t0 + t] = L;
        }
        // W -= (1/b) G^T diag(eta) K ; c -= (1/b) G^T eta   (W_{i-1} -> W_i)
        if (nb < b) continue;  // the partial last mini-batch is not committed
        for (int idx = tid; idx < d * d; idx += kThreads) {
            const int j = idx / d, i = idx - j * d;
            float acc = 0.f;
            for (int s = 0; s < b; ++s) acc = fmaf(et[s] * G[s * d + j], Kt[s * d + i], acc);
            W[j * dp + i] -= acc * inv_b;
        }
        for (int j = tid; j < d; j += kThreads) {
            float acc = 0.f;
            for (int s = 0; s < b; ++s) acc = fmaf(et[s], G[s * d + j], acc);
            c[j] -= acc * inv_b;
        }
    }
    __syncthreads();
    bool bad = false;
    for (int idx = tid; idx < d * d; idx += kThreads) {
        const float w = W[(idx / d) * dp + idx % d];
        bad |= !isfinite(w);
        if (p.W_out) p.W_out[(size_t)chain * d * d + idx] = w;
    }
    for (int j = tid; j < d; j += kThreads) {
        bad |= !isfinite(c[j]);
        if (p.c_out) p.c_out[(size_t)chain * d + j] = c[j];
    }
    if (bad) set_status(p.status, TTT_ERR_NONFINITE);
}

size_t linear_f32_smem(int d, int b)
{
    return sizeof(float) * ((size_t)d * (d + 1) + d + 4 * (size_t)b * d + (size_t)b * b + b);
}

}  // namespace

bool linear_f32_supported(int io, int d, int mb)
{
    return (io == TTT_F32 || io == TTT_BF16) && d >= 1 && d <= 128 && mb >= 1 && mb <= 64 &&
           linear_f32_smem(d, mb) <= 227 * 1024;
}

template <typename IO, typename ZT>
cudaError_t launch_linear_f32_t(const LinearParams &p, int chains, cudaStream_t s)
{
    const size_t smem = linear_f32_smem(p.d, p.mb);
    cudaError_t e = ensure_smem<linear_f32_kernel<IO, ZT>>((int)smem);
    if (e != cudaSuccess) return e;
    linear_f32_kernel<IO, ZT><<<chains, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_linear_f32(const LinearParams &p, int io, int chains, cudaStream_t s)
{
    if (io == TTT_F32)
        return p.z_f32 ? launch_linear_f32_t<float, float>(p, chains, s) : launch_linear_f32_t<float, __nv_bfloat16>(p, chains, s);
    return p.z_f32 ? launch_linear_f32_t<__nv_bfloat16, float>(p, chains, s)
                   : launch_linear_f32_t<__nv_bfloat16, __nv_bfloat16>(p, chains, s);
}

}  // namespace ttt
