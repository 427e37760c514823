// ttt_mlp_f32.cu -- TTT-MLP inner loop in plain fp32 (FFMA).
//
// f_res(x) = W2 gelu_tanh(W1 x + c1) + c2, f(x) = x + LN(f_res(x)): the
// TTT-MLP of the "TTT layer" section of the "Test-Time Training(TTT)과 LLM
// 메모리" survey page (2-layer MLP, hidden 4x, GELU, LN + residual), trained
// by the mini-batch rule of Eq. 5 of the "End-to-End Test-Time Training for
// Long Context" review (section 2.3). Per mini-batch, matrix form:
//   Z1 = K W1^T + c1, X2 = gelu(Z1), Y = X2 W2^T + c2       (anchor weights)
//   G  = d l / d Y (through x + LN),  G1 = (G W2) * gelu'(Z1)
//   Z1q = Q W1^T + c1 - A1 G1,  A1 = causal (eta_s/b)(q_t.k_s + 1)
//   Yq  = gelu(Z1q) W2^T + c2 - A2 G,  A2 = causal (eta_s/b)(x2q_t.x2k_s + 1)
//   Z = Q + LN(Yq); W2 -= (1/b) G^T diag(eta) X2, W1 -= (1/b) G1^T diag(eta) K.
// One CTA per chain; both weight matrices live in shared memory.
#include <cuda_bf16.h>

#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr float kGeluA = 0.7978845608028654f;  // sqrt(2/pi)
constexpr float kGeluC = 0.044715f;

__device__ __forceinline__ float gelu(float u)
{
    return 0.5f * u * (1.f + tanhf(kGeluA * (u + kGeluC * u * u * u)));
}

__device__ __forceinline__ float gelu_prime(float u)
{
    const float th = tanhf(kGeluA * (u + kGeluC * u * u * u));
    return 0.5f * (1.f + th) + 0.5f * u * (1.f - th * th) * kGeluA * (1.f + 3.f * kGeluC * u * u);
}

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

size_t mlp_f32_floats(int d, int h, int b)
{
    return 2 * (size_t)h * d + h + d + 5 * (size_t)b * d + 3 * (size_t)b * h + (size_t)b * b + b;
}

// LayerNorm over one row of length d held in shared memory, one warp per row.
// Returns mean and rstd.
__device__ __forceinline__ void row_stats(const float *y, int d, float eps, int lane, float &mu, float &rstd)
{
    float s = 0.f;
    for (int j = lane; j < d; j += 32) s += y[j];
    mu = warp_sum(s) / (float)d;
    float v = 0.f;
    for (int j = lane; j < d; j += 32) v += (y[j] - mu) * (y[j] - mu);
    rstd = rsqrtf(warp_sum(v) / (float)d + eps);
}

template <typename IO, typename ZT>
__global__ void __launch_bounds__(kThreads) mlp_f32_kernel(MlpParams p)
{
    extern __shared__ float sm[];
    const int d = p.d, h = p.hidden, b = p.mb, T = p.T;
    float *W1 = sm;               // [h][d]
    float *W2 = W1 + h * d;       // [d][h]
    float *c1 = W2 + d * h;       // [h]
    float *c2 = c1 + h;           // [d]
    float *Kt = c2 + d;           // [b][d]
    float *Qt = Kt + b * d;
    float *Vt = Qt + b * d;
    float *G = Vt + b * d;        // [b][d]
    float *Yq = G + b * d;        // [b][d]
    float *Hk = Yq + b * d;       // [b][h]  Z1 of keys, then G1
    float *X2 = Hk + b * h;       // [b][h]  gelu(Z1) of keys
    float *Hq = X2 + b * h;       // [b][h]  Z1 of queries, then gelu
    float *A = Hq + b * h;        // [b][b]
    float *et = A + b * b;        // [b]

    const int chain = blockIdx.x, bi = chain / p.H, hi = chain % p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *W10 = p.W1 + bi * p.w_bstride + (long long)hi * h * d;
    const float *W20 = p.W2 + bi * p.w_bstride + (long long)hi * h * d;
    const float *c10 = p.c1 + bi * p.c1_bstride + (long long)hi * h;
    const float *c20 = p.c2 + bi * p.c2_bstride + (long long)hi * d;
    const float *lg = p.ln_g + (long long)hi * d, *lb = p.ln_b + (long long)hi * d;
    const size_t tok0 = (size_t)chain * T;
    const IO *Qg = static_cast<const IO *>(p.Q) + tok0 * d;
    const IO *Kg = static_cast<const IO *>(p.K) + tok0 * d;
    const IO *Vg = static_cast<const IO *>(p.V) + tok0 * d;
    ZT *Zg = static_cast<ZT *>(p.Z) + tok0 * d;
    const float *eg = p.eta + tok0;
    const float inv_b = 1.f / (float)b, inv_d = 1.f / (float)d;

    for (int i = tid; i < h * d; i += kThreads) {
        W1[i] = W10[i];
        W2[i] = W20[i];
    }
    for (int i = tid; i < h; i += kThreads) c1[i] = c10[i];
    for (int i = tid; i < d; i += kThreads) c2[i] = c20[i];

    for (int t0 = 0; t0 < T; t0 += b) {
        // nb < b only for a partial last mini-batch (rows past T zero, eta 0;
        // outputs stored, update not applied).
        const int nb = T - t0 < b ? T - t0 : b;
        __syncthreads();
        for (int i = tid; i < b * d; i += kThreads) {
            const size_t gi = (size_t)t0 * d + i;
            const bool in = i < nb * d;
            Kt[i] = in ? ld_io<IO>(Kg + gi) : 0.f;
            Qt[i] = in ? ld_io<IO>(Qg + gi) : 0.f;
            Vt[i] = in ? ld_io<IO>(Vg + gi) : 0.f;
        }
        for (int s = tid; s < b; s += kThreads) {
            const float e = s < nb ? eg[t0 + s] : 0.f;  // eta, or the gate logit
            et[s] = s >= nb ? 0.f : p.eta_gate ? p.eta_base / (1.f + __expf(-e)) : e;
        }
        __syncthreads();
        // Z1 = K W1^T + c1 ; X2 = gelu(Z1)
        for (int i = tid; i < b * h; i += kThreads) {
            const int s = i / h, j = i - s * h;
            const float *w = W1 + j * d, *k = Kt + s * d;
            float acc = c1[j];
            for (int u = 0; u < d; ++u) acc = fmaf(w[u], k[u], acc);
            Hk[i] = acc;
            X2[i] = gelu(acc);
        }
        __syncthreads();
        // Y = X2 W2^T + c2 (into Yq)
        for (int i = tid; i < b * d; i += kThreads) {
            const int s = i / d, r = i - s * d;
            const float *w = W2 + r * h, *x = X2 + s * h;
            float acc = c2[r];
            for (int u = 0; u < h; ++u) acc = fmaf(w[u], x[u], acc);
            Yq[i] = acc;
        }
        __syncthreads();
        // G = d||k + LN(y) - v||^2 / dy
        for (int s = warp; s < b; s += kWarps) {
            const float *y = Yq + s * d;
            float mu, rstd;
            row_stats(y, d, p.eps, lane, mu, rstd);
            float l = 0.f, m1 = 0.f, m2 = 0.f;
            for (int j = lane; j < d; j += 32) {
                const float yh = (y[j] - mu) * rstd;
                const float e = Kt[s * d + j] + lg[j] * yh + lb[j] - Vt[s * d + j];
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
                const float e = Kt[s * d + j] + lg[j] * yh + lb[j] - Vt[s * d + j];
                G[s * d + j] = rstd * (2.f * e * lg[j] - m1 - yh * m2);
            }
            if (lane == 0 && p.inner_loss && s < nb) p.inner_loss[tok0 + t0 + s] = l;
        }
        // A1 = causal (eta_s/b)(q_t.k_s + 1)
        for (int i = tid; i < b * b; i += kThreads) {
            const int t = i / b, s = i - t * b;
            float v = 0.f;
            if (p.prefix && s <= t) {  // the anchor rule sees no update of the batch
                float acc = 1.f;
                for (int u = 0; u < d; ++u) acc = fmaf(Qt[t * d + u], Kt[s * d + u], acc);
                v = et[s] * inv_b * acc;
            }
            A[i] = v;
        }
        __syncthreads();
        // G1 = (G W2) * gelu'(Z1)   (in place of Z1)
        for (int i = tid; i < b * h; i += kThreads) {
            const int s = i / h, j = i - s * h;
            float acc = 0.f;
            for (int r = 0; r < d; ++r) acc = fmaf(G[s * d + r], W2[r * h + j], acc);
            Hk[i] = acc * gelu_prime(Hk[i]);
        }
        __syncthreads();
        // Z1q = Q W1^T + c1 - A1 G1 ; X2q = gelu(Z1q)
        for (int i = tid; i < b * h; i += kThreads) {
            const int t = i / h, j = i - t * h;
            const float *w = W1 + j * d, *q = Qt + t * d;
            float acc = c1[j];
            for (int u = 0; u < d; ++u) acc = fmaf(w[u], q[u], acc);
            for (int s = 0; s <= t; ++s) acc = fmaf(-A[t * b + s], Hk[s * h + j], acc);
            Hq[i] = gelu(acc);
        }
        __syncthreads();
        // A2 = causal (eta_s/b)(x2q_t . x2k_s + 1)
        for (int i = tid; i < b * b; i += kThreads) {
            const int t = i / b, s = i - t * b;
            float v = 0.f;
            if (p.prefix && s <= t) {  // the anchor rule sees no update of the batch
                float acc = 1.f;
                for (int u = 0; u < h; ++u) acc = fmaf(Hq[t * h + u], X2[s * h + u], acc);
                v = et[s] * inv_b * acc;
            }
            A[i] = v;
        }
        __syncthreads();
        // Yq = X2q W2^T + c2 - A2 G
        for (int i = tid; i < b * d; i += kThreads) {
            const int t = i / d, r = i - t * d;
            const float *w = W2 + r * h, *x = Hq + t * h;
            float acc = c2[r];
            for (int u = 0; u < h; ++u) acc = fmaf(w[u], x[u], acc);
            for (int s = 0; s <= t; ++s) acc = fmaf(-A[t * b + s], G[s * d + r], acc);
            Yq[i] = acc;
        }
        __syncthreads();
        // Z = Q + LN(Yq), loss (rows of the batch that exist)
        for (int t = warp; t < nb; t += kWarps) {
            const float *y = Yq + t * d;
            float mu, rstd;
            row_stats(y, d, p.eps, lane, mu, rstd);
            float L = 0.f;
            for (int j = lane; j < d; j += 32) {
                const float z = Qt[t * d + j] + lg[j] * (y[j] - mu) * rstd + lb[j];
                st_io<ZT>(Zg + (size_t)(t0 + t) * d + j, z);
                L += (z - Vt[t * d + j]) * (z - Vt[t * d + j]);
            }
            L = warp_sum(L);
            if (lane == 0 && p.loss) p.loss[tok0 + t0 + t] = L;
        }
        // W2 -= (1/b) G^T diag(eta) X2 ; c2 -= (1/b) G^T eta
        if (nb < b) continue;  // the partial last mini-batch is not committed
        for (int i = tid; i < d * h; i += kThreads) {
            const int r = i / h, j = i - r * h;
            float acc = 0.f;
            for (int s = 0; s < b; ++s) acc = fmaf(et[s] * G[s * d + r], X2[s * h + j], acc);
            W2[i] -= acc * inv_b;
        }
        // W1 -= (1/b) G1^T diag(eta) K ; c1 -= (1/b) G1^T eta
        for (int i = tid; i < h * d; i += kThreads) {
            const int j = i / d, u = i - j * d;
            float acc = 0.f;
            for (int s = 0; s < b; ++s) acc = fmaf(et[s] * Hk[s * h + j], Kt[s * d + u], acc);
            W1[i] -= acc * inv_b;
        }
        for (int j = tid; j < h; j += kThreads) {
            float acc = 0.f;
            for (int s = 0; s < b; ++s) acc = fmaf(et[s], Hk[s * h + j], acc);
            c1[j] -= acc * inv_b;
        }
        for (int r = tid; r < d; r += kThreads) {
            float acc = 0.f;
            for (int s = 0; s < b; ++s) acc = fmaf(et[s], G[s * d + r], acc);
            c2[r] -= acc * inv_b;
        }
    }
    __syncthreads();
    bool bad = false;
    for (int i = tid; i < h * d; i += kThreads) {
        bad |= !isfinite(W1[i]) || !isfinite(W2[i]);
        if (p.W1_out) p.W1_out[(size_t)chain * h * d + i] = W1[i];
        if (p.W2_out) p.W2_out[(size_t)chain * h * d + i] = W2[i];
    }
    for (int j = tid; j < h; j += kThreads) {
        bad |= !isfinite(c1[j]);
        if (p.c1_out) p.c1_out[(size_t)chain * h + j] = c1[j];
    }
    for (int r = tid; r < d; r += kThreads) {
        bad |= !isfinite(c2[r]);
        if (p.c2_out) p.c2_out[(size_t)chain * d + r] = c2[r];
    }
    if (bad && p.status) atomicCAS(p.status, 0, TTT_ERR_NONFINITE);
}

constexpr size_t kMaxSmem = 227 * 1024;

}  // namespace

bool mlp_f32_supported(int io, int d, int hidden, int mb)
{
    return (io == TTT_F32 || io == TTT_BF16) && d >= 1 && d <= 256 && hidden >= 1 && hidden <= 1024 &&
           mb >= 1 && mb <= 64 && mlp_f32_floats(d, hidden, mb) * sizeof(float) <= kMaxSmem;
}

template <typename IO, typename ZT>
cudaError_t launch_mlp_f32_t(const MlpParams &p, int chains, cudaStream_t s)
{
    const size_t smem = mlp_f32_floats(p.d, p.hidden, p.mb) * sizeof(float);
    cudaError_t e = ensure_smem<mlp_f32_kernel<IO, ZT>>((int)smem);
    if (e != cudaSuccess) return e;
    mlp_f32_kernel<IO, ZT><<<chains, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_mlp_f32(const MlpParams &p, int io, int chains, cudaStream_t s)
{
    if (io == TTT_F32)
        return p.z_f32 ? launch_mlp_f32_t<float, float>(p, chains, s) : launch_mlp_f32_t<float, __nv_bfloat16>(p, chains, s);
    return p.z_f32 ? launch_mlp_f32_t<__nv_bfloat16, float>(p, chains, s)
                   : launch_mlp_f32_t<__nv_bfloat16, __nv_bfloat16>(p, chains, s);
}

}  // namespace ttt
