// ttt_linear_bwd.cu -- gradients of the TTT-Linear inner loop for outer-loop
// training: reverse mode through the mini-batch rule, fp32 (FFMA), d <= 128.
//
// Forward of mini-batch i, anchor (W, c) = (W_{i-1}, c_{i-1}), rows k_s, q_t,
// v_s, learning rates eta_s (the prefix-rule matrix form of Eq. 5 of the
// "End-to-End Test-Time Training for Long Context" review, section 2.3, with
// the output of Eq. 5 of the survey's "TTT layer" section):
//   y_s  = W k_s + c,   yh_s = (y_s - mean) r_s,  r_s = 1/sqrt(var + eps)
//   e_s  = k_s + gamma*yh_s + beta - v_s,  u_s = 2 gamma*e_s
//   g_s  = r_s (u_s - mean(u_s) - yh_s mean(u_s*yh_s))        (= d l_s / d y_s)
//   A_ts = (eta_s/b)(q_t.k_s + 1), s <= t
//   p_t  = W q_t + c - sum_{s<=t} A_ts g_s,   z_t = q_t + gamma*ph_t + beta
//   W'   = W - (1/b) sum_s eta_s g_s k_s^T,   c' = c - (1/b) sum_s eta_s g_s
// The update contains the inner gradient g, so the reverse pass differentiates
// the LayerNorm backward once more (the gradients of gradients of the review's
// section 2.2). With dz_t = dJ/dz_t and the carried (dW', dc') of the state
// after the batch, the kernel forms, per batch and in this order:
//   dp_t  = r^p_t (gamma*dz_t - mean(.) - ph_t mean(gamma*dz_t*ph_t))
//   DA_ts = -dp_t.g_s (s <= t),            R_s = dW' k_s + dc'
//   dg_s  = -sum_{t>=s} A_ts dp_t - (eta_s/b) R_s
//   deta_s = (1/b) (sum_{t>=s} DA_ts (q_t.k_s + 1) - g_s.R_s)
//   dq_t  = dz_t + W^T dp_t + sum_{s<=t} DA_ts (eta_s/b) k_s
//   g_s = r_s P_s u_s with P_s = I - 11^T/d - yh_s yh_s^T/d (symmetric), so
//   du_s  = r_s P_s dg_s,  de_s = 2 gamma*du_s,  dv_s = -de_s
//   dyh_s = gamma*de_s - r_s (dg_s mean(u_s*yh_s) + mean(dg_s*yh_s) u_s)
//   dsigma_s = -r_s dg_s.g_s
//   dy_s  = r_s (dyh_s - mean(dyh_s) - yh_s mean(dyh_s*yh_s)) + dsigma_s yh_s/d
//   dk_s  = W^T dy_s + de_s + sum_{t>=s} DA_ts (eta_s/b) q_t - (eta_s/b) dW'^T g_s
//   dW    = dW' + sum_t dp_t q_t^T + sum_s dy_s k_s^T,  dc = dc' + sum_t dp_t + sum_s dy_s
//   dgamma += sum_t dz_t*ph_t + sum_s 2 du_s*(gamma*yh_s + e_s),
//   dbeta  += sum_t dz_t + sum_s de_s.
//
// One CTA per (sequence, head) chain. A forward sweep stores every anchor
// (W_{i-1}, c_{i-1}) in the caller's workspace (checkpointing every mini-batch:
// n (d^2 + d) floats per chain); the reverse sweep reloads them from the last
// batch to the first and recomputes the batch's forward from its anchor. The
// tiled kernel also keeps each mini-batch's key side (yh, e, g and the two row
// statistics, after the checkpoints) and the reverse sweep reads it back instead
// of recomputing y_s and the key LayerNorm.
#include <cuda_bf16.h>
#include <type_traits>


#include "ttt_internal.h"

// Scratch of ttt_linear_backward_noalloc: the library's own device memory for the
// per-mini-batch checkpoints, for callers that cannot allocate a workspace.
// TTT_NOALLOC_SCRATCH_BYTES per GPU that loads the library, held until exit;
// every call of that entry point on a GPU shares it.
static __device__ __align__(256) float g_noalloc_scratch[TTT_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace ttt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxPer = 4;  // row elements per lane (d <= 128)

template <typename IO>
__device__ __forceinline__ float ldx(const IO *p);
template <>
__device__ __forceinline__ float ldx<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float ldx<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__device__ __forceinline__ float wsum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

struct Smem {
    float *W, *dW;                                  // [d][d + 1]
    float *c, *dc, *gam, *bet, *dgam, *dbet;        // [d]
    float *K, *Q, *E, *DZ, *Yh, *P, *G, *DP, *R, *KA, *DU;  // [b][d]
    float *QK, *DA;                                 // [b][b]
    float *et, *det, *rk, *m2k;                     // [b]
};

__host__ __device__ inline size_t bwd_smem_floats(int d, int b)
{
    return 2 * (size_t)d * (d + 1) + 6 * (size_t)d + 11 * (size_t)b * d + 2 * (size_t)b * b + 4 * (size_t)b;
}

__device__ Smem carve(float *sm, int d, int b)
{
    Smem s;
    const int dp = d + 1, bd = b * d;
    s.W = sm;
    s.dW = s.W + d * dp;
    s.c = s.dW + d * dp;
    s.dc = s.c + d;
    s.gam = s.dc + d;
    s.bet = s.gam + d;
    s.dgam = s.bet + d;
    s.dbet = s.dgam + d;
    s.K = s.dbet + d;
    s.Q = s.K + bd;
    s.E = s.Q + bd;
    s.DZ = s.E + bd;
    s.Yh = s.DZ + bd;
    s.P = s.Yh + bd;
    s.G = s.P + bd;
    s.DP = s.G + bd;
    s.R = s.DP + bd;
    s.KA = s.R + bd;
    s.DU = s.KA + bd;
    s.QK = s.DU + bd;
    s.DA = s.QK + b * b;
    s.et = s.DA + b * b;
    s.det = s.et + b;
    s.rk = s.det + b;
    s.m2k = s.rk + b;
    return s;
}

// Row s of Yh holds y_s on entry; leaves yh_s in Yh, e_s in E (which holds v_s
// on entry), g_s in G, and r_s, mean(u_s*yh_s) in rk, m2k. One warp per row.
__device__ __forceinline__ void key_rows(const Smem &S, int d, int b, float eps, int warp, int lane)
{
    const float inv_d = 1.f / (float)d;
    for (int s = warp; s < b; s += kWarps) {
        float *y = S.Yh + s * d, *e = S.E + s * d;
        const float *k = S.K + s * d;
        float mu = 0.f;
        for (int j = lane; j < d; j += 32) mu += y[j];
        mu = wsum(mu) * inv_d;
        float var = 0.f;
        for (int j = lane; j < d; j += 32) var += (y[j] - mu) * (y[j] - mu);
        const float r = rsqrtf(wsum(var) * inv_d + eps);
        float m1 = 0.f, m2 = 0.f;
        for (int j = lane; j < d; j += 32) {
            const float yh = (y[j] - mu) * r;
            const float ee = k[j] + S.gam[j] * yh + S.bet[j] - e[j];
            const float u = 2.f * S.gam[j] * ee;
            y[j] = yh;
            e[j] = ee;
            m1 += u;
            m2 += u * yh;
        }
        m1 = wsum(m1) * inv_d;
        m2 = wsum(m2) * inv_d;
        for (int j = lane; j < d; j += 32) S.G[s * d + j] = r * (2.f * S.gam[j] * e[j] - m1 - y[j] * m2);
        if (lane == 0) {
            S.rk[s] = r;
            S.m2k[s] = m2;
        }
    }
}

template <typename IO>
__global__ void __launch_bounds__(kThreads) linear_bwd_kernel(LinearBwdParams p)
{
    extern __shared__ float sm[];
    const int d = p.d, b = p.mb, T = p.T, dp = d + 1, n = T / b;
    const Smem S = carve(sm, d, b);
    const int chain = blockIdx.x;
    const int bi = chain / p.H, hi = chain % p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t tok0 = (size_t)chain * T;
    const IO *Qg = static_cast<const IO *>(p.Q) + tok0 * d;
    const IO *Kg = static_cast<const IO *>(p.K) + tok0 * d;
    const IO *Vg = static_cast<const IO *>(p.V) + tok0 * d;
    const IO *DZg = static_cast<const IO *>(p.dZ) + tok0 * d;
    const float *eg = p.eta + tok0;
    float *ws = p.ws + (size_t)chain * n * ((size_t)d * d + d);
    const float inv_b = 1.f / (float)b, inv_d = 1.f / (float)d;

    {
        const float *W0 = p.W0 + bi * p.w0_bstride + (long long)hi * d * d;
        const float *c0 = p.c0 + bi * p.c0_bstride + (long long)hi * d;
        for (int idx = tid; idx < d * d; idx += kThreads) {
            S.W[(idx / d) * dp + idx % d] = W0[idx];
            S.dW[(idx / d) * dp + idx % d] = p.dW_n ? p.dW_n[(size_t)chain * d * d + idx] : 0.f;
        }
        for (int j = tid; j < d; j += kThreads) {
            S.c[j] = c0[j];
            S.dc[j] = p.dc_n ? p.dc_n[(size_t)chain * d + j] : 0.f;
            S.gam[j] = p.ln_g[hi * d + j];
            S.bet[j] = p.ln_b[hi * d + j];
            S.dgam[j] = 0.f;
            S.dbet[j] = 0.f;
        }
    }
    auto load_eta = [&](int t0) {
        for (int s = tid; s < b; s += kThreads) {
            const float e = eg[t0 + s];
            S.et[s] = p.eta_gate ? p.eta_base / (1.f + __expf(-e)) : e;
        }
    };

    // ---- forward sweep: anchors into the workspace, W_{i-1} -> W_i
    for (int i = 0; i < n; ++i) {
        const int t0 = i * b;
        __syncthreads();
        float *wsi = ws + (size_t)i * ((size_t)d * d + d);
        for (int idx = tid; idx < d * d; idx += kThreads) wsi[idx] = S.W[(idx / d) * dp + idx % d];
        for (int j = tid; j < d; j += kThreads) wsi[d * d + j] = S.c[j];
        for (int idx = tid; idx < b * d; idx += kThreads) {
            S.K[idx] = ldx<IO>(Kg + (size_t)t0 * d + idx);
            S.E[idx] = ldx<IO>(Vg + (size_t)t0 * d + idx);
        }
        load_eta(t0);
        __syncthreads();
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int s = idx / d, j = idx - s * d;
            const float *w = S.W + j * dp, *k = S.K + s * d;
            float acc = S.c[j];
            for (int ii = 0; ii < d; ++ii) acc = fmaf(w[ii], k[ii], acc);
            S.Yh[idx] = acc;
        }
        __syncthreads();
        key_rows(S, d, b, p.eps, warp, lane);
        __syncthreads();
        for (int idx = tid; idx < d * d; idx += kThreads) {
            const int j = idx / d, ii = idx - j * d;
            float acc = 0.f;
            for (int s = 0; s < b; ++s) acc = fmaf(S.et[s] * S.G[s * d + j], S.K[s * d + ii], acc);
            S.W[j * dp + ii] -= acc * inv_b;
        }
        for (int j = tid; j < d; j += kThreads) {
            float acc = 0.f;
            for (int s = 0; s < b; ++s) acc = fmaf(S.et[s], S.G[s * d + j], acc);
            S.c[j] -= acc * inv_b;
        }
    }

    // ---- reverse sweep
    for (int i = n - 1; i >= 0; --i) {
        const int t0 = i * b;
        __syncthreads();
        const float *wsi = ws + (size_t)i * ((size_t)d * d + d);
        for (int idx = tid; idx < d * d; idx += kThreads) S.W[(idx / d) * dp + idx % d] = wsi[idx];
        for (int j = tid; j < d; j += kThreads) S.c[j] = wsi[d * d + j];
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const size_t g = (size_t)t0 * d + idx;
            S.K[idx] = ldx<IO>(Kg + g);
            S.Q[idx] = ldx<IO>(Qg + g);
            S.E[idx] = ldx<IO>(Vg + g);
            S.DZ[idx] = ldx<IO>(DZg + g);
        }
        load_eta(t0);
        __syncthreads();
        // y_s = W k_s + c, W q_t + c, q_t.k_s + 1
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int s = idx / d, j = idx - s * d;
            const float *w = S.W + j * dp, *k = S.K + s * d, *q = S.Q + s * d;
            float ak = S.c[j], aq = S.c[j];
            for (int ii = 0; ii < d; ++ii) {
                ak = fmaf(w[ii], k[ii], ak);
                aq = fmaf(w[ii], q[ii], aq);
            }
            S.Yh[idx] = ak;
            S.P[idx] = aq;
        }
        for (int idx = tid; idx < b * b; idx += kThreads) {
            const int t = idx / b, s = idx - t * b;
            const float *q = S.Q + t * d, *k = S.K + s * d;
            float acc = 1.f;
            for (int ii = 0; ii < d; ++ii) acc = fmaf(q[ii], k[ii], acc);
            S.QK[idx] = acc;
        }
        __syncthreads();
        key_rows(S, d, b, p.eps, warp, lane);
        __syncthreads();
        // p_t = W q_t + c - sum_{s<=t} A_ts g_s
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int t = idx / d, j = idx - t * d;
            float acc = S.P[idx];
            for (int s = 0; s <= t; ++s) acc = fmaf(-S.et[s] * inv_b * S.QK[t * b + s], S.G[s * d + j], acc);
            S.P[idx] = acc;
        }
        __syncthreads();
        // output LayerNorm: ph_t into P, dp_t into DP
        for (int t = warp; t < b; t += kWarps) {
            float *y = S.P + t * d;
            const float *dz = S.DZ + t * d;
            float mu = 0.f;
            for (int j = lane; j < d; j += 32) mu += y[j];
            mu = wsum(mu) * inv_d;
            float var = 0.f;
            for (int j = lane; j < d; j += 32) var += (y[j] - mu) * (y[j] - mu);
            const float r = rsqrtf(wsum(var) * inv_d + p.eps);
            float a1 = 0.f, a2 = 0.f;
            for (int j = lane; j < d; j += 32) {
                const float ph = (y[j] - mu) * r, dh = S.gam[j] * dz[j];
                y[j] = ph;
                a1 += dh;
                a2 += dh * ph;
            }
            a1 = wsum(a1) * inv_d;
            a2 = wsum(a2) * inv_d;
            for (int j = lane; j < d; j += 32) S.DP[t * d + j] = r * (S.gam[j] * dz[j] - a1 - y[j] * a2);
        }
        __syncthreads();
        for (int j = tid; j < d; j += kThreads) {
            float ag = 0.f, ab = 0.f;
            for (int t = 0; t < b; ++t) {
                ag = fmaf(S.DZ[t * d + j], S.P[t * d + j], ag);
                ab += S.DZ[t * d + j];
            }
            S.dgam[j] += ag;
            S.dbet[j] += ab;
        }
        for (int idx = tid; idx < b * b; idx += kThreads) {
            const int t = idx / b, s = idx - t * b;
            float acc = 0.f;
            if (s <= t) {
                const float *x = S.DP + t * d, *g = S.G + s * d;
                for (int j = 0; j < d; ++j) acc = fmaf(x[j], g[j], acc);
            }
            S.DA[idx] = -acc;
        }
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int s = idx / d, j = idx - s * d;
            const float *w = S.dW + j * dp, *k = S.K + s * d;
            float acc = S.dc[j];
            for (int ii = 0; ii < d; ++ii) acc = fmaf(w[ii], k[ii], acc);
            S.R[idx] = acc;  // dW' k_s + dc'
        }
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int s = idx / d, ii = idx - s * d;
            const float *g = S.G + s * d;
            float acc = 0.f;
            for (int j = 0; j < d; ++j) acc = fmaf(S.dW[j * dp + ii], g[j], acc);
            S.KA[idx] = -S.et[s] * inv_b * acc;  // -(eta_s/b) dW'^T g_s
        }
        __syncthreads();
        // dq_t; the q-side of dk_s; dg_s (into P, whose ph is no longer needed); deta_s
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int t = idx / d, ii = idx - t * d;
            const float *x = S.DP + t * d;
            float acc = S.DZ[idx];
            for (int j = 0; j < d; ++j) acc = fmaf(S.W[j * dp + ii], x[j], acc);
            for (int s = 0; s <= t; ++s) acc = fmaf(S.DA[t * b + s] * S.et[s] * inv_b, S.K[s * d + ii], acc);
            p.dQ[(tok0 + t0) * d + idx] = acc;
        }
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int s = idx / d, ii = idx - s * d;
            float acc = 0.f;
            for (int t = s; t < b; ++t) acc = fmaf(S.DA[t * b + s], S.Q[t * d + ii], acc);
            S.KA[idx] += S.et[s] * inv_b * acc;
        }
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int s = idx / d, j = idx - s * d;
            const float es = S.et[s] * inv_b;
            float acc = 0.f;
            for (int t = s; t < b; ++t) acc = fmaf(S.QK[t * b + s], S.DP[t * d + j], acc);
            S.P[idx] = -es * (acc + S.R[idx]);
        }
        for (int s = warp; s < b; s += kWarps) {
            float acc = 0.f;
            for (int t = s + lane; t < b; t += 32) acc = fmaf(S.DA[t * b + s], S.QK[t * b + s], acc);
            for (int j = lane; j < d; j += 32) acc = fmaf(-S.G[s * d + j], S.R[s * d + j], acc);
            acc = wsum(acc);
            if (lane == 0) S.det[s] = acc * inv_b;
        }
        __syncthreads();
        // through g_s = r_s P_s u_s and the key LayerNorm: dy_s into P, du_s into DU, dv_s
        for (int s = warp; s < b; s += kWarps) {
            const float r = S.rk[s], m2 = S.m2k[s];
            float h[kMaxPer], yh[kMaxPer], u[kMaxPer], dyh[kMaxPer];
            float hm = 0.f, hy = 0.f, hg = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxPer; ++q) {
                const int j = lane + 32 * q;
                h[q] = yh[q] = u[q] = 0.f;
                if (j < d) {
                    h[q] = S.P[s * d + j];
                    yh[q] = S.Yh[s * d + j];
                    u[q] = 2.f * S.gam[j] * S.E[s * d + j];
                    hm += h[q];
                    hy += h[q] * yh[q];
                    hg += h[q] * S.G[s * d + j];
                }
            }
            hm = wsum(hm) * inv_d;
            hy = wsum(hy) * inv_d;
            hg = wsum(hg);
            float am = 0.f, ay = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxPer; ++q) {
                const int j = lane + 32 * q;
                dyh[q] = 0.f;
                if (j < d) {
                    const float du = r * (h[q] - hm - yh[q] * hy);
                    const float de = 2.f * S.gam[j] * du;
                    S.DU[s * d + j] = du;
                    p.dV[(tok0 + t0 + s) * d + j] = -de;
                    dyh[q] = S.gam[j] * de - r * (h[q] * m2 + hy * u[q]);
                    am += dyh[q];
                    ay += dyh[q] * yh[q];
                }
            }
            am = wsum(am) * inv_d;
            ay = wsum(ay) * inv_d;
            const float dsig = -r * hg;
#pragma unroll
            for (int q = 0; q < kMaxPer; ++q) {
                const int j = lane + 32 * q;
                if (j < d) S.P[s * d + j] = r * (dyh[q] - am - yh[q] * ay) + dsig * yh[q] * inv_d;
            }
        }
        __syncthreads();
        // dk_s, the weight gradients carried to batch i - 1, dgamma/dbeta, deta
        for (int idx = tid; idx < b * d; idx += kThreads) {
            const int s = idx / d, ii = idx - s * d;
            const float *x = S.P + s * d;
            float acc = S.KA[idx] + 2.f * S.gam[ii] * S.DU[idx];
            for (int j = 0; j < d; ++j) acc = fmaf(S.W[j * dp + ii], x[j], acc);
            p.dK[(tok0 + t0) * d + idx] = acc;
        }
        for (int idx = tid; idx < d * d; idx += kThreads) {
            const int j = idx / d, ii = idx - j * d;
            float acc = 0.f;
            for (int t = 0; t < b; ++t) {
                acc = fmaf(S.DP[t * d + j], S.Q[t * d + ii], acc);
                acc = fmaf(S.P[t * d + j], S.K[t * d + ii], acc);
            }
            S.dW[j * dp + ii] += acc;
        }
        for (int j = tid; j < d; j += kThreads) {
            float ac = 0.f, ag = 0.f, ab = 0.f;
            for (int s = 0; s < b; ++s) {
                const float du = S.DU[s * d + j];
                ac += S.DP[s * d + j] + S.P[s * d + j];
                ag = fmaf(2.f * du, S.gam[j] * S.Yh[s * d + j] + S.E[s * d + j], ag);
                ab = fmaf(2.f * S.gam[j], du, ab);
            }
            S.dc[j] += ac;
            S.dgam[j] += ag;
            S.dbet[j] += ab;
        }
        for (int s = tid; s < b; s += kThreads) {
            float v = S.det[s];
            if (p.eta_gate) {
                const float sg = 1.f / (1.f + __expf(-eg[t0 + s]));
                v *= p.eta_base * sg * (1.f - sg);
            }
            p.deta[tok0 + t0 + s] = v;
        }
    }
    __syncthreads();
    bool bad = false;
    for (int idx = tid; idx < d * d; idx += kThreads) {
        const float v = S.dW[(idx / d) * dp + idx % d];
        bad |= !isfinite(v);
        p.dW0[(size_t)chain * d * d + idx] = v;
    }
    for (int j = tid; j < d; j += kThreads) {
        bad |= !isfinite(S.dc[j]) || !isfinite(S.dgam[j]) || !isfinite(S.dbet[j]);
        p.dc0[(size_t)chain * d + j] = S.dc[j];
        p.dln_g[(size_t)chain * d + j] = S.dgam[j];
        p.dln_b[(size_t)chain * d + j] = S.dbet[j];
    }
    if (bad && p.status) atomicCAS(p.status, 0, TTT_ERR_NONFINITE);
}

// ------------------------------------------------------------------ tiled kernel (compile-time D, MB)
//
// The same steps with the sizes fixed at compile time. Rows of every b x D
// tile and of W, dW are padded to LD = D + 4 floats: 16-byte rows, so float4
// loads along a row are free of bank conflicts whichever rows the lanes hold.
// NT threads. Each thread keeps RPT accumulators (rows rg, rg + NG, ... of one
// column) for the b x D products and a TR x TC block (rows tid / 16 + (NT / 16) x,
// columns 4 (tid % 16) + 64 q + k) for the D x D outer products; the LayerNorm
// rows of a warp are reduced together. The workspace layout is the general
// kernel's.
template <int D, int MB, int NT>
struct Tiled {
    static constexpr int LD = D + 4;
    static constexpr int NW = NT / 32;       // warps
    static constexpr int NG = NT / D;        // row groups of the b x D products
    static constexpr int RPT = MB / NG;      // rows per thread
    static constexpr int TR = D * 16 / NT;   // outer-product rows per thread (strided by NT / 16)
    static constexpr int TC = D / 16;        // outer-product columns per thread (float4 groups 64 apart)
    static constexpr int RW = MB / NW;       // LayerNorm rows per warp
    static constexpr int EL = D / 32;        // row elements per lane
    static_assert(NG * D == NT && RPT * NG == MB && RW * NW == MB && EL * 32 == D && TC % 4 == 0 &&
                      TR * (NT / 16) == D,
                  "tiling");
    static constexpr size_t kFloats = 2 * (size_t)D * LD + 6 * D + 10 * (size_t)MB * LD + 2 * MB * MB + 4 * MB;
};

struct SmemT {
    float *W, *dW, *c, *dc, *gam, *bet, *dgam, *dbet;
    float *K, *Q, *E, *DZ, *Yh, *P, *G, *DP, *R, *KA;  // R also holds du_s once dg_s is formed
    float *QK, *DA, *et, *det, *rk, *m2k;
};

template <int D, int MB, int NT>
__device__ SmemT carve_t(float *sm)
{
    using C = Tiled<D, MB, NT>;
    SmemT s;
    float *p = sm;
    auto take = [&](size_t n) { float *q = p; p += n; return q; };
    s.W = take(D * C::LD);
    s.dW = take(D * C::LD);
    s.c = take(D);
    s.dc = take(D);
    s.gam = take(D);
    s.bet = take(D);
    s.dgam = take(D);
    s.dbet = take(D);
    s.K = take(MB * C::LD);
    s.Q = take(MB * C::LD);
    s.E = take(MB * C::LD);
    s.DZ = take(MB * C::LD);
    s.Yh = take(MB * C::LD);
    s.P = take(MB * C::LD);
    s.G = take(MB * C::LD);
    s.DP = take(MB * C::LD);
    s.R = take(MB * C::LD);
    s.KA = take(MB * C::LD);
    s.QK = take(MB * MB);
    s.DA = take(MB * MB);
    s.et = take(MB);
    s.det = take(MB);
    s.rk = take(MB);
    s.m2k = take(MB);
    return s;
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

template <typename IO>
__device__ __forceinline__ float4 ldg4(const IO *p);
template <>
__device__ __forceinline__ float4 ldg4<float>(const float *p) { return *reinterpret_cast<const float4 *>(p); }
template <>
__device__ __forceinline__ float4 ldg4<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// One 4-element chunk of an input tile as loaded from global memory, before
// conversion to fp32 (the register form of the next mini-batch's prefetch).
template <typename IO>
struct RawChunk;
template <>
struct RawChunk<float> {
    using T = float4;
};
template <>
struct RawChunk<__nv_bfloat16> {
    using T = uint2;
};
template <typename IO>
__device__ __forceinline__ typename RawChunk<IO>::T ldraw(const IO *p)
{
    return *reinterpret_cast<const typename RawChunk<IO>::T *>(p);
}
__device__ __forceinline__ float4 cvt4(const float4 &r) { return r; }
__device__ __forceinline__ float4 cvt4(const uint2 &u)
{
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

template <int N>
__device__ __forceinline__ void wsum_n(float (&v)[N])
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int r = 0; r < N; ++r) v[r] += __shfl_xor_sync(0xffffffffu, v[r], o);
}

// acc[r] += sum_i X[row r][i] M[c][i] (and acc2 with X2): the "times M^T" products.
template <int D, int MB, int NT, bool TWO>
__device__ __forceinline__ void prod_mt(float (&acc)[Tiled<D, MB, NT>::RPT], float (&acc2)[Tiled<D, MB, NT>::RPT],
                                        const float *X, const float *X2, const float *M, int c, int rg)
{
    using C = Tiled<D, MB, NT>;
#pragma unroll 4
    for (int i = 0; i < D; i += 4) {
        const float4 m = ld4(M + c * C::LD + i);
#pragma unroll
        for (int r = 0; r < C::RPT; ++r) {
            const float4 x = ld4(X + (rg + C::NG * r) * C::LD + i);
            acc[r] = fmaf(x.x, m.x, fmaf(x.y, m.y, fmaf(x.z, m.z, fmaf(x.w, m.w, acc[r]))));
            if (TWO) {
                const float4 x2 = ld4(X2 + (rg + C::NG * r) * C::LD + i);
                acc2[r] = fmaf(x2.x, m.x, fmaf(x2.y, m.y, fmaf(x2.z, m.z, fmaf(x2.w, m.w, acc2[r]))));
            }
        }
    }
}

// acc[r] += sum_j X[row r][j] M[j][c]: the "times M" products.
template <int D, int MB, int NT>
__device__ __forceinline__ void prod_m(float (&acc)[Tiled<D, MB, NT>::RPT], const float *X, const float *M, int c,
                                       int rg)
{
    using C = Tiled<D, MB, NT>;
#pragma unroll 2
    for (int j = 0; j < D; j += 4) {
        const float m0 = M[j * C::LD + c], m1 = M[(j + 1) * C::LD + c];
        const float m2 = M[(j + 2) * C::LD + c], m3 = M[(j + 3) * C::LD + c];
#pragma unroll
        for (int r = 0; r < C::RPT; ++r) {
            const float4 x = ld4(X + (rg + C::NG * r) * C::LD + j);
            acc[r] = fmaf(x.x, m0, fmaf(x.y, m1, fmaf(x.z, m2, fmaf(x.w, m3, acc[r]))));
        }
    }
}

// acc[x][y] += sum_t sc_t A[t][row x] B[t][col y] (sc_t = 1 without a scale),
// with this thread's block rows / columns.
template <int D, int MB, int NT, bool SCALE>
__device__ __forceinline__ void outer_acc(float (&acc)[Tiled<D, MB, NT>::TR][Tiled<D, MB, NT>::TC],
                                          const float *A, const float *Bm, const float *sc, int tid)
{
    using C = Tiled<D, MB, NT>;
    const int r0 = tid >> 4, c0 = 4 * (tid & 15);
#pragma unroll 2
    for (int t = 0; t < MB; ++t) {
        float a[C::TR], bb[C::TC];
#pragma unroll
        for (int x = 0; x < C::TR; ++x) a[x] = A[t * C::LD + r0 + (NT / 16) * x];
#pragma unroll
        for (int q = 0; q < C::TC / 4; ++q) {
            const float4 bv = ld4(Bm + t * C::LD + c0 + 64 * q);
            bb[4 * q] = bv.x, bb[4 * q + 1] = bv.y, bb[4 * q + 2] = bv.z, bb[4 * q + 3] = bv.w;
        }
        if (SCALE) {
            const float s = sc[t];
#pragma unroll
            for (int x = 0; x < C::TR; ++x) a[x] *= s;
        }
#pragma unroll
        for (int x = 0; x < C::TR; ++x)
#pragma unroll
            for (int y = 0; y < C::TC; ++y) acc[x][y] = fmaf(a[x], bb[y], acc[x][y]);
    }
}

// M[row x][col y] += f * acc[x][y] for this thread's block.
template <int D, int MB, int NT>
__device__ __forceinline__ void outer_store(float *M, const float (&acc)[Tiled<D, MB, NT>::TR][Tiled<D, MB, NT>::TC],
                                            float f, int tid)
{
    using C = Tiled<D, MB, NT>;
    const int r0 = tid >> 4, c0 = 4 * (tid & 15);
#pragma unroll
    for (int x = 0; x < C::TR; ++x)
#pragma unroll
        for (int q = 0; q < C::TC / 4; ++q) {
            float *row = M + (r0 + (NT / 16) * x) * C::LD + c0 + 64 * q;
            float4 v = ld4(row);
            v.x = fmaf(f, acc[x][4 * q], v.x);
            v.y = fmaf(f, acc[x][4 * q + 1], v.y);
            v.z = fmaf(f, acc[x][4 * q + 2], v.z);
            v.w = fmaf(f, acc[x][4 * q + 3], v.w);
            st4(row, v);
        }
}

// Key rows (tiled): Yh holds y_s on entry; leaves yh_s in Yh, e_s in E (v_s on
// entry), g_s in G, r_s and mean(u_s*yh_s) in rk, m2k.
template <int D, int MB, int NT>
__device__ __forceinline__ void key_rows_t(const SmemT &S, float eps, int warp, int lane)
{
    using C = Tiled<D, MB, NT>;
    constexpr float inv_d = 1.f / (float)D;
    float y[C::RW][C::EL], mu[C::RW], var[C::RW], m1[C::RW], m2[C::RW], r_[C::RW];
#pragma unroll
    for (int r = 0; r < C::RW; ++r) {
        mu[r] = 0.f;
#pragma unroll
        for (int e = 0; e < C::EL; ++e) {
            y[r][e] = S.Yh[(warp + C::NW * r) * C::LD + lane + 32 * e];
            mu[r] += y[r][e];
        }
    }
    wsum_n(mu);
#pragma unroll
    for (int r = 0; r < C::RW; ++r) {
        mu[r] *= inv_d;
        var[r] = 0.f;
#pragma unroll
        for (int e = 0; e < C::EL; ++e) var[r] = fmaf(y[r][e] - mu[r], y[r][e] - mu[r], var[r]);
    }
    wsum_n(var);
#pragma unroll
    for (int r = 0; r < C::RW; ++r) {
        const int s = warp + C::NW * r;
        r_[r] = rsqrtf(var[r] * inv_d + eps);
        m1[r] = m2[r] = 0.f;
#pragma unroll
        for (int e = 0; e < C::EL; ++e) {
            const int j = lane + 32 * e;
            const float yh = (y[r][e] - mu[r]) * r_[r];
            const float ee = S.K[s * C::LD + j] + S.gam[j] * yh + S.bet[j] - S.E[s * C::LD + j];
            const float u = 2.f * S.gam[j] * ee;
            y[r][e] = yh;
            S.Yh[s * C::LD + j] = yh;
            S.E[s * C::LD + j] = ee;
            m1[r] += u;
            m2[r] = fmaf(u, yh, m2[r]);
        }
    }
    wsum_n(m1);
    wsum_n(m2);
#pragma unroll
    for (int r = 0; r < C::RW; ++r) {
        const int s = warp + C::NW * r;
        m1[r] *= inv_d;
        m2[r] *= inv_d;
#pragma unroll
        for (int e = 0; e < C::EL; ++e) {
            const int j = lane + 32 * e;
            S.G[s * C::LD + j] = r_[r] * (2.f * S.gam[j] * S.E[s * C::LD + j] - m1[r] - y[r][e] * m2[r]);
        }
        if (lane == 0) {
            S.rk[s] = r_[r];
            S.m2k[s] = m2[r];
        }
    }
}

// ------------------------------------------------------------------ tensor-core products (tf32)
// The contractions of the tiled kernel on mma.sync m16n8k8 with tf32 operands
// (fp32 range, operands rounded to nearest to 10 mantissa bits) and fp32
// accumulation, operands from the shared-memory tiles (see the operand sources
// below). Accumulator element r of a tile is (m0 + g + 8 (r >> 1),
// n0 + 2 c4 + (r & 1)).
// An fp32 value as a tf32 mma operand, rounded to nearest: the tensor cores
// read the top 19 bits of the container (sign, exponent, 10 mantissa bits),
// so adding half of the dropped part (bit 12) first makes their truncation a
// rounding (ties away from zero). One integer add instead of a conversion
// instruction on a slower pipe.
__device__ __forceinline__ uint32_t to_tf32(float x) { return __float_as_uint(x) + 0x1000u; }

// x with the 13 bits the tensor cores drop cleared: hi of the split x = hi + lo
// (lo = x - hi is exact, below 2^-10 |x|, and its own tf32 rounding costs
// 2^-21 |x| at most).
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Operand sources. A fragment (16 x 8, rows m0.., columns k0..): lane (g, c4)
// holds A(m0 + g, k0 + c4), A(m0 + g + 8, k0 + c4), A(m0 + g, k0 + c4 + 4),
// A(m0 + g + 8, k0 + c4 + 4); B fragment (8 x 8): B(k0 + c4, n0 + g),
// B(k0 + c4 + 4, n0 + g). ARows / BRowsT read a row-major fp32 tile with one
// ldmatrix: viewed as 16-bit pairs, an 8 x 4 block of fp32 is an 8 x 8 b16
// matrix, and ldmatrix hands lane (g, c4) the 32-bit word (row g, column c4),
// which is the fragment element. Row starts must be 16-byte aligned. EXACT
// marks a source whose values tf32 holds exactly (tiles of bf16 inputs: 8
// mantissa bits), so split precision needs no low part for it.
template <bool EXACT = false>
struct ARows {  // A(m, k) = p[m * ld + k]
    static constexpr bool kExact = EXACT;
    const float *p;
    int ld;
    __device__ __forceinline__ void frag(uint32_t (&a)[4], int m0, int k0, int lane) const
    {
        const int row = m0 + (lane & 7) + 8 * ((lane >> 3) & 1), col = k0 + 4 * (lane >> 4);
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                     : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p + row * ld + col))));
    }
};
template <bool EXACT = false>
struct BRowsT {  // B(k, n) = p[n * ld + k]
    static constexpr bool kExact = EXACT;
    const float *p;
    int ld;
    __device__ __forceinline__ void frag(uint32_t (&b)[2], int k0, int n0, int lane) const
    {
        const int l = lane & 15, row = n0 + (l & 7), col = k0 + 4 * (l >> 3);
        asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                     : "=r"(b[0]), "=r"(b[1])
                     : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p + row * ld + col))));
    }
};
template <class F, bool EXACT = false>
struct AFn {  // A(m, k) = f(m, k)
    static constexpr bool kExact = EXACT;
    F f;
    __device__ __forceinline__ void frag(uint32_t (&a)[4], int m0, int k0, int lane) const
    {
        const int g = lane >> 2, c4 = lane & 3;
        a[0] = __float_as_uint(f(m0 + g, k0 + c4));
        a[1] = __float_as_uint(f(m0 + g + 8, k0 + c4));
        a[2] = __float_as_uint(f(m0 + g, k0 + c4 + 4));
        a[3] = __float_as_uint(f(m0 + g + 8, k0 + c4 + 4));
    }
};
template <class F, bool EXACT = false>
struct BFn {  // B(k, n) = f(k, n)
    static constexpr bool kExact = EXACT;
    F f;
    __device__ __forceinline__ void frag(uint32_t (&b)[2], int k0, int n0, int lane) const
    {
        const int g = lane >> 2, c4 = lane & 3;
        b[0] = __float_as_uint(f(k0 + c4, n0 + g));
        b[1] = __float_as_uint(f(k0 + c4 + 4, n0 + g));
    }
};
template <bool EXACT = false, class F>
__device__ __forceinline__ AFn<F, EXACT> afn(F f) { return AFn<F, EXACT>{f}; }
template <bool EXACT = false, class F>
__device__ __forceinline__ BFn<F, EXACT> bfn(F f) { return BFn<F, EXACT>{f}; }
struct NoOp {  // an absent second product
    static constexpr bool kExact = true;
    __device__ __forceinline__ void frag(uint32_t (&a)[4], int, int, int) const {}
    __device__ __forceinline__ void frag(uint32_t (&b)[2], int, int, int) const {}
};

// X3: split precision. Each operand x is carried as hi = tf32(x) and lo =
// tf32(x - hi), and the product as hi*hi + hi*lo + lo*hi (three mma): about
// 21 of the 24 fp32 mantissa bits, for the products whose rounding would
// otherwise be carried through the inner loop's recurrence.
template <bool X3 = false, class SA, class SB>
__device__ __forceinline__ void mma_k8(float (&acc)[4], const SA &sa, const SB &sb, int m0, int n0, int k0, int lane)
{
    uint32_t a[4], b[2];
    sa.frag(a, m0, k0, lane);
    sb.frag(b, k0, n0, lane);
    uint32_t ah[4], bh[2];
    if constexpr (X3) {
        uint32_t al[4], bl[2];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if constexpr (SA::kExact) {
                ah[r] = a[r];
            } else {
                const float h = tf32_hi(__uint_as_float(a[r]));
                ah[r] = __float_as_uint(h);
                al[r] = to_tf32(__uint_as_float(a[r]) - h);
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if constexpr (SB::kExact) {
                bh[r] = b[r];
            } else {
                const float h = tf32_hi(__uint_as_float(b[r]));
                bh[r] = __float_as_uint(h);
                bl[r] = to_tf32(__uint_as_float(b[r]) - h);
            }
        }
        if constexpr (!SA::kExact) mma_tf32(acc, al[0], al[1], al[2], al[3], bh[0], bh[1]);
        if constexpr (!SB::kExact) mma_tf32(acc, ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
    } else {
#pragma unroll
        for (int r = 0; r < 4; ++r) ah[r] = a[r] + 0x1000u;
#pragma unroll
        for (int r = 0; r < 2; ++r) bh[r] = b[r] + 0x1000u;
    }
    mma_tf32(acc, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
}

// acc += sum over k < K of A(m0 + ., k) B(k, n0 + .), in two independent chains
// (even and odd k8 blocks) that are added at the end.
template <int K, bool X3 = false, class FA, class FB>
__device__ __forceinline__ void mma_run(float (&acc)[4], const FA &fa, const FB &fb, int m0, int n0, int lane)
{
    if constexpr (K == 8) {
        mma_k8<X3>(acc, fa, fb, m0, n0, 0, lane);
    } else {
        float odd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < K; k0 += 16) {
            mma_k8<X3>(acc, fa, fb, m0, n0, k0, lane);
            mma_k8<X3>(odd, fa, fb, m0, n0, k0 + 8, lane);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] += odd[r];
    }
}

// The 16 x N result R(m, n) = init(m, n) + sum_k A1(m, k) B1(k, n) [+ sum_k A2(m, k) B2(k, n)]
// (operand sources fa*, fb*): warp w forms the n-tiles w, w + NW, ... and hands
// every element to out(m, n, v).
template <int N, int NW, int K1, int K2, bool X3 = false, class FI, class FA1, class FB1, class FA2, class FB2,
          class FO>
__device__ __forceinline__ void tc_rows(const FI &init, const FA1 &fa1, const FB1 &fb1, const FA2 &fa2, const FB2 &fb2,
                                        const FO &out, int warp, int lane)
{
    const int g = lane >> 2, c4 = lane & 3;
#pragma unroll
    for (int nt = warp; nt < N / 8; nt += NW) {
        const int n0 = 8 * nt;
        float acc[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] = init(g + 8 * (r >> 1), n0 + 2 * c4 + (r & 1));
        mma_run<K1, X3>(acc, fa1, fb1, 0, n0, lane);
        if constexpr (K2 > 0) {
            float acc2[4] = {0.f, 0.f, 0.f, 0.f};
            mma_run<K2, X3>(acc2, fa2, fb2, 0, n0, lane);
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[r] += acc2[r];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) out(g + 8 * (r >> 1), n0 + 2 * c4 + (r & 1), acc[r]);
    }
}

// The D x D result of one or two outer-product sums over the MB tokens,
// sum_t A1(x, t) B1(t, y) [+ sum_t A2(x, t) B2(t, y)] (operand sources), handed to out(x, y, v);
// warp w forms the 16 x 8 tiles w, w + NW, ... (D / 16 x D / 8 of them).
template <int D, int MB, int NW, bool TWO, bool X3 = false, class FA1, class FB1, class FA2, class FB2, class FO>
__device__ __forceinline__ void tc_outer(const FA1 &fa1, const FB1 &fb1, const FA2 &fa2, const FB2 &fb2, const FO &out,
                                         int warp, int lane)
{
    constexpr int MTL = D / 16, TILES = MTL * (D / 8);
    static_assert(TILES % NW == 0, "whole tiles per warp");
    const int g = lane >> 2, c4 = lane & 3;
#pragma unroll
    for (int q = 0; q < TILES / NW; ++q) {
        const int tile = warp + NW * q;
        const int m0 = 16 * (tile % MTL), n0 = 8 * (tile / MTL);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < MB; k0 += 8) {
            mma_k8<X3>(acc, fa1, fb1, m0, n0, k0, lane);
            if constexpr (TWO) mma_k8<X3>(acc, fa2, fb2, m0, n0, k0, lane);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) out(m0 + g + 8 * (r >> 1), n0 + 2 * c4 + (r & 1), acc[r]);
    }
}

// MATH 0: fp32 FFMA throughout. MATH 1: every contraction on the tensor cores
// in split precision (three tf32 products per product: fp32-grade results).
// MATH 2: the same with one tf32 product, except in the forward sweep, which
// recomputes the weight trajectory and keeps split precision.
template <typename IO, int D, int MB, int NT, int MATH = 0>
__global__ void __launch_bounds__(NT, 1) linear_bwd_tiled_kernel(LinearBwdParams p)
{
    constexpr bool TC = MATH != 0, X3 = MATH == 1;
    constexpr bool QE = std::is_same<IO, __nv_bfloat16>::value;  // K, Q tiles hold bf16 values: exact in tf32
    using C = Tiled<D, MB, NT>;
    const NoOp none{};
    constexpr int LD = C::LD, NG = C::NG, RPT = C::RPT, RW = C::RW, EL = C::EL, NW = C::NW;
    constexpr float inv_b = 1.f / (float)MB, inv_d = 1.f / (float)D;
    extern __shared__ __align__(16) float smt[];
    const SmemT S = carve_t<D, MB, NT>(smt);
    const int T = p.T, n = T / MB;
    const int chain = blockIdx.x;
    const int bi = chain / p.H, hi = chain % p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int col = tid % D, rg = tid / D;  // b x D products: column, row group
    const size_t tok0 = (size_t)chain * T;
    const IO *Qg = static_cast<const IO *>(p.Q) + tok0 * D;
    const IO *Kg = static_cast<const IO *>(p.K) + tok0 * D;
    const IO *Vg = static_cast<const IO *>(p.V) + tok0 * D;
    const IO *DZg = static_cast<const IO *>(p.dZ) + tok0 * D;
    const float *eg = p.eta + tok0;
    // workspace of the chain: every mini-batch's starting state (W, c), then every
    // mini-batch's key side (yh, e, g [MB][D] and r, mean(u yh) [MB]) for the reverse sweep.
    // SAVE goes with the register prefetch (PF, 256 threads); at d = 64 the key side is
    // prefetched into registers too (PFS), at d = 128 (no registers to spare) it is loaded
    // at the start of its mini-batch.
    constexpr bool SAVE = NT == 256, PFS = SAVE && D == 64;
    constexpr size_t SVL = (size_t)MB * (3 * D + 2);
    float *ws = p.ws + (size_t)chain * (n * ((size_t)D * D + D) + (size_t)T * (3 * D + 2));
    float *svb = ws + (size_t)n * ((size_t)D * D + D);

    {
        const float *W0 = p.W0 + bi * p.w0_bstride + (long long)hi * D * D;
        const float *c0 = p.c0 + bi * p.c0_bstride + (long long)hi * D;
        for (int q = tid; q < D * D / 4; q += NT) {
            const int j = (4 * q) / D, i = (4 * q) % D;
            st4(S.W + j * LD + i, ld4(W0 + 4 * q));
            st4(S.dW + j * LD + i, p.dW_n ? ld4(p.dW_n + (size_t)chain * D * D + 4 * q) : make_float4(0.f, 0.f, 0.f, 0.f));
        }
        for (int j = tid; j < D; j += NT) {
            S.c[j] = c0[j];
            S.dc[j] = p.dc_n ? p.dc_n[(size_t)chain * D + j] : 0.f;
            S.gam[j] = p.ln_g[hi * D + j];
            S.bet[j] = p.ln_b[hi * D + j];
            S.dgam[j] = 0.f;
            S.dbet[j] = 0.f;
        }
    }
    auto load_tile = [&](float *dst, const IO *src) {
        for (int q = tid; q < MB * D / 4; q += NT) {
            const int s = (4 * q) / D, i = (4 * q) % D;
            st4(dst + s * LD + i, ldg4<IO>(src + 4 * q));
        }
    };
    auto load_eta = [&](int t0) {
        for (int s = tid; s < MB; s += NT) {
            const float e = eg[t0 + s];
            S.et[s] = p.eta_gate ? p.eta_base / (1.f + __expf(-e)) : e;
        }
    };
    // Register prefetch of the next mini-batch (256-thread kernels, which have
    // registers to spare): its global loads are issued at the start of the
    // current mini-batch's last phase and land in shared memory after it.
    constexpr bool PF = NT == 256;
    constexpr int CT = (MB * D / 4 + NT - 1) / NT, CW = (D * D / 4 + NT - 1) / NT;
    using RC = typename RawChunk<IO>::T;
    RC pk[CT], pq[CT], pv[CT], pz[CT];
    float4 pw[CW];
    float pc = 0.f, pe = 0.f;
    float4 sy[CT], se[CT], sg[CT];  // prefetched key side (SAVE)
    float sr = 0.f, sm2 = 0.f;
    auto issue_tiles = [&](int t0, bool rev) {
#pragma unroll
        for (int u = 0; u < CT; ++u) {
            const int q = tid + u * NT;
            if (q < MB * D / 4) {
                const size_t g = (size_t)t0 * D + 4 * q;
                pk[u] = ldraw<IO>(Kg + g);
                if (!(SAVE && rev)) pv[u] = ldraw<IO>(Vg + g);  // the reverse sweep reads e, not v
                if (rev) {
                    pq[u] = ldraw<IO>(Qg + g);
                    pz[u] = ldraw<IO>(DZg + g);
                }
            }
        }
        pe = tid < MB ? eg[t0 + tid] : 0.f;
    };
    auto commit_tiles = [&](bool rev) {
#pragma unroll
        for (int u = 0; u < CT; ++u) {
            const int q = tid + u * NT;
            if (q < MB * D / 4) {
                const int s = (4 * q) / D, ii = (4 * q) % D;
                st4(S.K + s * LD + ii, cvt4(pk[u]));
                if (!(SAVE && rev)) st4(S.E + s * LD + ii, cvt4(pv[u]));
                if (rev) {
                    st4(S.Q + s * LD + ii, cvt4(pq[u]));
                    st4(S.DZ + s * LD + ii, cvt4(pz[u]));
                }
            }
        }
        if (tid < MB) S.et[tid] = p.eta_gate ? p.eta_base / (1.f + __expf(-pe)) : pe;
    };
    auto issue_saved = [&](int i) {
        const float *sv = svb + (size_t)i * SVL;
#pragma unroll
        for (int u = 0; u < CT; ++u) {
            const int q = tid + u * NT;
            if (q < MB * D / 4) {
                sy[u] = ld4(sv + 4 * q);
                se[u] = ld4(sv + MB * D + 4 * q);
                sg[u] = ld4(sv + 2 * MB * D + 4 * q);
            }
        }
        sr = tid < MB ? sv[3 * MB * D + tid] : 0.f;
        sm2 = tid < MB ? sv[3 * MB * D + MB + tid] : 0.f;
    };
    auto commit_saved = [&]() {
#pragma unroll
        for (int u = 0; u < CT; ++u) {
            const int q = tid + u * NT;
            if (q < MB * D / 4) {
                const int s = (4 * q) / D, ii = (4 * q) % D;
                st4(S.Yh + s * LD + ii, sy[u]);
                st4(S.E + s * LD + ii, se[u]);
                st4(S.G + s * LD + ii, sg[u]);
            }
        }
        if (tid < MB) {
            S.rk[tid] = sr;
            S.m2k[tid] = sm2;
        }
    };
    auto issue_anchor = [&](int i) {
        const float *wsi = ws + (size_t)i * ((size_t)D * D + D);
#pragma unroll
        for (int u = 0; u < CW; ++u) {
            const int q = tid + u * NT;
            if (q < D * D / 4) pw[u] = ld4(wsi + 4 * q);
        }
        pc = tid < D ? wsi[D * D + tid] : 0.f;
    };
    auto commit_anchor = [&]() {
#pragma unroll
        for (int u = 0; u < CW; ++u) {
            const int q = tid + u * NT;
            if (q < D * D / 4) st4(S.W + ((4 * q) / D) * LD + (4 * q) % D, pw[u]);
        }
        if (tid < D) S.c[tid] = pc;
    };

    // ---- forward sweep
    if (PF) issue_tiles(0, false);
    for (int i = 0; i < n; ++i) {
        const int t0 = i * MB;
        __syncthreads();
        float *wsi = ws + (size_t)i * ((size_t)D * D + D);
        for (int q = tid; q < D * D / 4; q += NT) {
            const int j = (4 * q) / D, ii = (4 * q) % D;
            st4(wsi + 4 * q, ld4(S.W + j * LD + ii));
        }
        for (int j = tid; j < D; j += NT) wsi[D * D + j] = S.c[j];
        if (PF) {
            commit_tiles(false);
        } else {
            load_tile(S.K, Kg + (size_t)t0 * D);
            load_tile(S.E, Vg + (size_t)t0 * D);
            load_eta(t0);
        }
        __syncthreads();
        if constexpr (TC) {  // the forward sweep recomputes the trajectory: split precision
            tc_rows<D, NW, D, 0, true>([&](int, int n) { return S.c[n]; }, ARows<QE>{S.K, LD}, BRowsT<>{S.W, LD}, none, none,
                                       [&](int m, int n, float v) { S.Yh[m * LD + n] = v; }, warp, lane);
        } else {
            float a[RPT], dummy[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) a[r] = S.c[col];
            prod_mt<D, MB, NT, false>(a, dummy, S.K, nullptr, S.W, col, rg);
#pragma unroll
            for (int r = 0; r < RPT; ++r) S.Yh[(rg + NG * r) * LD + col] = a[r];
        }
        __syncthreads();
        key_rows_t<D, MB, NT>(S, p.eps, warp, lane);
        __syncthreads();
        if (PF && i + 1 < n) issue_tiles(t0 + MB, false);
        if (SAVE) {
            float *sv = svb + (size_t)i * SVL;
            for (int q = tid; q < MB * D / 4; q += NT) {
                const int s = (4 * q) / D, ii = (4 * q) % D;
                st4(sv + 4 * q, ld4(S.Yh + s * LD + ii));
                st4(sv + MB * D + 4 * q, ld4(S.E + s * LD + ii));
                st4(sv + 2 * MB * D + 4 * q, ld4(S.G + s * LD + ii));
            }
            for (int x = tid; x < MB; x += NT) {
                sv[3 * MB * D + x] = S.rk[x];
                sv[3 * MB * D + MB + x] = S.m2k[x];
            }
        }
        if constexpr (TC) {
            tc_outer<D, MB, NW, false, true>(afn([&](int x, int t) { return S.et[t] * S.G[t * LD + x]; }),
                                             bfn<QE>([&](int t, int y) { return S.K[t * LD + y]; }), none, none,
                                       [&](int x, int y, float v) { S.W[x * LD + y] = fmaf(-inv_b, v, S.W[x * LD + y]); },
                                       warp, lane);
        } else {
            float acc[C::TR][C::TC] = {};
            outer_acc<D, MB, NT, true>(acc, S.G, S.K, S.et, tid);
            outer_store<D, MB, NT>(S.W, acc, -inv_b, tid);
        }
        for (int j = tid; j < D; j += NT) {
            float a = 0.f;
#pragma unroll 4
            for (int s = 0; s < MB; ++s) a = fmaf(S.et[s], S.G[s * LD + j], a);
            S.c[j] -= a * inv_b;
        }
    }

    // ---- reverse sweep
    if (PF) {
        __syncthreads();  // the forward sweep's last anchor store is visible
        issue_tiles((n - 1) * MB, true);
        issue_anchor(n - 1);
        if (PFS) issue_saved(n - 1);
    }
    for (int i = n - 1; i >= 0; --i) {
        const int t0 = i * MB;
        __syncthreads();
        if (PF) {
            commit_tiles(true);
            commit_anchor();
            if (PFS) {
                commit_saved();
            } else if (SAVE) {
                const float *sv = svb + (size_t)i * SVL;
                for (int q = tid; q < MB * D / 4; q += NT) {
                    const int s = (4 * q) / D, ii = (4 * q) % D;
                    st4(S.Yh + s * LD + ii, ld4(sv + 4 * q));
                    st4(S.E + s * LD + ii, ld4(sv + MB * D + 4 * q));
                    st4(S.G + s * LD + ii, ld4(sv + 2 * MB * D + 4 * q));
                }
                for (int x = tid; x < MB; x += NT) {
                    S.rk[x] = sv[3 * MB * D + x];
                    S.m2k[x] = sv[3 * MB * D + MB + x];
                }
            }
        } else {
            const float *wsi = ws + (size_t)i * ((size_t)D * D + D);
            for (int q = tid; q < D * D / 4; q += NT) {
                const int j = (4 * q) / D, ii = (4 * q) % D;
                st4(S.W + j * LD + ii, ld4(wsi + 4 * q));
            }
            for (int j = tid; j < D; j += NT) S.c[j] = wsi[D * D + j];
            load_tile(S.K, Kg + (size_t)t0 * D);
            load_tile(S.Q, Qg + (size_t)t0 * D);
            load_tile(S.E, Vg + (size_t)t0 * D);
            load_tile(S.DZ, DZg + (size_t)t0 * D);
            load_eta(t0);
        }
        __syncthreads();
        // y_s = W k_s + c, W q_t + c; R_s = dW' k_s + dc'; q_t.k_s + 1
        if constexpr (TC) {
            tc_rows<D, NW, D, 0, X3>([&](int, int n) { return S.c[n]; }, ARows<QE>{S.Q, LD}, BRowsT<>{S.W, LD}, none, none,
                                 [&](int m, int n, float v) { S.P[m * LD + n] = v; }, warp, lane);
            tc_rows<D, NW, D, 0, X3>([&](int, int n) { return S.dc[n]; }, ARows<QE>{S.K, LD}, BRowsT<>{S.dW, LD}, none, none,
                                 [&](int m, int n, float v) { S.R[m * LD + n] = v; }, warp, lane);
            if (!SAVE)
                tc_rows<D, NW, D, 0, X3>([&](int, int n) { return S.c[n]; }, ARows<QE>{S.K, LD}, BRowsT<>{S.W, LD}, none,
                                         none,
                                     [&](int m, int n, float v) { S.Yh[m * LD + n] = v; }, warp, lane);
            tc_rows<MB, NW, D, 0, X3>([](int, int) { return 1.f; }, ARows<QE>{S.Q, LD}, BRowsT<QE>{S.K, LD}, none, none,
                                  [&](int t, int sc, float v) { S.QK[t * MB + sc] = v; }, warp, lane);
        } else {
            float ak[RPT], aq[RPT], ar[RPT], dummy[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                ak[r] = aq[r] = S.c[col];
                ar[r] = S.dc[col];
            }
            if (SAVE) {
                prod_mt<D, MB, NT, false>(aq, dummy, S.Q, nullptr, S.W, col, rg);  // y_s was saved
            } else {
                prod_mt<D, MB, NT, true>(ak, aq, S.K, S.Q, S.W, col, rg);
            }
            prod_mt<D, MB, NT, false>(ar, dummy, S.K, nullptr, S.dW, col, rg);
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int s = rg + NG * r;
                if (!SAVE) S.Yh[s * LD + col] = ak[r];
                S.P[s * LD + col] = aq[r];
                S.R[s * LD + col] = ar[r];
            }
            for (int idx = tid; idx < MB * MB; idx += NT) {
                const int t = idx / MB, s = idx % MB;
                float acc = 1.f;
#pragma unroll 4
                for (int ii = 0; ii < D; ii += 4) {
                    const float4 q = ld4(S.Q + t * LD + ii), k = ld4(S.K + s * LD + ii);
                    acc = fmaf(q.x, k.x, fmaf(q.y, k.y, fmaf(q.z, k.z, fmaf(q.w, k.w, acc))));
                }
                S.QK[idx] = acc;
            }
        }
        __syncthreads();
        if (!SAVE) {
            key_rows_t<D, MB, NT>(S, p.eps, warp, lane);
            __syncthreads();
        }
        // p_t = W q_t + c - sum_{s<=t} A_ts g_s
        if constexpr (TC) {
            tc_rows<D, NW, MB, 0, X3>([&](int t, int n) { return S.P[t * LD + n]; },
                                  afn([&](int t, int sc) { return sc <= t ? -S.QK[t * MB + sc] * S.et[sc] * inv_b : 0.f; }),
                                  bfn([&](int sc, int n) { return S.G[sc * LD + n]; }), none, none,
                                  [&](int t, int n, float v) { S.P[t * LD + n] = v; }, warp, lane);
        } else {
            float a[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) a[r] = S.P[(rg + NG * r) * LD + col];
            for (int s = 0; s < MB; ++s) {
                const float g = S.G[s * LD + col] * S.et[s] * inv_b;
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const int t = rg + NG * r;
                    if (s <= t) a[r] = fmaf(-S.QK[t * MB + s], g, a[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < RPT; ++r) S.P[(rg + NG * r) * LD + col] = a[r];
        }
        __syncthreads();
        // output LayerNorm rows: ph_t into P, dp_t into DP
        {
            float y[RW][EL], dz[RW][EL], mu[RW], var[RW], a1[RW], a2[RW], rr[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int t = warp + NW * r;
                mu[r] = 0.f;
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    y[r][e] = S.P[t * LD + lane + 32 * e];
                    dz[r][e] = S.DZ[t * LD + lane + 32 * e];
                    mu[r] += y[r][e];
                }
            }
            wsum_n(mu);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                mu[r] *= inv_d;
                var[r] = 0.f;
#pragma unroll
                for (int e = 0; e < EL; ++e) var[r] = fmaf(y[r][e] - mu[r], y[r][e] - mu[r], var[r]);
            }
            wsum_n(var);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int t = warp + NW * r;
                rr[r] = rsqrtf(var[r] * inv_d + p.eps);
                a1[r] = a2[r] = 0.f;
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    const int j = lane + 32 * e;
                    const float ph = (y[r][e] - mu[r]) * rr[r], dh = S.gam[j] * dz[r][e];
                    y[r][e] = ph;
                    S.P[t * LD + j] = ph;
                    a1[r] += dh;
                    a2[r] = fmaf(dh, ph, a2[r]);
                }
            }
            wsum_n(a1);
            wsum_n(a2);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int t = warp + NW * r;
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    const int j = lane + 32 * e;
                    S.DP[t * LD + j] = rr[r] * (S.gam[j] * dz[r][e] - a1[r] * inv_d - y[r][e] * a2[r] * inv_d);
                }
            }
        }
        __syncthreads();
        for (int j = tid; j < D; j += NT) {
            float ag = 0.f, ab = 0.f;
#pragma unroll 4
            for (int t = 0; t < MB; ++t) {
                ag = fmaf(S.DZ[t * LD + j], S.P[t * LD + j], ag);
                ab += S.DZ[t * LD + j];
            }
            S.dgam[j] += ag;
            S.dbet[j] += ab;
        }
        if constexpr (TC) {
            tc_rows<MB, NW, D, 0, X3>([](int, int) { return 0.f; }, ARows<>{S.DP, LD}, BRowsT<>{S.G, LD}, none, none,
                                  [&](int t, int sc, float v) { S.DA[t * MB + sc] = sc <= t ? -v : 0.f; }, warp, lane);
        } else {
            for (int idx = tid; idx < MB * MB; idx += NT) {
                const int t = idx / MB, s = idx % MB;
                float acc = 0.f;
                if (s <= t) {
#pragma unroll 4
                    for (int j = 0; j < D; j += 4) {
                        const float4 x = ld4(S.DP + t * LD + j), g = ld4(S.G + s * LD + j);
                        acc = fmaf(x.x, g.x, fmaf(x.y, g.y, fmaf(x.z, g.z, fmaf(x.w, g.w, acc))));
                    }
                }
                S.DA[idx] = -acc;
            }
        }
        __syncthreads();
        // dq_t; dk_s's q- and dW'-parts (KA); dg_s (into P); deta_s
        if constexpr (TC) {
            float *dQc = p.dQ + (tok0 + t0) * D;
            tc_rows<D, NW, D, MB, X3>([&](int t, int n) { return S.DZ[t * LD + n]; },
                                  ARows<>{S.DP, LD}, bfn([&](int j, int n) { return S.W[j * LD + n]; }),
                                  afn([&](int t, int sc) { return sc <= t ? S.DA[t * MB + sc] * S.et[sc] * inv_b : 0.f; }),
                                  bfn<QE>([&](int sc, int n) { return S.K[sc * LD + n]; }),
                                  [&](int t, int n, float v) { dQc[t * D + n] = v; }, warp, lane);
            tc_rows<D, NW, MB, D, X3>([](int, int) { return 0.f; },
                                  afn([&](int sc, int t) { return t >= sc ? S.DA[t * MB + sc] : 0.f; }),
                                  bfn<QE>([&](int t, int n) { return S.Q[t * LD + n]; }), ARows<>{S.G, LD},
                                  bfn([&](int j, int n) { return -S.dW[j * LD + n]; }),
                                  [&](int sc, int n, float v) { S.KA[sc * LD + n] = S.et[sc] * inv_b * v; }, warp, lane);
            tc_rows<D, NW, MB, 0, X3>([&](int sc, int n) { return S.R[sc * LD + n]; },
                                  afn([&](int sc, int t) { return t >= sc ? S.QK[t * MB + sc] : 0.f; }),
                                  bfn([&](int t, int n) { return S.DP[t * LD + n]; }), none, none,
                                  [&](int sc, int n, float v) { S.P[sc * LD + n] = -S.et[sc] * inv_b * v; }, warp, lane);
        }
        if constexpr (!TC) {
            float a[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) a[r] = S.DZ[(rg + NG * r) * LD + col];
            prod_m<D, MB, NT>(a, S.DP, S.W, col, rg);
            for (int s = 0; s < MB; ++s) {
                const float k = S.K[s * LD + col] * S.et[s] * inv_b;
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const int t = rg + NG * r;
                    if (s <= t) a[r] = fmaf(S.DA[t * MB + s], k, a[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < RPT; ++r) p.dQ[(tok0 + t0 + rg + NG * r) * D + col] = a[r];
        }
        if constexpr (!TC) {
            float a[RPT], mix[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) a[r] = mix[r] = 0.f;
            prod_m<D, MB, NT>(a, S.G, S.dW, col, rg);
            for (int t = 0; t < MB; ++t) {
                const float q = S.Q[t * LD + col];
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const int s = rg + NG * r;
                    if (t >= s) mix[r] = fmaf(S.DA[t * MB + s], q, mix[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int s = rg + NG * r;
                S.KA[s * LD + col] = S.et[s] * inv_b * (mix[r] - a[r]);
            }
        }
        if constexpr (!TC) {
            float a[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) a[r] = 0.f;
            for (int t = 0; t < MB; ++t) {
                const float x = S.DP[t * LD + col];
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const int s = rg + NG * r;
                    if (t >= s) a[r] = fmaf(S.QK[t * MB + s], x, a[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int s = rg + NG * r;
                S.P[s * LD + col] = -S.et[s] * inv_b * (a[r] + S.R[s * LD + col]);
            }
        }
        for (int s = warp; s < MB; s += NW) {
            float acc = 0.f;
            for (int t = s + lane; t < MB; t += 32) acc = fmaf(S.DA[t * MB + s], S.QK[t * MB + s], acc);
#pragma unroll
            for (int e = 0; e < EL; ++e) acc = fmaf(-S.G[s * LD + lane + 32 * e], S.R[s * LD + lane + 32 * e], acc);
            acc = wsum(acc);
            if (lane == 0) S.det[s] = acc * inv_b;
        }
        __syncthreads();
        // through g_s = r_s P_s u_s and the key LayerNorm: dy_s into P, du_s into R, dv_s
        {
            float h[RW][EL], yh[RW][EL], u[RW][EL], dyh[RW][EL];
            float hm[RW], hy[RW], hg[RW], am[RW], ay[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int s = warp + NW * r;
                hm[r] = hy[r] = hg[r] = 0.f;
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    const int j = lane + 32 * e;
                    h[r][e] = S.P[s * LD + j];
                    yh[r][e] = S.Yh[s * LD + j];
                    u[r][e] = 2.f * S.gam[j] * S.E[s * LD + j];
                    hm[r] += h[r][e];
                    hy[r] = fmaf(h[r][e], yh[r][e], hy[r]);
                    hg[r] = fmaf(h[r][e], S.G[s * LD + j], hg[r]);
                }
            }
            wsum_n(hm);
            wsum_n(hy);
            wsum_n(hg);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int s = warp + NW * r;
                const float rs = S.rk[s], m2 = S.m2k[s];
                hm[r] *= inv_d;
                hy[r] *= inv_d;
                am[r] = ay[r] = 0.f;
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    const int j = lane + 32 * e;
                    const float du = rs * (h[r][e] - hm[r] - yh[r][e] * hy[r]);
                    const float de = 2.f * S.gam[j] * du;
                    S.R[s * LD + j] = du;
                    p.dV[(tok0 + t0 + s) * D + j] = -de;
                    dyh[r][e] = S.gam[j] * de - rs * (h[r][e] * m2 + hy[r] * u[r][e]);
                    am[r] += dyh[r][e];
                    ay[r] = fmaf(dyh[r][e], yh[r][e], ay[r]);
                }
            }
            wsum_n(am);
            wsum_n(ay);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int s = warp + NW * r;
                const float rs = S.rk[s], dsig = -rs * hg[r];
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    const int j = lane + 32 * e;
                    S.P[s * LD + j] =
                        rs * (dyh[r][e] - am[r] * inv_d - yh[r][e] * ay[r] * inv_d) + dsig * yh[r][e] * inv_d;
                }
            }
        }
        __syncthreads();
        // dk_s; dW, dc carried to batch i - 1; dgamma, dbeta; deta
        if (PF && i > 0) {
            issue_tiles(t0 - MB, true);
            issue_anchor(i - 1);
            if (PFS) issue_saved(i - 1);
            // d = 128 loads the key side at the start of its mini-batch (no registers to
            // hold it meanwhile): have L2 fetch it now, so that those loads hit L2; and
            // the tiles and starting state two mini-batches ahead, so that the register
            // prefetch of the next step finds them there too (at d = 64 neither helps).
            if (SAVE && !PFS) {
                auto l2 = [&](const void *a, size_t bytes) {
                    const char *c = static_cast<const char *>(a);
                    for (size_t o = (size_t)tid * 128; o < bytes; o += (size_t)NT * 128)
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + o));
                };
                l2(svb + (size_t)(i - 1) * SVL, SVL * 4);
                if (i > 1) {
                    const size_t t2 = (size_t)(t0 - 2 * MB) * D;
                    l2(Kg + t2, (size_t)MB * D * sizeof(IO));
                    l2(Qg + t2, (size_t)MB * D * sizeof(IO));
                    l2(DZg + t2, (size_t)MB * D * sizeof(IO));
                    l2(ws + (size_t)(i - 2) * ((size_t)D * D + D), ((size_t)D * D + D) * 4);
                }
            }
        }
        if constexpr (TC) {
            float *dKc = p.dK + (tok0 + t0) * D;
            tc_rows<D, NW, D, 0, X3>([&](int sc, int n) { return S.KA[sc * LD + n] + 2.f * S.gam[n] * S.R[sc * LD + n]; },
                                 ARows<>{S.P, LD}, bfn([&](int j, int n) { return S.W[j * LD + n]; }), none, none,
                                 [&](int sc, int n, float v) { dKc[sc * D + n] = v; }, warp, lane);
            tc_outer<D, MB, NW, true, X3>(afn([&](int x, int t) { return S.DP[t * LD + x]; }),
                                          bfn<QE>([&](int t, int y) { return S.Q[t * LD + y]; }),
                                          afn([&](int x, int t) { return S.P[t * LD + x]; }),
                                          bfn<QE>([&](int t, int y) { return S.K[t * LD + y]; }),
                                      [&](int x, int y, float v) { S.dW[x * LD + y] += v; }, warp, lane);
        } else {
            {
                float a[RPT];
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const int s = rg + NG * r;
                    a[r] = S.KA[s * LD + col] + 2.f * S.gam[col] * S.R[s * LD + col];
                }
                prod_m<D, MB, NT>(a, S.P, S.W, col, rg);
#pragma unroll
                for (int r = 0; r < RPT; ++r) p.dK[(tok0 + t0 + rg + NG * r) * D + col] = a[r];
            }
            float acc[C::TR][C::TC] = {};
            outer_acc<D, MB, NT, false>(acc, S.DP, S.Q, nullptr, tid);
            outer_acc<D, MB, NT, false>(acc, S.P, S.K, nullptr, tid);
            outer_store<D, MB, NT>(S.dW, acc, 1.f, tid);
        }
        for (int j = tid; j < D; j += NT) {
            float ac = 0.f, ag = 0.f, ab = 0.f;
#pragma unroll 4
            for (int s = 0; s < MB; ++s) {
                const float du = S.R[s * LD + j];
                ac += S.DP[s * LD + j] + S.P[s * LD + j];
                ag = fmaf(2.f * du, S.gam[j] * S.Yh[s * LD + j] + S.E[s * LD + j], ag);
                ab = fmaf(2.f * S.gam[j], du, ab);
            }
            S.dc[j] += ac;
            S.dgam[j] += ag;
            S.dbet[j] += ab;
        }
        for (int s = tid; s < MB; s += NT) {
            float v = S.det[s];
            if (p.eta_gate) {
                const float sg = 1.f / (1.f + __expf(-eg[t0 + s]));
                v *= p.eta_base * sg * (1.f - sg);
            }
            p.deta[tok0 + t0 + s] = v;
        }
    }
    __syncthreads();
    bool bad = false;
    for (int q = tid; q < D * D / 4; q += NT) {
        const int j = (4 * q) / D, ii = (4 * q) % D;
        const float4 v = ld4(S.dW + j * LD + ii);
        bad |= !isfinite(v.x) || !isfinite(v.y) || !isfinite(v.z) || !isfinite(v.w);
        st4(p.dW0 + (size_t)chain * D * D + 4 * q, v);
    }
    for (int j = tid; j < D; j += NT) {
        bad |= !isfinite(S.dc[j]) || !isfinite(S.dgam[j]) || !isfinite(S.dbet[j]);
        p.dc0[(size_t)chain * D + j] = S.dc[j];
        p.dln_g[(size_t)chain * D + j] = S.dgam[j];
        p.dln_b[(size_t)chain * D + j] = S.dbet[j];
    }
    if (bad && p.status) atomicCAS(p.status, 0, TTT_ERR_NONFINITE);
}

template <typename IO, int D, int MB, int NT, int MATH = 0>
cudaError_t launch_tiled(const LinearBwdParams &p, int chains, cudaStream_t s)
{
    const size_t smem = sizeof(float) * Tiled<D, MB, NT>::kFloats;
    cudaError_t e = ensure_smem<linear_bwd_tiled_kernel<IO, D, MB, NT, MATH>>((int)smem);
    if (e != cudaSuccess) return e;
    linear_bwd_tiled_kernel<IO, D, MB, NT, MATH><<<chains, NT, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_bwd_io(const LinearBwdParams &p, int chains, cudaStream_t s, size_t smem_generic)
{
    // b = 16, d = 64 or 128: tensor cores, split precision (fp32-grade) or one tf32 product
    if (p.d == 64 && p.mb == 16)
        return p.tf32 ? launch_tiled<IO, 64, 16, 256, 2>(p, chains, s) : launch_tiled<IO, 64, 16, 256, 1>(p, chains, s);
    if (p.d == 128 && p.mb == 16)
        return p.tf32 ? launch_tiled<IO, 128, 16, 256, 2>(p, chains, s) : launch_tiled<IO, 128, 16, 256, 1>(p, chains, s);
    cudaError_t e = ensure_smem<linear_bwd_kernel<IO>>((int)smem_generic);
    if (e != cudaSuccess) return e;
    linear_bwd_kernel<IO><<<chains, kThreads, smem_generic, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t linear_bwd_smem(int d, int mb) { return sizeof(float) * bwd_smem_floats(d, mb); }

bool linear_bwd_supported(int io, int d, int mb)
{
    return (io == TTT_F32 || io == TTT_BF16) && d >= 1 && d <= 32 * kMaxPer && mb >= 1 && mb <= 64 &&
           linear_bwd_smem(d, mb) <= 227 * 1024;
}

cudaError_t linear_bwd_noalloc_scratch(void **ptr)
{
    // In host code g_noalloc_scratch names a host-side stand-in, not device
    // memory. The runtime gives its device address in the current device's
    // context; it is looked up on every call (a cheap table lookup) rather than
    // cached, so a context that was torn down and made again (cudaDeviceReset)
    // or another context on the same device never sees a stale address.
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *ptr = p;
    return cudaSuccess;
}

size_t linear_bwd_workspace_bytes(int B, int H, int T, int d, int mb)
{
    // per chain: every mini-batch's starting state (W, c), then every token's key side
    // (yh, e, g and the two row statistics of its mini-batch)
    return (size_t)B * H * ((size_t)(T / mb) * ((size_t)d * d + d) + (size_t)T * (3 * d + 2)) * sizeof(float);
}

cudaError_t launch_linear_bwd(const LinearBwdParams &p, int io, int chains, cudaStream_t s)
{
    const size_t smem = linear_bwd_smem(p.d, p.mb);
    return io == TTT_F32 ? launch_bwd_io<float>(p, chains, s, smem) : launch_bwd_io<__nv_bfloat16>(p, chains, s, smem);
}

}  // namespace ttt
