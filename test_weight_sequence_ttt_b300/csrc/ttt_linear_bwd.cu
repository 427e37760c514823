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
// batch to the first and recomputes the batch's forward from its anchor.
#include <cuda_bf16.h>

#include "ttt_internal.h"

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

}  // namespace

size_t linear_bwd_smem(int d, int mb) { return sizeof(float) * bwd_smem_floats(d, mb); }

bool linear_bwd_supported(int io, int d, int mb)
{
    return (io == TTT_F32 || io == TTT_BF16) && d >= 1 && d <= 32 * kMaxPer && mb >= 1 && mb <= 64 &&
           linear_bwd_smem(d, mb) <= 227 * 1024;
}

size_t linear_bwd_workspace_bytes(int B, int H, int T, int d, int mb)
{
    return (size_t)B * H * (size_t)(T / mb) * ((size_t)d * d + d) * sizeof(float);
}

cudaError_t launch_linear_bwd(const LinearBwdParams &p, int io, int chains, cudaStream_t s)
{
    const size_t smem = linear_bwd_smem(p.d, p.mb);
    if (io == TTT_F32) {
        cudaError_t e = ensure_smem<linear_bwd_kernel<float>>((int)smem);
        if (e != cudaSuccess) return e;
        linear_bwd_kernel<float><<<chains, kThreads, smem, s>>>(p);
    } else {
        cudaError_t e = ensure_smem<linear_bwd_kernel<__nv_bfloat16>>((int)smem);
        if (e != cudaSuccess) return e;
        linear_bwd_kernel<__nv_bfloat16><<<chains, kThreads, smem, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace ttt
