// ttt_mlp_bwd.cuh -- gradients of the TTT-MLP inner loop for outer-loop training:
// reverse mode through the mini-batch rule, fp32 (FFMA).
//
// Forward of mini-batch i, anchor (W1, c1, W2, c2) (the prefix-rule matrix form
// of Eq. 5 of the "End-to-End Test-Time Training for Long Context" review,
// section 2.3, with the output of Eq. 5 of the survey's "TTT layer" section;
// f_res(x) = W2 gelu(W1 x + c1) + c2, residual LayerNorm form):
//   Z1 = K W1^T + c1,  X2 = gelu(Z1),  Y = X2 W2^T + c2
//   G  = d l / d Y through the key LayerNorm (as for TTT-Linear)
//   P1 = G W2,  G1 = P1 * gelu'(Z1)                            (= d l / d Z1)
//   A1 = causal (eta_s/b)(q_t.k_s + 1),     Z1q = Q W1^T + c1 - A1 G1,  X2q = gelu(Z1q)
//   A2 = causal (eta_s/b)(x2q_t.x2_s + 1),  Yq = X2q W2^T + c2 - A2 G,  Z = Q + LN(Yq)
//   W1' = W1 - (1/b) G1^T diag(eta) K, c1' = c1 - (1/b) G1^T eta,
//   W2' = W2 - (1/b) G^T diag(eta) X2,  c2' = c2 - (1/b) G^T eta.
// The reverse pass, per mini-batch from the last to the first, with the carried
// gradients (dW1', dc1', dW2', dc2') of the state after it:
//   dYq  = output LayerNorm backward of dZ;   dW2 += dYq^T X2q, dc2 += sum dYq
//   DA2  = -dYq G^T (causal);  dZ1q = (dYq W2 + (DA2 eta/b) X2) * gelu'(Z1q)
//   dG   = -A2^T dYq - (eta/b) R2,  R2 = dW2' x2_s + dc2'
//   dX2  = (DA2 eta/b)^T X2q - (eta/b) dW2'^T g_s
//   DA1  = -dZ1q G1^T (causal);  dQ = dZ + dZ1q W1 + (DA1 eta/b) K
//   dK   = (DA1 eta/b)^T Q - (eta/b) dW1'^T g1_s + ...,   dG1 = -A1^T dZ1q - (eta/b) R1,  R1 = dW1' k_s + dc1'
//   deta_s = (1/b)(sum_t DA1_ts (q_t.k_s + 1) + DA2_ts (x2q_t.x2_s + 1) - g1_s.R1_s - g_s.R2_s)
//   dP1  = dG1 * gelu'(Z1),  dZ1 = dG1 * P1 * gelu''(Z1),  dG += dP1 W2^T,  dW2 += G^T dP1
//   dG -> dY through the key LayerNorm backward once more (second order, as for TTT-Linear),
//         dV = -de, dK += de
//   dX2 += dY W2,  dZ1 += dX2 * gelu'(Z1),  dK += dZ1 W1
//   dW1 += dZ1q^T Q + dZ1^T K,  dW2 += dY^T X2,  dc1 += sum(dZ1q + dZ1),  dc2 += sum dY.
//
// Two kernels. mlp_bwd_kernel<b> (b in {1, 2, 4, 8}, and 16 where the cluster
// kernel does not apply): one CTA of 512 threads per (sequence, head) chain. The
// mini-batch tiles live in shared memory; the weights do not fit beside them
// (W1, W2, dW1, dW2 are 256 KB at d = 64, h = 256), so a forward sweep writes every
// mini-batch's starting state (W1, c1, W2, c2) to the caller's workspace, the
// reverse sweep reads the anchors from there (they stay in L2), and dW1, dW2
// accumulate in the workspace. W2 and dW2 are kept there transposed, [h][d] like
// W1, so that every product with a d-wide output reads a weight column coalesced
// across the lanes and every product with an h-wide output reads one
// 16-byte-aligned weight row per thread. mlp_bwd_cluster_kernel (b = 16): the same
// steps with one chain over two CTAs, each holding half of the hidden units' weights
// in shared memory (see its own comment below).
//
// The kernels are instantiated in ttt_mlp_bwd_*.cu (several translation units,
// so that they compile in parallel) and dispatched from ttt_mlp_bwd.cu.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "ttt_internal.h"

namespace ttt {
namespace mlpb {

constexpr int kNT = 512;
constexpr int kNW = kNT / 32;
constexpr int kMaxPer = 4;  // row elements per lane of the LayerNorm rows (d <= 128)

constexpr float kGeluA = 0.7978845608028654f;  // sqrt(2 / pi)
constexpr float kGeluC = 0.044715f;

// gelu_tanh and its first and second derivatives.
__device__ __forceinline__ float gelu0(float u) { return 0.5f * u * (1.f + tanhf(kGeluA * fmaf(kGeluC * u * u, u, u))); }
__device__ __forceinline__ float gelu1(float u)
{
    const float th = tanhf(kGeluA * fmaf(kGeluC * u * u, u, u)), w1 = kGeluA * fmaf(3.f * kGeluC, u * u, 1.f);
    return 0.5f * (1.f + th) + 0.5f * u * (1.f - th * th) * w1;
}
__device__ __forceinline__ float gelu2(float u)
{
    const float th = tanhf(kGeluA * fmaf(kGeluC * u * u, u, u)), w1 = kGeluA * fmaf(3.f * kGeluC, u * u, 1.f);
    const float w2 = 6.f * kGeluA * kGeluC * u;
    return (1.f - th * th) * (w1 + 0.5f * u * (w2 - 2.f * th * w1 * w1));
}

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

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

// Floats of one mini-batch's saved key side (Z1 and P1 by CTA half, yh, e, g, and the
// two row statistics): the two-CTA kernel's forward sweep writes it, its reverse
// sweep reads it back instead of recomputing.
__host__ __device__ inline size_t mlp_bwd_saved_floats(int d, int h, int b)
{
    return 2 * (size_t)b * h + 3 * (size_t)b * d + 2 * (size_t)b;
}

__host__ __device__ inline size_t mlp_bwd_smem_floats(int d, int h, int b)
{
    return 2 * (size_t)h + 6 * (size_t)d + 13 * (size_t)b * d + 9 * (size_t)b * h + 4 * (size_t)b * b + 4 * (size_t)b;
}

struct MSmem {
    float *c1, *dc1, *c2, *dc2, *gam, *bet, *dgam, *dbet;
    float *K, *Q, *E, *DZ, *Yh, *P, *G, *DYq, *DG, *R2, *DY, *KA, *DU;  // [b][d]
    float *Z1, *X2, *P1, *G1, *Z1q, *X2q, *DG1, *DX2, *R1;             // [b][h]
    float *QK1, *QK2, *DA1, *DA2;                                       // [b][b]
    float *et, *det, *rk, *m2k;                                          // [b]
};

__device__ inline MSmem mcarve(float *sm, int d, int h, int b)
{
    MSmem s;
    float *p = sm;
    auto take = [&](size_t n) { float *q = p; p += n; return q; };
    s.c1 = take(h);
    s.dc1 = take(h);
    s.c2 = take(d);
    s.dc2 = take(d);
    s.gam = take(d);
    s.bet = take(d);
    s.dgam = take(d);
    s.dbet = take(d);
    float **bd[] = {&s.K, &s.Q, &s.E, &s.DZ, &s.Yh, &s.P, &s.G, &s.DYq, &s.DG, &s.R2, &s.DY, &s.KA, &s.DU};
    for (float **q : bd) *q = take((size_t)b * d);
    float **bh[] = {&s.Z1, &s.X2, &s.P1, &s.G1, &s.Z1q, &s.X2q, &s.DG1, &s.DX2, &s.R1};
    for (float **q : bh) *q = take((size_t)b * h);
    s.QK1 = take(b * b);
    s.QK2 = take(b * b);
    s.DA1 = take(b * b);
    s.DA2 = take(b * b);
    s.et = take(b);
    s.det = take(b);
    s.rk = take(b);
    s.m2k = take(b);
    return s;
}

// out(s, n) for the MB rows s of A and the N rows n of W (row-major, Kd columns):
// acc = sum_k A[s][k] W[n][k]; epi(s, n, acc). Each work item is one weight row
// and RB rows of A, so each weight element is read MB / RB times.
template <int MB, int RB, int UNR, typename Epi>
__device__ __forceinline__ void prod_rows_rb(const float *A, const float *W, int ldw, int N, int Kd, Epi &epi)
{
    for (int it = threadIdx.x; it < N * (MB / RB); it += kNT) {
        const int n = it % N, s0 = (it / N) * RB;
        float acc[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) acc[r] = 0.f;
        const float *w = W + (size_t)n * ldw;
#pragma unroll UNR
        for (int k = 0; k < Kd; k += 4) {
            const float4 wv = ld4(w + k);
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float4 a = ld4(A + (s0 + r) * Kd + k);
                acc[r] = fmaf(a.x, wv.x, fmaf(a.y, wv.y, fmaf(a.z, wv.z, fmaf(a.w, wv.w, acc[r]))));
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) epi(s0 + r, n, acc[r]);
    }
}

// out(s, n) = sum_j A[s][j] W[j][n] (W row-major [Kd][N]); lanes hold consecutive n.
template <int MB, int RB, int UNR, typename Epi>
__device__ __forceinline__ void prod_cols_rb(const float *A, const float *W, int ldw, int N, int Kd, Epi &epi)
{
    for (int it = threadIdx.x; it < N * (MB / RB); it += kNT) {
        const int n = it % N, s0 = (it / N) * RB;
        float acc[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) acc[r] = 0.f;
#pragma unroll UNR
        for (int j = 0; j < Kd; j += 4) {
            const float w0 = W[(size_t)j * ldw + n], w1 = W[(size_t)(j + 1) * ldw + n];
            const float w2 = W[(size_t)(j + 2) * ldw + n], w3 = W[(size_t)(j + 3) * ldw + n];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float4 a = ld4(A + (s0 + r) * Kd + j);
                acc[r] = fmaf(a.x, w0, fmaf(a.y, w1, fmaf(a.z, w2, fmaf(a.w, w3, acc[r]))));
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) epi(s0 + r, n, acc[r]);
    }
}

// Rows of A per work item: as many as keep every thread busy (at most 8).
template <int MB>
__device__ __forceinline__ int rows_per_item(int N)
{
    return (MB >= 8 && N * MB >= 8 * kNT) ? 8 : (MB >= 4 && N * MB >= 4 * kNT) ? 4 : (MB >= 2) ? 2 : 1;
}

// The products with W row-major and rows ldw floats apart (ldw = Kd for
// prod_rows, N for prod_cols unless the rows are padded). UNR is the unrolling
// of the weight loop: deep where the weights come from L2 (more loads in
// flight), shallow where they sit in shared memory (fewer registers).
template <int MB, int UNR = 8, typename Epi>
__device__ __forceinline__ void prod_rows_ld(const float *A, const float *W, int ldw, int N, int Kd, Epi epi)
{
    switch (rows_per_item<MB>(N)) {
    case 8: prod_rows_rb<MB, (MB >= 8 ? 8 : 1), UNR>(A, W, ldw, N, Kd, epi); break;
    case 4: prod_rows_rb<MB, (MB >= 4 ? 4 : 1), UNR>(A, W, ldw, N, Kd, epi); break;
    case 2: prod_rows_rb<MB, (MB >= 2 ? 2 : 1), UNR>(A, W, ldw, N, Kd, epi); break;
    default: prod_rows_rb<MB, 1, UNR>(A, W, ldw, N, Kd, epi);
    }
}

template <int MB, int UNR = 4, typename Epi>
__device__ __forceinline__ void prod_cols_ld(const float *A, const float *W, int ldw, int N, int Kd, Epi epi)
{
    switch (rows_per_item<MB>(N)) {
    case 8: prod_cols_rb<MB, (MB >= 8 ? 8 : 1), UNR>(A, W, ldw, N, Kd, epi); break;
    case 4: prod_cols_rb<MB, (MB >= 4 ? 4 : 1), UNR>(A, W, ldw, N, Kd, epi); break;
    case 2: prod_cols_rb<MB, (MB >= 2 ? 2 : 1), UNR>(A, W, ldw, N, Kd, epi); break;
    default: prod_cols_rb<MB, 1, UNR>(A, W, ldw, N, Kd, epi);
    }
}

template <int MB, typename Epi>
__device__ __forceinline__ void prod_rows(const float *A, const float *W, int N, int Kd, Epi epi)
{
    prod_rows_ld<MB, 8>(A, W, Kd, N, Kd, epi);
}

template <int MB, typename Epi>
__device__ __forceinline__ void prod_cols(const float *A, const float *W, int N, int Kd, Epi epi)
{
    prod_cols_ld<MB, 4>(A, W, N, N, Kd, epi);
}

// Outer products over the mini-batch, 4 x 4 blocks per work item: for rows
// r0 + (R/4) x and columns c0..c0+3, acc[x] = sum_s sc_s A[s][r] B[s][c] summed over
// up to three (A, B) pairs (A [MB][R], B [MB][C] in shared memory); epi(r, c0, acc).
template <int MB, typename Epi>
__device__ __forceinline__ void outer4(int R, int C, const float *A0, const float *B0, const float *A1,
                                       const float *B1, const float *A2, const float *B2, const float *sc, Epi epi)
{
    const int RQ = R / 4, CQ = C / 4;
    for (int it = threadIdx.x; it < RQ * CQ; it += kNT) {
        const int r0 = it / CQ, c0 = 4 * (it % CQ);
        float4 acc[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[x] = make_float4(0.f, 0.f, 0.f, 0.f);
        auto pair = [&](const float *A, const float *B) {
#pragma unroll 4
            for (int s = 0; s < MB; ++s) {
                const float4 bv = ld4(B + s * C + c0);
                const float f = sc ? sc[s] : 1.f;
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float a = f * A[s * R + r0 + RQ * x];
                    acc[x].x = fmaf(a, bv.x, acc[x].x);
                    acc[x].y = fmaf(a, bv.y, acc[x].y);
                    acc[x].z = fmaf(a, bv.z, acc[x].z);
                    acc[x].w = fmaf(a, bv.w, acc[x].w);
                }
            }
        };
        pair(A0, B0);
        if (A1) pair(A1, B1);
        if (A2) pair(A2, B2);
#pragma unroll
        for (int x = 0; x < 4; ++x) epi(r0 + RQ * x, c0, acc[x]);
    }
}

// out[t][s] = sum_k X[t][k] Y[s][k] + add for s <= t (causal) else 0; sign applied.
template <int MB>
__device__ __forceinline__ void gram(float *out, const float *X, const float *Y, int Kd, float add, float sign,
                                     bool causal)
{
    for (int it = threadIdx.x; it < MB * MB; it += kNT) {
        const int t = it / MB, s = it % MB;
        float acc = 0.f;
        if (!causal || s <= t) {
            acc = add;
            for (int k = 0; k < Kd; k += 4) {
                const float4 x = ld4(X + t * Kd + k), y = ld4(Y + s * Kd + k);
                acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
            }
        }
        out[it] = sign * acc;
    }
}

// Key rows: Yh holds y_s on entry; leaves yh_s in Yh, e_s in E (v_s on entry),
// g_s in G, r_s and mean(u_s*yh_s) in rk, m2k. One warp per row.
__device__ __forceinline__ void key_rows(const MSmem &S, int d, int b, float eps, int warp, int lane)
{
    const float inv_d = 1.f / (float)d;
    for (int s = warp; s < b; s += kNW) {
        float *y = S.Yh + s * d, *e = S.E + s * d;
        float mu = 0.f;
        for (int j = lane; j < d; j += 32) mu += y[j];
        mu = wsum(mu) * inv_d;
        float var = 0.f;
        for (int j = lane; j < d; j += 32) var += (y[j] - mu) * (y[j] - mu);
        const float r = rsqrtf(wsum(var) * inv_d + eps);
        float m1 = 0.f, m2 = 0.f;
        for (int j = lane; j < d; j += 32) {
            const float yh = (y[j] - mu) * r;
            const float ee = S.K[s * d + j] + S.gam[j] * yh + S.bet[j] - e[j];
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

template <typename IO, int MB>
__global__ void __launch_bounds__(kNT, 1) mlp_bwd_kernel(MlpBwdParams p)
{
    extern __shared__ __align__(16) float smm[];
    const int d = p.d, h = p.hidden, T = p.T, n = T / MB;
    const MSmem S = mcarve(smm, d, h, MB);
    const int chain = blockIdx.x;
    const int bi = chain / p.H, hi = chain % p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float inv_b = 1.f / (float)MB, inv_d = 1.f / (float)d;
    const size_t tok0 = (size_t)chain * T;
    const IO *Qg = static_cast<const IO *>(p.Q) + tok0 * d;
    const IO *Kg = static_cast<const IO *>(p.K) + tok0 * d;
    const IO *Vg = static_cast<const IO *>(p.V) + tok0 * d;
    const IO *DZg = static_cast<const IO *>(p.dZ) + tok0 * d;
    const float *eg = p.eta + tok0;
    const size_t hd = (size_t)h * d, slot = 2 * hd + h + d;
    float *ws = p.ws + (size_t)chain * (n * slot + 2 * hd);
    float *dW1 = ws + n * slot, *dW2 = dW1 + hd;  // [h][d] both (dW2 transposed)
    auto W1s = [&](int i) { return ws + (size_t)i * slot; };
    auto c1s = [&](int i) { return ws + (size_t)i * slot + hd; };
    auto W2s = [&](int i) { return ws + (size_t)i * slot + hd + h; };  // W2^T [h][d]
    auto c2s = [&](int i) { return ws + (size_t)i * slot + 2 * hd + h; };

    {
        const float *W1 = p.W1 + bi * p.w_bstride + (long long)hi * hd;
        const float *W2 = p.W2 + bi * p.w_bstride + (long long)hi * hd;
        const float *c1 = p.c1 + bi * p.c1_bstride + (long long)hi * h;
        const float *c2 = p.c2 + bi * p.c2_bstride + (long long)hi * d;
        for (size_t q = tid; q < hd; q += kNT) {
            const size_t m = q / d, j = q % d, qt = j * h + m;  // [h][d] index q <- [d][h] index qt
            W1s(0)[q] = W1[q];
            W2s(0)[q] = W2[qt];
            dW1[q] = p.dW1_n ? p.dW1_n[(size_t)chain * hd + q] : 0.f;
            dW2[q] = p.dW2_n ? p.dW2_n[(size_t)chain * hd + qt] : 0.f;
        }
        for (int j = tid; j < h; j += kNT) {
            c1s(0)[j] = c1[j];
            S.dc1[j] = p.dc1_n ? p.dc1_n[(size_t)chain * h + j] : 0.f;
        }
        for (int j = tid; j < d; j += kNT) {
            c2s(0)[j] = c2[j];
            S.dc2[j] = p.dc2_n ? p.dc2_n[(size_t)chain * d + j] : 0.f;
            S.gam[j] = p.ln_g[hi * d + j];
            S.bet[j] = p.ln_b[hi * d + j];
            S.dgam[j] = 0.f;
            S.dbet[j] = 0.f;
        }
    }
    auto load_eta = [&](int t0) {
        for (int s = tid; s < MB; s += kNT) {
            const float e = eg[t0 + s];
            S.et[s] = p.eta_gate ? p.eta_base / (1.f + __expf(-e)) : e;
        }
    };
    // The anchor's key side: Z1, X2 = gelu(Z1), Y -> key LayerNorm -> G, P1 = G W2, G1.
    auto key_side = [&](const float *W1, const float *W2) {
        prod_rows<MB>(S.K, W1, h, d, [&](int s, int m, float a) {
            const float z = a + S.c1[m];
            S.Z1[s * h + m] = z;
            S.X2[s * h + m] = gelu0(z);
        });
        __syncthreads();
        prod_cols<MB>(S.X2, W2, d, h, [&](int s, int j, float a) { S.Yh[s * d + j] = a + S.c2[j]; });
        __syncthreads();
        key_rows(S, d, MB, p.eps, warp, lane);
        __syncthreads();
        prod_rows<MB>(S.G, W2, h, d, [&](int s, int m, float a) {
            S.P1[s * h + m] = a;
            S.G1[s * h + m] = a * gelu1(S.Z1[s * h + m]);
        });
    };

    // ---- forward sweep: the starting state of every mini-batch into the workspace
    for (int i = 0; i < n; ++i) {
        const int t0 = i * MB;
        __syncthreads();
        for (int j = tid; j < h; j += kNT) S.c1[j] = c1s(i)[j];
        for (int j = tid; j < d; j += kNT) S.c2[j] = c2s(i)[j];
        for (int q = tid; q < MB * d; q += kNT) {
            S.K[q] = ldx<IO>(Kg + (size_t)t0 * d + q);
            S.E[q] = ldx<IO>(Vg + (size_t)t0 * d + q);
        }
        load_eta(t0);
        __syncthreads();
        key_side(W1s(i), W2s(i));
        __syncthreads();
        if (i + 1 < n) {
            const float *W1 = W1s(i), *W2 = W2s(i);
            float *W1n = W1s(i + 1), *W2n = W2s(i + 1);
            outer4<MB>(h, d, S.G1, S.K, nullptr, nullptr, nullptr, nullptr, S.et, [&](int m, int k, float4 a) {
                const float4 w = ld4(W1 + (size_t)m * d + k);
                *reinterpret_cast<float4 *>(W1n + (size_t)m * d + k) =
                    make_float4(w.x - a.x * inv_b, w.y - a.y * inv_b, w.z - a.z * inv_b, w.w - a.w * inv_b);
            });
            outer4<MB>(h, d, S.X2, S.G, nullptr, nullptr, nullptr, nullptr, S.et, [&](int m, int j, float4 a) {
                const float4 w = ld4(W2 + (size_t)m * d + j);
                *reinterpret_cast<float4 *>(W2n + (size_t)m * d + j) =
                    make_float4(w.x - a.x * inv_b, w.y - a.y * inv_b, w.z - a.z * inv_b, w.w - a.w * inv_b);
            });
            for (int m = tid; m < h; m += kNT) {
                float a = 0.f;
                for (int s = 0; s < MB; ++s) a = fmaf(S.et[s], S.G1[s * h + m], a);
                c1s(i + 1)[m] = S.c1[m] - a * inv_b;
            }
            for (int j = tid; j < d; j += kNT) {
                float a = 0.f;
                for (int s = 0; s < MB; ++s) a = fmaf(S.et[s], S.G[s * d + j], a);
                c2s(i + 1)[j] = S.c2[j] - a * inv_b;
            }
        }
    }

    // ---- reverse sweep
    for (int i = n - 1; i >= 0; --i) {
        const int t0 = i * MB;
        const float *W1 = W1s(i), *W2 = W2s(i);
        __syncthreads();
        for (int j = tid; j < h; j += kNT) S.c1[j] = c1s(i)[j];
        for (int j = tid; j < d; j += kNT) S.c2[j] = c2s(i)[j];
        for (int q = tid; q < MB * d; q += kNT) {
            const size_t g = (size_t)t0 * d + q;
            S.K[q] = ldx<IO>(Kg + g);
            S.Q[q] = ldx<IO>(Qg + g);
            S.E[q] = ldx<IO>(Vg + g);
            S.DZ[q] = ldx<IO>(DZg + g);
        }
        load_eta(t0);
        __syncthreads();
        key_side(W1, W2);
        prod_rows<MB>(S.Q, W1, h, d, [&](int s, int m, float a) { S.Z1q[s * h + m] = a + S.c1[m]; });
        gram<MB>(S.QK1, S.Q, S.K, d, 1.f, 1.f, false);
        __syncthreads();
        // Z1q = Q W1^T + c1 - A1 G1, X2q = gelu(Z1q)
        for (int q = tid; q < MB * h; q += kNT) {
            const int t = q / h, m = q % h;
            float a = S.Z1q[q];
            for (int s = 0; s <= t; ++s) a = fmaf(-S.et[s] * inv_b * S.QK1[t * MB + s], S.G1[s * h + m], a);
            S.Z1q[q] = a;
            S.X2q[q] = gelu0(a);
        }
        __syncthreads();
        gram<MB>(S.QK2, S.X2q, S.X2, h, 1.f, 1.f, false);
        prod_cols<MB>(S.X2q, W2, d, h, [&](int s, int j, float a) { S.P[s * d + j] = a + S.c2[j]; });
        __syncthreads();
        for (int q = tid; q < MB * d; q += kNT) {
            const int t = q / d, j = q % d;
            float a = S.P[q];
            for (int s = 0; s <= t; ++s) a = fmaf(-S.et[s] * inv_b * S.QK2[t * MB + s], S.G[s * d + j], a);
            S.P[q] = a;
        }
        __syncthreads();
        // output LayerNorm rows: ph_t into P, dYq_t
        for (int t = warp; t < MB; t += kNW) {
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
            for (int j = lane; j < d; j += 32) S.DYq[t * d + j] = r * (S.gam[j] * dz[j] - a1 - y[j] * a2);
        }
        __syncthreads();
        for (int j = tid; j < d; j += kNT) {
            float ag = 0.f, ab = 0.f;
            for (int t = 0; t < MB; ++t) {
                ag = fmaf(S.DZ[t * d + j], S.P[t * d + j], ag);
                ab += S.DZ[t * d + j];
            }
            S.dgam[j] += ag;
            S.dbet[j] += ab;
        }
        gram<MB>(S.DA2, S.DYq, S.G, d, 0.f, -1.f, true);
        prod_cols<MB>(S.X2, dW2, d, h, [&](int s, int j, float a) { S.R2[s * d + j] = a + S.dc2[j]; });
        prod_rows<MB>(S.K, dW1, h, d, [&](int s, int m, float a) { S.R1[s * h + m] = a + S.dc1[m]; });
        __syncthreads();
        // dZ1q (into Z1q), dG, the q- and dW2'-sides of dX2, deta (layer 2)
        prod_rows<MB>(S.DYq, W2, h, d, [&](int t, int m, float a) {
            for (int s = 0; s <= t; ++s) a = fmaf(S.DA2[t * MB + s] * S.et[s] * inv_b, S.X2[s * h + m], a);
            S.Z1q[t * h + m] = a * gelu1(S.Z1q[t * h + m]);
        });
        for (int q = tid; q < MB * d; q += kNT) {
            const int s = q / d, j = q % d;
            float a = 0.f;
            for (int t = s; t < MB; ++t) a = fmaf(S.QK2[t * MB + s], S.DYq[t * d + j], a);
            S.DG[q] = -S.et[s] * inv_b * (a + S.R2[q]);
        }
        prod_rows<MB>(S.G, dW2, h, d, [&](int s, int m, float a) {
            float mix = 0.f;
            for (int t = s; t < MB; ++t) mix = fmaf(S.DA2[t * MB + s], S.X2q[t * h + m], mix);
            S.DX2[s * h + m] = S.et[s] * inv_b * (mix - a);
        });
        for (int s = warp; s < MB; s += kNW) {
            float a = 0.f;
            for (int t = s + lane; t < MB; t += 32) a = fmaf(S.DA2[t * MB + s], S.QK2[t * MB + s], a);
            for (int j = lane; j < d; j += 32) a = fmaf(-S.G[s * d + j], S.R2[s * d + j], a);
            a = wsum(a);
            if (lane == 0) S.det[s] = a * inv_b;
        }
        __syncthreads();
        gram<MB>(S.DA1, S.Z1q, S.G1, h, 0.f, -1.f, true);
        __syncthreads();
        // dq_t; the q- and dW1'-sides of dk_s (KA); dG1; deta (layer 1)
        prod_cols<MB>(S.Z1q, W1, d, h, [&](int t, int k, float a) {
            a += S.DZ[t * d + k];
            for (int s = 0; s <= t; ++s) a = fmaf(S.DA1[t * MB + s] * S.et[s] * inv_b, S.K[s * d + k], a);
            p.dQ[(tok0 + t0 + t) * d + k] = a;
        });
        prod_cols<MB>(S.G1, dW1, d, h, [&](int s, int k, float a) {
            float mix = 0.f;
            for (int t = s; t < MB; ++t) mix = fmaf(S.DA1[t * MB + s], S.Q[t * d + k], mix);
            S.KA[s * d + k] = S.et[s] * inv_b * (mix - a);
        });
        for (int q = tid; q < MB * h; q += kNT) {
            const int s = q / h, m = q % h;
            float a = 0.f;
            for (int t = s; t < MB; ++t) a = fmaf(S.QK1[t * MB + s], S.Z1q[t * h + m], a);
            S.DG1[q] = -S.et[s] * inv_b * (a + S.R1[q]);
        }
        for (int s = warp; s < MB; s += kNW) {
            float a = 0.f;
            for (int t = s + lane; t < MB; t += 32) a = fmaf(S.DA1[t * MB + s], S.QK1[t * MB + s], a);
            for (int m = lane; m < h; m += 32) a = fmaf(-S.G1[s * h + m], S.R1[s * h + m], a);
            a = wsum(a);
            if (lane == 0) S.det[s] += a * inv_b;
        }
        __syncthreads();
        // through G1 = P1 * gelu'(Z1): dP1 (into DG1), the gelu'' part of dZ1 (into R1)
        for (int q = tid; q < MB * h; q += kNT) {
            const float z = S.Z1[q], g1 = S.DG1[q];
            S.R1[q] = g1 * S.P1[q] * gelu2(z);
            S.DG1[q] = g1 * gelu1(z);
        }
        __syncthreads();
        prod_cols<MB>(S.DG1, W2, d, h, [&](int s, int j, float a) { S.DG[s * d + j] += a; });
        __syncthreads();
        // through G and the key LayerNorm (second order): dY into DY, du into DU, dv
        for (int s = warp; s < MB; s += kNW) {
            const float r = S.rk[s], m2 = S.m2k[s];
            float hv[kMaxPer], yh[kMaxPer], u[kMaxPer], dyh[kMaxPer];
            float hm = 0.f, hy = 0.f, hg = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxPer; ++q) {
                const int j = lane + 32 * q;
                hv[q] = yh[q] = u[q] = 0.f;
                if (j < d) {
                    hv[q] = S.DG[s * d + j];
                    yh[q] = S.Yh[s * d + j];
                    u[q] = 2.f * S.gam[j] * S.E[s * d + j];
                    hm += hv[q];
                    hy += hv[q] * yh[q];
                    hg += hv[q] * S.G[s * d + j];
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
                    const float du = r * (hv[q] - hm - yh[q] * hy);
                    const float de = 2.f * S.gam[j] * du;
                    S.DU[s * d + j] = du;
                    p.dV[(tok0 + t0 + s) * d + j] = -de;
                    dyh[q] = S.gam[j] * de - r * (hv[q] * m2 + hy * u[q]);
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
                if (j < d) S.DY[s * d + j] = r * (dyh[q] - am - yh[q] * ay) + dsig * yh[q] * inv_d;
            }
        }
        __syncthreads();
        // dX2 += dY W2;  dZ1 = (gelu'' part) + dX2 * gelu'(Z1)  (into R1)
        prod_rows<MB>(S.DY, W2, h, d, [&](int s, int m, float a) {
            const int q = s * h + m;
            S.R1[q] += (S.DX2[q] + a) * gelu1(S.Z1[q]);
        });
        __syncthreads();
        // dk_s; dW1, dW2, dc1, dc2 carried to batch i - 1; dgamma, dbeta; deta
        prod_cols<MB>(S.R1, W1, d, h, [&](int s, int k, float a) {
            p.dK[(tok0 + t0 + s) * d + k] = a + S.KA[s * d + k] + 2.f * S.gam[k] * S.DU[s * d + k];
        });
        outer4<MB>(h, d, S.Z1q, S.Q, S.R1, S.K, nullptr, nullptr, nullptr, [&](int m, int k, float4 a) {
            float4 *o = reinterpret_cast<float4 *>(dW1 + (size_t)m * d + k);
            const float4 v = *o;
            *o = make_float4(v.x + a.x, v.y + a.y, v.z + a.z, v.w + a.w);
        });
        outer4<MB>(h, d, S.X2q, S.DYq, S.DG1, S.G, S.X2, S.DY, nullptr, [&](int m, int j, float4 a) {
            float4 *o = reinterpret_cast<float4 *>(dW2 + (size_t)m * d + j);
            const float4 v = *o;
            *o = make_float4(v.x + a.x, v.y + a.y, v.z + a.z, v.w + a.w);
        });
        for (int m = tid; m < h; m += kNT) {
            float a = 0.f;
            for (int s = 0; s < MB; ++s) a += S.Z1q[s * h + m] + S.R1[s * h + m];
            S.dc1[m] += a;
        }
        for (int j = tid; j < d; j += kNT) {
            float ac = 0.f, ag = 0.f, ab = 0.f;
            for (int s = 0; s < MB; ++s) {
                const float du = S.DU[s * d + j];
                ac += S.DYq[s * d + j] + S.DY[s * d + j];
                ag = fmaf(2.f * du, S.gam[j] * S.Yh[s * d + j] + S.E[s * d + j], ag);
                ab = fmaf(2.f * S.gam[j], du, ab);
            }
            S.dc2[j] += ac;
            S.dgam[j] += ag;
            S.dbet[j] += ab;
        }
        for (int s = tid; s < MB; s += kNT) {
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
    for (size_t q = tid; q < hd; q += kNT) {
        const size_t m = q / d, j = q % d;
        const float a = dW1[q], c = dW2[q];
        bad |= !isfinite(a) || !isfinite(c);
        p.dW1[(size_t)chain * hd + q] = a;
        p.dW2[(size_t)chain * hd + j * h + m] = c;
    }
    for (int m = tid; m < h; m += kNT) {
        bad |= !isfinite(S.dc1[m]);
        p.dc1[(size_t)chain * h + m] = S.dc1[m];
    }
    for (int j = tid; j < d; j += kNT) {
        bad |= !isfinite(S.dc2[j]) || !isfinite(S.dgam[j]) || !isfinite(S.dbet[j]);
        p.dc2[(size_t)chain * d + j] = S.dc2[j];
        p.dln_g[(size_t)chain * d + j] = S.dgam[j];
        p.dln_b[(size_t)chain * d + j] = S.dbet[j];
    }
    if (bad && p.status) atomicCAS(p.status, 0, TTT_ERR_NONFINITE);
}

// ------------------------------------------------------------------ two-CTA cluster kernel (b = 16)
//
// The same steps with one chain split over a cluster of two CTAs: CTA r owns
// the hidden units [r h/2, (r+1) h/2), so its halves of W1 and W2^T (rows of d
// floats padded to d + 4, so that float4 loads along a row are free of bank
// conflicts) fit in shared memory beside the tiles and every product reads its
// weights there. The h-wide quantities (Z1, X2, G1, dZ1q, ...) stay local. The
// d-wide sums over h (Y, Yq, R2, the dW1'-part of dK, dQ, the dP1-part of dG,
// dK) and the two Grams over h (X2q X2^T, dZ1q G1^T) are added across the pair
// through distributed shared memory: each CTA's epilogue writes its partial
// both into its own tile and into the peer's receive slot, one cluster barrier,
// then each CTA adds the peer's part to its own. Both CTAs add the same two
// operands, so the d-wide results, and all that is computed from them in both
// CTAs (the LayerNorm rows, G, dY), agree bit for bit. Receive slots alternate
// between exchanges: a slot is written again only after the peer has passed
// the next barrier, and the peer reads each slot right after the barrier that
// filled it. CTA 0 writes the token gradients and the d-wide parameter
// gradients; each CTA writes its halves of dW1, dc1, dW2. The forward sweep also
// keeps each mini-batch's key side (Z1, P1, yh, e, g and the row statistics) in the
// workspace, so the reverse sweep skips the three products, the exchange and the
// LayerNorm rows that would recompute it.
constexpr int kCB = 16;  // mini-batch size of the cluster kernel

__host__ __device__ inline size_t mlp_bwd_cluster_smem_floats(int d, int h)
{
    const size_t hh = h / 2, ldw = d + 4, b = kCB;
    const size_t xs = (2 * b * d + b > b * b + b * d) ? 2 * b * d + b : b * b + b * d;
    return 2 * hh * ldw + 2 * hh + 6 * (size_t)d + 13 * b * d + 9 * b * hh + 4 * b * b + 5 * b + 2 * xs;
}

// The 16 x 16 Gram out[t][s] = sign (sum_k X[t][k] Y[s][k] + add) for s <= t when
// causal (else 0), with one warp per row t: the lanes split k (k = lane + 32 j:
// no shared-memory bank conflicts, where one thread per entry reads 16 rows at
// one column) and reduce the row's 16 partial sums over the warp, splitting them
// as they go (16 shuffles). rout, if given, receives a copy. Kd <= 128 (callers
// with a longer row use gram).
__device__ __forceinline__ void gram_w(float *out, float *rout, const float *X, const float *Y, int Kd, float add,
                                       float sign, bool causal, int warp, int lane)
{
    constexpr int MB = 16;
    static_assert(kNW == MB, "one warp per row of the Gram");
    const int t = warp;
    float xr[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int k = lane + 32 * j;
        xr[j] = k < Kd ? X[t * Kd + k] : 0.f;
    }
    float v[MB];
#pragma unroll
    for (int r = 0; r < MB; ++r) {
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = lane + 32 * j;
            if (k < Kd) a = fmaf(xr[j], Y[r * Kd + k], a);
        }
        v[r] = a;
    }
    const int b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1, b1 = (lane >> 1) & 1;
    float v8[8], v4[4], v2[2];
#pragma unroll
    for (int q = 0; q < 8; ++q)
        v8[q] = (b4 ? v[8 + q] : v[q]) + __shfl_xor_sync(0xffffffffu, b4 ? v[q] : v[8 + q], 16);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        v4[q] = (b3 ? v8[4 + q] : v8[q]) + __shfl_xor_sync(0xffffffffu, b3 ? v8[q] : v8[4 + q], 8);
#pragma unroll
    for (int q = 0; q < 2; ++q)
        v2[q] = (b2 ? v4[2 + q] : v4[q]) + __shfl_xor_sync(0xffffffffu, b2 ? v4[q] : v4[2 + q], 4);
    float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
    v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
    const int sc = 8 * b4 + 4 * b3 + 2 * b2 + b1;  // the column this lane (and lane ^ 1) now holds
    if ((lane & 1) == 0) {
        const float r = (!causal || sc <= t) ? sign * (v1 + add) : 0.f;
        out[t * MB + sc] = r;
        if (rout) rout[t * MB + sc] = r;
    }
}

// DC, HC: d and the hidden width fixed at compile time (0: read from p). The
// fixed sizes fold the index arithmetic and each product helper's choice of work
// split, and unroll the loops whose bounds they set: for d = 64, h = 256 the
// kernel runs in about 0.7 of the time the runtime-sized one takes.
template <typename IO, int DC = 0, int HC = 0>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kNT, 1) mlp_bwd_cluster_kernel(MlpBwdParams p)
{
    constexpr int MB = kCB;
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(16) float smc[];
    const int d = DC ? DC : p.d, h = HC ? HC : p.hidden, HH = h / 2, LW = d + 4, T = p.T, n = T / MB;
    const int rank = (int)cluster.block_rank(), peer = rank ^ 1;
    const int chain = blockIdx.x / 2;
    const int bi = chain / p.H, hi = chain % p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float inv_b = 1.f / (float)MB, inv_d = 1.f / (float)d;
    const int XS = (2 * MB * d + MB > MB * MB + MB * d) ? 2 * MB * d + MB : MB * MB + MB * d;

    float *q = smc;
    auto take = [&](size_t k) { float *r = q; q += k; return r; };
    float *W1h = take((size_t)HH * LW), *W2h = take((size_t)HH * LW);  // [HH][d + 4]; W2h = rows of W2^T
    float *c1h = take(HH), *dc1h = take(HH);
    MSmem S;
    S.c1 = c1h;
    S.dc1 = dc1h;
    S.c2 = take(d);
    S.dc2 = take(d);
    S.gam = take(d);
    S.bet = take(d);
    S.dgam = take(d);
    S.dbet = take(d);
    float **bd[] = {&S.K, &S.Q, &S.E, &S.DZ, &S.Yh, &S.P, &S.G, &S.DYq, &S.DG, &S.R2, &S.DY, &S.KA, &S.DU};
    for (float **x : bd) *x = take((size_t)MB * d);
    float **bh[] = {&S.Z1, &S.X2, &S.P1, &S.G1, &S.Z1q, &S.X2q, &S.DG1, &S.DX2, &S.R1};
    for (float **x : bh) *x = take((size_t)MB * HH);
    S.QK1 = take(MB * MB);
    S.QK2 = take(MB * MB);
    S.DA1 = take(MB * MB);
    S.DA2 = take(MB * MB);
    S.et = take(MB);
    S.det = take(MB);
    S.rk = take(MB);
    S.m2k = take(MB);
    float *dpart = take(MB);           // this CTA's part of -g1_s.R1_s (deta, layer 1)
    float *RX = take(2 * (size_t)XS);  // receive slots
    int xk = 0;                        // exchanges so far (slot = xk & 1)
    auto recv = [&]() { return RX + (xk & 1) * XS; };
    auto remote = [&]() { return cluster.map_shared_rank(RX + (xk & 1) * XS, peer); };

    const size_t tok0 = (size_t)chain * T;
    const IO *Qg = static_cast<const IO *>(p.Q) + tok0 * d;
    const IO *Kg = static_cast<const IO *>(p.K) + tok0 * d;
    const IO *Vg = static_cast<const IO *>(p.V) + tok0 * d;
    const IO *DZg = static_cast<const IO *>(p.dZ) + tok0 * d;
    const float *eg = p.eta + tok0;
    const size_t hd = (size_t)h * d, slot = 2 * hd + h + d, r0 = (size_t)rank * HH;
    const size_t SV = mlp_bwd_saved_floats(d, h, MB);
    float *ws = p.ws + (size_t)chain * (n * slot + 2 * hd + n * SV);
    float *dW1h = ws + n * slot + r0 * d, *dW2h = ws + n * slot + hd + r0 * d;  // this CTA's rows
    // saved key side of mini-batch i: Z1 [2][MB][HH] and P1 [2][MB][HH] by CTA, then yh, e, g
    // [MB][d] and r, mean(u yh) [MB]
    auto Svs = [&](int i) { return ws + n * slot + 2 * hd + (size_t)i * SV; };
    auto W1s = [&](int i) { return ws + (size_t)i * slot + r0 * d; };
    auto c1s = [&](int i) { return ws + (size_t)i * slot + hd + r0; };
    auto W2s = [&](int i) { return ws + (size_t)i * slot + hd + h + r0 * d; };
    auto c2s = [&](int i) { return ws + (size_t)i * slot + 2 * hd + h; };

    {
        const float *W1 = p.W1 + bi * p.w_bstride + (long long)hi * hd;
        const float *W2 = p.W2 + bi * p.w_bstride + (long long)hi * hd;
        const float *c1 = p.c1 + bi * p.c1_bstride + (long long)hi * h;
        const float *c2 = p.c2 + bi * p.c2_bstride + (long long)hi * d;
        for (int x = tid; x < HH * d; x += kNT) {
            const int m = x / d, j = x % d;
            const size_t gm = r0 + m;
            W1h[m * LW + j] = W1[gm * d + j];
            W2h[m * LW + j] = W2[(size_t)j * h + gm];
            dW1h[x] = p.dW1_n ? p.dW1_n[(size_t)chain * hd + gm * d + j] : 0.f;
            dW2h[x] = p.dW2_n ? p.dW2_n[(size_t)chain * hd + (size_t)j * h + gm] : 0.f;
        }
        for (int m = tid; m < HH; m += kNT) {
            c1h[m] = c1[r0 + m];
            dc1h[m] = p.dc1_n ? p.dc1_n[(size_t)chain * h + r0 + m] : 0.f;
        }
        for (int j = tid; j < d; j += kNT) {
            S.c2[j] = c2[j];
            S.dc2[j] = p.dc2_n ? p.dc2_n[(size_t)chain * d + j] : 0.f;
            S.gam[j] = p.ln_g[hi * d + j];
            S.bet[j] = p.ln_b[hi * d + j];
            S.dgam[j] = 0.f;
            S.dbet[j] = 0.f;
        }
    }
    auto load_eta = [&](int t0) {
        for (int s = tid; s < MB; s += kNT) {
            const float e = eg[t0 + s];
            S.et[s] = p.eta_gate ? p.eta_base / (1.f + __expf(-e)) : e;
        }
    };
    // Ask L2 for the 128-byte lines of [a, a + bytes), the threads splitting the
    // lines. The forward sweep does this for the next mini-batch's tiles, the
    // reverse sweep for the mini-batch before the current one: its starting
    // state and kept key side were written long before and left L2, and its
    // loads then find them there.
    auto pf = [&](const void *a, size_t bytes) {
        const char *c = static_cast<const char *>(a);
        for (size_t o = (size_t)tid * 128; o < bytes; o += (size_t)kNT * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(c + o));
    };
    auto prefetch_rev = [&](int i) {  // what reverse step i loads from global memory
        const size_t t0 = (size_t)i * MB;
        pf(W1s(i), (size_t)HH * d * 4);
        pf(W2s(i), (size_t)HH * d * 4);
        pf(c1s(i), (size_t)HH * 4);
        pf(c2s(i), (size_t)d * 4);
        const float *sv = Svs(i);
        pf(sv + (size_t)rank * MB * HH, (size_t)MB * HH * 4);
        pf(sv + (size_t)(2 + rank) * MB * HH, (size_t)MB * HH * 4);
        pf(sv + (size_t)4 * MB * HH, ((size_t)3 * MB * d + 2 * MB) * 4);
        pf(Kg + t0 * d, (size_t)MB * d * sizeof(IO));
        pf(Qg + t0 * d, (size_t)MB * d * sizeof(IO));
        pf(DZg + t0 * d, (size_t)MB * d * sizeof(IO));
        pf(eg + t0, MB * 4);
    };
    // Y = X2 W2^T + c2 summed over both halves into Yh (the key side's only exchange).
    auto key_side = [&]() {
        prod_rows_ld<MB, 2>(S.K, W1h, LW, HH, d, [&](int s, int m, float a) {
            const float z = a + c1h[m];
            S.Z1[s * HH + m] = z;
            S.X2[s * HH + m] = gelu0(z);
        });
        __syncthreads();
        {
            float *rm = remote();
            prod_cols_ld<MB, 2>(S.X2, W2h, LW, d, HH, [&](int s, int j, float a) {
                S.Yh[s * d + j] = a;
                rm[s * d + j] = a;
            });
        }
        cluster.sync();
        {
            const float *rv = recv();
            for (int x = tid; x < MB * d; x += kNT) S.Yh[x] = (S.Yh[x] + rv[x]) + S.c2[x % d];
            ++xk;
        }
        __syncthreads();
        key_rows(S, d, MB, p.eps, warp, lane);
        __syncthreads();
        prod_rows_ld<MB, 2>(S.G, W2h, LW, HH, d, [&](int s, int m, float a) {
            S.P1[s * HH + m] = a;
            S.G1[s * HH + m] = a * gelu1(S.Z1[s * HH + m]);
        });
    };

    // ---- forward sweep
    for (int i = 0; i < n; ++i) {
        const int t0 = i * MB;
        __syncthreads();
        {
            float *w1 = W1s(i), *w2 = W2s(i);
            for (int x = tid; x < HH * d / 4; x += kNT) {
                const int m = (4 * x) / d, j = (4 * x) % d;
                *reinterpret_cast<float4 *>(w1 + 4 * x) = ld4(W1h + m * LW + j);
                *reinterpret_cast<float4 *>(w2 + 4 * x) = ld4(W2h + m * LW + j);
            }
            for (int m = tid; m < HH; m += kNT) c1s(i)[m] = c1h[m];
            if (rank == 0)
                for (int j = tid; j < d; j += kNT) c2s(i)[j] = S.c2[j];
        }
        for (int x = tid; x < MB * d; x += kNT) {
            S.K[x] = ldx<IO>(Kg + (size_t)t0 * d + x);
            S.E[x] = ldx<IO>(Vg + (size_t)t0 * d + x);
        }
        load_eta(t0);
        if (i + 1 < n) {  // the next mini-batch's tiles into L2
            pf(Kg + (size_t)(t0 + MB) * d, (size_t)MB * d * sizeof(IO));
            pf(Vg + (size_t)(t0 + MB) * d, (size_t)MB * d * sizeof(IO));
            pf(eg + t0 + MB, MB * 4);
        }
        __syncthreads();
        key_side();
        __syncthreads();
        {
            float *sv = Svs(i);
            float *z = sv + (size_t)rank * MB * HH, *pp = sv + (size_t)(2 + rank) * MB * HH;
            for (int x = tid; x < MB * HH / 4; x += kNT) {
                st4(z + 4 * x, ld4(S.Z1 + 4 * x));
                st4(pp + 4 * x, ld4(S.P1 + 4 * x));
            }
            if (rank == 0) {
                float *yd = sv + (size_t)4 * MB * HH;
                for (int x = tid; x < MB * d / 4; x += kNT) {
                    st4(yd + 4 * x, ld4(S.Yh + 4 * x));
                    st4(yd + MB * d + 4 * x, ld4(S.E + 4 * x));
                    st4(yd + 2 * MB * d + 4 * x, ld4(S.G + 4 * x));
                }
                for (int x = tid; x < MB; x += kNT) {
                    yd[3 * MB * d + x] = S.rk[x];
                    yd[3 * MB * d + MB + x] = S.m2k[x];
                }
            }
        }
        outer4<MB>(HH, d, S.G1, S.K, nullptr, nullptr, nullptr, nullptr, S.et, [&](int m, int k, float4 a) {
            float *w = W1h + m * LW + k;
            w[0] -= a.x * inv_b;
            w[1] -= a.y * inv_b;
            w[2] -= a.z * inv_b;
            w[3] -= a.w * inv_b;
        });
        outer4<MB>(HH, d, S.X2, S.G, nullptr, nullptr, nullptr, nullptr, S.et, [&](int m, int j, float4 a) {
            float *w = W2h + m * LW + j;
            w[0] -= a.x * inv_b;
            w[1] -= a.y * inv_b;
            w[2] -= a.z * inv_b;
            w[3] -= a.w * inv_b;
        });
        for (int m = tid; m < HH; m += kNT) {
            float a = 0.f;
            for (int s = 0; s < MB; ++s) a = fmaf(S.et[s], S.G1[s * HH + m], a);
            c1h[m] -= a * inv_b;
        }
        for (int j = tid; j < d; j += kNT) {
            float a = 0.f;
            for (int s = 0; s < MB; ++s) a = fmaf(S.et[s], S.G[s * d + j], a);
            S.c2[j] -= a * inv_b;
        }
    }

    // ---- reverse sweep
    for (int i = n - 1; i >= 0; --i) {
        const int t0 = i * MB;
        __syncthreads();
        {
            const float *w1 = W1s(i), *w2 = W2s(i);
            for (int x = tid; x < HH * d / 4; x += kNT) {
                const int m = (4 * x) / d, j = (4 * x) % d;
                *reinterpret_cast<float4 *>(W1h + m * LW + j) = ld4(w1 + 4 * x);
                *reinterpret_cast<float4 *>(W2h + m * LW + j) = ld4(w2 + 4 * x);
            }
            for (int m = tid; m < HH; m += kNT) c1h[m] = c1s(i)[m];
            for (int j = tid; j < d; j += kNT) S.c2[j] = c2s(i)[j];
        }
        for (int x = tid; x < MB * d; x += kNT) {
            const size_t g = (size_t)t0 * d + x;
            S.K[x] = ldx<IO>(Kg + g);
            S.Q[x] = ldx<IO>(Qg + g);
            S.DZ[x] = ldx<IO>(DZg + g);
        }
        load_eta(t0);
        {
            // the key side of this mini-batch, as the forward sweep left it
            const float *sv = Svs(i);
            const float *z = sv + (size_t)rank * MB * HH, *pp = sv + (size_t)(2 + rank) * MB * HH;
            const float *yd = sv + (size_t)4 * MB * HH;
            for (int x = tid; x < MB * HH / 4; x += kNT) {
                const float4 zz = ld4(z + 4 * x), pv = ld4(pp + 4 * x);
                st4(S.Z1 + 4 * x, zz);
                st4(S.P1 + 4 * x, pv);
                st4(S.X2 + 4 * x, make_float4(gelu0(zz.x), gelu0(zz.y), gelu0(zz.z), gelu0(zz.w)));
                st4(S.G1 + 4 * x, make_float4(pv.x * gelu1(zz.x), pv.y * gelu1(zz.y), pv.z * gelu1(zz.z),
                                              pv.w * gelu1(zz.w)));
            }
            for (int x = tid; x < MB * d / 4; x += kNT) {
                st4(S.Yh + 4 * x, ld4(yd + 4 * x));
                st4(S.E + 4 * x, ld4(yd + MB * d + 4 * x));
                st4(S.G + 4 * x, ld4(yd + 2 * MB * d + 4 * x));
            }
            for (int x = tid; x < MB; x += kNT) {
                S.rk[x] = yd[3 * MB * d + x];
                S.m2k[x] = yd[3 * MB * d + MB + x];
            }
        }
        if (i > 0) prefetch_rev(i - 1);
        __syncthreads();
        prod_rows_ld<MB, 2>(S.Q, W1h, LW, HH, d, [&](int s, int m, float a) { S.Z1q[s * HH + m] = a + c1h[m]; });
        if (d <= 128)
            gram_w(S.QK1, nullptr, S.Q, S.K, d, 1.f, 1.f, false, warp, lane);
        else
            gram<MB>(S.QK1, S.Q, S.K, d, 1.f, 1.f, false);
        __syncthreads();
        for (int x = tid; x < MB * HH; x += kNT) {
            const int t = x / HH, m = x % HH;
            float a = S.Z1q[x];
            for (int s = 0; s <= t; ++s) a = fmaf(-S.et[s] * inv_b * S.QK1[t * MB + s], S.G1[s * HH + m], a);
            S.Z1q[x] = a;
            S.X2q[x] = gelu0(a);
        }
        __syncthreads();
        // exchange: the X2q X2^T Gram (partial over h, at 0) and X2q W2^T (at MB*MB)
        {
            float *rm = remote();
            if (HH <= 128) {
                gram_w(S.QK2, rm, S.X2q, S.X2, HH, 0.f, 1.f, false, warp, lane);
            } else {
                for (int it = tid; it < MB * MB; it += kNT) {
                    const int t = it / MB, s = it % MB;
                    float acc = 0.f;
                    for (int k = 0; k < HH; k += 4) {
                        const float4 x = ld4(S.X2q + t * HH + k), y = ld4(S.X2 + s * HH + k);
                        acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
                    }
                    S.QK2[it] = acc;
                    rm[it] = acc;
                }
            }
            prod_cols_ld<MB, 2>(S.X2q, W2h, LW, d, HH, [&](int s, int j, float a) {
                S.P[s * d + j] = a;
                rm[MB * MB + s * d + j] = a;
            });
        }
        cluster.sync();
        {
            const float *rv = recv();
            for (int it = tid; it < MB * MB; it += kNT) S.QK2[it] = (S.QK2[it] + rv[it]) + 1.f;
            for (int x = tid; x < MB * d; x += kNT) S.P[x] = (S.P[x] + rv[MB * MB + x]) + S.c2[x % d];
            ++xk;
        }
        __syncthreads();
        for (int x = tid; x < MB * d; x += kNT) {
            const int t = x / d, j = x % d;
            float a = S.P[x];
            for (int s = 0; s <= t; ++s) a = fmaf(-S.et[s] * inv_b * S.QK2[t * MB + s], S.G[s * d + j], a);
            S.P[x] = a;
        }
        __syncthreads();
        // output LayerNorm rows (both CTAs): ph_t into P, dYq_t
        for (int t = warp; t < MB; t += kNW) {
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
            for (int j = lane; j < d; j += 32) S.DYq[t * d + j] = r * (S.gam[j] * dz[j] - a1 - y[j] * a2);
        }
        __syncthreads();
        for (int j = tid; j < d; j += kNT) {
            float ag = 0.f, ab = 0.f;
            for (int t = 0; t < MB; ++t) {
                ag = fmaf(S.DZ[t * d + j], S.P[t * d + j], ag);
                ab += S.DZ[t * d + j];
            }
            S.dgam[j] += ag;
            S.dbet[j] += ab;
        }
        if (d <= 128)
            gram_w(S.DA2, nullptr, S.DYq, S.G, d, 0.f, -1.f, true, warp, lane);
        else
            gram<MB>(S.DA2, S.DYq, S.G, d, 0.f, -1.f, true);
        prod_rows_ld<MB>(S.K, dW1h, d, HH, d, [&](int s, int m, float a) { S.R1[s * HH + m] = a + dc1h[m]; });
        {
            float *rm = remote();
            prod_cols_ld<MB>(S.X2, dW2h, d, d, HH, [&](int s, int j, float a) {
                S.R2[s * d + j] = a;
                rm[s * d + j] = a;
            });
        }
        cluster.sync();
        {
            const float *rv = recv();
            for (int x = tid; x < MB * d; x += kNT) S.R2[x] = (S.R2[x] + rv[x]) + S.dc2[x % d];
            ++xk;
        }
        __syncthreads();
        // dZ1q (into Z1q), dG, the q- and dW2'-sides of dX2, deta (layer 2)
        prod_rows_ld<MB, 2>(S.DYq, W2h, LW, HH, d, [&](int t, int m, float a) {
            for (int s = 0; s <= t; ++s) a = fmaf(S.DA2[t * MB + s] * S.et[s] * inv_b, S.X2[s * HH + m], a);
            S.Z1q[t * HH + m] = a * gelu1(S.Z1q[t * HH + m]);
        });
        for (int x = tid; x < MB * d; x += kNT) {
            const int s = x / d, j = x % d;
            float a = 0.f;
            for (int t = s; t < MB; ++t) a = fmaf(S.QK2[t * MB + s], S.DYq[t * d + j], a);
            S.DG[x] = -S.et[s] * inv_b * (a + S.R2[x]);
        }
        prod_rows_ld<MB>(S.G, dW2h, d, HH, d, [&](int s, int m, float a) {
            float mix = 0.f;
            for (int t = s; t < MB; ++t) mix = fmaf(S.DA2[t * MB + s], S.X2q[t * HH + m], mix);
            S.DX2[s * HH + m] = S.et[s] * inv_b * (mix - a);
        });
        for (int s = warp; s < MB; s += kNW) {
            float a = 0.f;
            for (int t = s + lane; t < MB; t += 32) a = fmaf(S.DA2[t * MB + s], S.QK2[t * MB + s], a);
            for (int j = lane; j < d; j += 32) a = fmaf(-S.G[s * d + j], S.R2[s * d + j], a);
            a = wsum(a);
            if (lane == 0) S.det[s] = a * inv_b;
        }
        __syncthreads();
        // exchange: the dZ1q G1^T Gram (partial over h)
        {
            float *rm = remote();
            if (HH <= 128) {
                gram_w(S.DA1, rm, S.Z1q, S.G1, HH, 0.f, 1.f, true, warp, lane);
            } else {
                for (int it = tid; it < MB * MB; it += kNT) {
                    const int t = it / MB, s = it % MB;
                    float acc = 0.f;
                    if (s <= t)
                        for (int k = 0; k < HH; k += 4) {
                            const float4 x = ld4(S.Z1q + t * HH + k), y = ld4(S.G1 + s * HH + k);
                            acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
                        }
                    S.DA1[it] = acc;
                    rm[it] = acc;
                }
            }
        }
        cluster.sync();
        {
            const float *rv = recv();
            for (int it = tid; it < MB * MB; it += kNT) S.DA1[it] = -(S.DA1[it] + rv[it]);
            ++xk;
        }
        __syncthreads();
        // exchange: dZ1q W1 (dQ, at 0), G1 dW1' (the dW1'-part of dK, at MB d) and -g1.R1 (deta,
        // at 2 MB d), each partial over h; dG1 is local
        {
            float *rm = remote();
            prod_cols_ld<MB, 2>(S.Z1q, W1h, LW, d, HH, [&](int t, int k, float a) {
                S.DY[t * d + k] = a;  // DY is free until the second-order rows
                rm[t * d + k] = a;
            });
            prod_cols_ld<MB>(S.G1, dW1h, d, d, HH, [&](int s, int k, float a) {
                S.KA[s * d + k] = a;
                rm[MB * d + s * d + k] = a;
            });
            for (int x = tid; x < MB * HH; x += kNT) {
                const int s = x / HH, m = x % HH;
                float a = 0.f;
                for (int t = s; t < MB; ++t) a = fmaf(S.QK1[t * MB + s], S.Z1q[t * HH + m], a);
                S.DG1[x] = -S.et[s] * inv_b * (a + S.R1[x]);
            }
            for (int s = warp; s < MB; s += kNW) {
                float a = 0.f;
                for (int m = lane; m < HH; m += 32) a = fmaf(-S.G1[s * HH + m], S.R1[s * HH + m], a);
                a = wsum(a);
                if (lane == 0) {
                    dpart[s] = a;
                    rm[2 * MB * d + s] = a;
                }
            }
        }
        cluster.sync();
        {
            const float *rv = recv();
            for (int x = tid; x < MB * d; x += kNT) {
                const int t = x / d, k = x % d;
                float a = (S.DY[x] + rv[x]) + S.DZ[x];
                for (int s = 0; s <= t; ++s) a = fmaf(S.DA1[t * MB + s] * S.et[s] * inv_b, S.K[s * d + k], a);
                if (rank == 0) p.dQ[(tok0 + t0 + t) * d + k] = a;
            }
            for (int x = tid; x < MB * d; x += kNT) {
                const int s = x / d, k = x % d;
                float mix = 0.f;
                for (int t = s; t < MB; ++t) mix = fmaf(S.DA1[t * MB + s], S.Q[t * d + k], mix);
                S.KA[x] = S.et[s] * inv_b * (mix - (S.KA[x] + rv[MB * d + x]));
            }
            for (int s = warp; s < MB; s += kNW) {
                float a = 0.f;
                for (int t = s + lane; t < MB; t += 32) a = fmaf(S.DA1[t * MB + s], S.QK1[t * MB + s], a);
                a = wsum(a);
                if (lane == 0) S.det[s] += (a + (dpart[s] + rv[2 * MB * d + s])) * inv_b;
            }
            ++xk;
        }
        __syncthreads();
        // through G1 = P1 * gelu'(Z1): dP1 (into DG1), the gelu'' part of dZ1 (into R1)
        for (int x = tid; x < MB * HH; x += kNT) {
            const float z = S.Z1[x], g1 = S.DG1[x];
            S.R1[x] = g1 * S.P1[x] * gelu2(z);
            S.DG1[x] = g1 * gelu1(z);
        }
        __syncthreads();
        // exchange: dP1 W2^T (the dP1-part of dG), partial over h
        {
            float *rm = remote();
            prod_cols_ld<MB, 2>(S.DG1, W2h, LW, d, HH, [&](int s, int j, float a) {
                S.DY[s * d + j] = a;
                rm[s * d + j] = a;
            });
        }
        cluster.sync();
        {
            const float *rv = recv();
            for (int x = tid; x < MB * d; x += kNT) S.DG[x] += S.DY[x] + rv[x];
            ++xk;
        }
        __syncthreads();
        // through G and the key LayerNorm (second order, both CTAs): dY into DY, du into DU, dv
        for (int s = warp; s < MB; s += kNW) {
            const float r = S.rk[s], m2 = S.m2k[s];
            float hv[kMaxPer], yh[kMaxPer], u[kMaxPer], dyh[kMaxPer];
            float hm = 0.f, hy = 0.f, hg = 0.f;
#pragma unroll
            for (int e = 0; e < kMaxPer; ++e) {
                const int j = lane + 32 * e;
                hv[e] = yh[e] = u[e] = 0.f;
                if (j < d) {
                    hv[e] = S.DG[s * d + j];
                    yh[e] = S.Yh[s * d + j];
                    u[e] = 2.f * S.gam[j] * S.E[s * d + j];
                    hm += hv[e];
                    hy += hv[e] * yh[e];
                    hg += hv[e] * S.G[s * d + j];
                }
            }
            hm = wsum(hm) * inv_d;
            hy = wsum(hy) * inv_d;
            hg = wsum(hg);
            float am = 0.f, ay = 0.f;
#pragma unroll
            for (int e = 0; e < kMaxPer; ++e) {
                const int j = lane + 32 * e;
                dyh[e] = 0.f;
                if (j < d) {
                    const float du = r * (hv[e] - hm - yh[e] * hy);
                    const float de = 2.f * S.gam[j] * du;
                    S.DU[s * d + j] = du;
                    if (rank == 0) p.dV[(tok0 + t0 + s) * d + j] = -de;
                    dyh[e] = S.gam[j] * de - r * (hv[e] * m2 + hy * u[e]);
                    am += dyh[e];
                    ay += dyh[e] * yh[e];
                }
            }
            am = wsum(am) * inv_d;
            ay = wsum(ay) * inv_d;
            const float dsig = -r * hg;
#pragma unroll
            for (int e = 0; e < kMaxPer; ++e) {
                const int j = lane + 32 * e;
                if (j < d) S.DY[s * d + j] = r * (dyh[e] - am - yh[e] * ay) + dsig * yh[e] * inv_d;
            }
        }
        __syncthreads();
        // dX2 += dY W2;  dZ1 = (gelu'' part) + dX2 * gelu'(Z1)  (into R1)
        prod_rows_ld<MB, 2>(S.DY, W2h, LW, HH, d, [&](int s, int m, float a) {
            const int x = s * HH + m;
            S.R1[x] += (S.DX2[x] + a) * gelu1(S.Z1[x]);
        });
        __syncthreads();
        // exchange: dZ1 W1 (the rest of dK), partial over h
        {
            float *rm = remote();
            prod_cols_ld<MB, 2>(S.R1, W1h, LW, d, HH, [&](int s, int k, float a) {
                S.DG[s * d + k] = a;  // DG is no longer needed
                rm[s * d + k] = a;
            });
        }
        cluster.sync();
        {
            const float *rv = recv();
            if (rank == 0)
                for (int x = tid; x < MB * d; x += kNT) {
                    const int s = x / d, k = x % d;
                    p.dK[(tok0 + t0 + s) * d + k] = (S.DG[x] + rv[x]) + S.KA[x] + 2.f * S.gam[k] * S.DU[x];
                }
            ++xk;
        }
        // this CTA's rows of dW1, dW2 (transposed) carried to batch i - 1; dc1, dc2; dgamma, dbeta; deta
        outer4<MB>(HH, d, S.Z1q, S.Q, S.R1, S.K, nullptr, nullptr, nullptr, [&](int m, int k, float4 a) {
            float4 *o = reinterpret_cast<float4 *>(dW1h + (size_t)m * d + k);
            const float4 v = *o;
            *o = make_float4(v.x + a.x, v.y + a.y, v.z + a.z, v.w + a.w);
        });
        outer4<MB>(HH, d, S.X2q, S.DYq, S.DG1, S.G, S.X2, S.DY, nullptr, [&](int m, int j, float4 a) {
            float4 *o = reinterpret_cast<float4 *>(dW2h + (size_t)m * d + j);
            const float4 v = *o;
            *o = make_float4(v.x + a.x, v.y + a.y, v.z + a.z, v.w + a.w);
        });
        for (int m = tid; m < HH; m += kNT) {
            float a = 0.f;
            for (int s = 0; s < MB; ++s) a += S.Z1q[s * HH + m] + S.R1[s * HH + m];
            dc1h[m] += a;
        }
        for (int j = tid; j < d; j += kNT) {
            float ac = 0.f, ag = 0.f, ab = 0.f;
            for (int s = 0; s < MB; ++s) {
                const float du = S.DU[s * d + j];
                ac += S.DYq[s * d + j] + S.DY[s * d + j];
                ag = fmaf(2.f * du, S.gam[j] * S.Yh[s * d + j] + S.E[s * d + j], ag);
                ab = fmaf(2.f * S.gam[j], du, ab);
            }
            S.dc2[j] += ac;
            S.dgam[j] += ag;
            S.dbet[j] += ab;
        }
        if (rank == 0)
            for (int s = tid; s < MB; s += kNT) {
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
    for (int x = tid; x < HH * d; x += kNT) {
        const int m = x / d, j = x % d;
        const float a = dW1h[x], c = dW2h[x];
        bad |= !isfinite(a) || !isfinite(c);
        p.dW1[(size_t)chain * hd + (r0 + m) * d + j] = a;
        p.dW2[(size_t)chain * hd + (size_t)j * h + r0 + m] = c;
    }
    for (int m = tid; m < HH; m += kNT) {
        bad |= !isfinite(dc1h[m]);
        p.dc1[(size_t)chain * h + r0 + m] = dc1h[m];
    }
    if (rank == 0)
        for (int j = tid; j < d; j += kNT) {
            bad |= !isfinite(S.dc2[j]) || !isfinite(S.dgam[j]) || !isfinite(S.dbet[j]);
            p.dc2[(size_t)chain * d + j] = S.dc2[j];
            p.dln_g[(size_t)chain * d + j] = S.dgam[j];
            p.dln_b[(size_t)chain * d + j] = S.dbet[j];
        }
    if (bad && p.status) atomicCAS(p.status, 0, TTT_ERR_NONFINITE);
    cluster.sync();  // neither CTA leaves while the other may still address its shared memory
}

template <typename IO>
cudaError_t launch_cluster(const MlpBwdParams &p, int chains, cudaStream_t s)
{
    const size_t smem = sizeof(float) * mlp_bwd_cluster_smem_floats(p.d, p.hidden);
    if (p.d == 64 && p.hidden == 256) {  // the TTT-MLP shape of d = 64 (hidden 4d), compiled for it
        cudaError_t e = ensure_smem<mlp_bwd_cluster_kernel<IO, 64, 256>>((int)smem);
        if (e != cudaSuccess) return e;
        mlp_bwd_cluster_kernel<IO, 64, 256><<<2 * chains, kNT, smem, s>>>(p);
        return cudaGetLastError();
    }
    cudaError_t e = ensure_smem<mlp_bwd_cluster_kernel<IO>>((int)smem);
    if (e != cudaSuccess) return e;
    mlp_bwd_cluster_kernel<IO><<<2 * chains, kNT, smem, s>>>(p);
    return cudaGetLastError();
}

inline bool cluster_ok(int d, int h, int mb)
{
    return mb == kCB && h % 8 == 0 && d % 4 == 0 && sizeof(float) * mlp_bwd_cluster_smem_floats(d, h) <= 227 * 1024;
}

template <typename IO, int MB>
cudaError_t launch_mb(const MlpBwdParams &p, int chains, cudaStream_t s)
{
    const size_t smem = sizeof(float) * mlp_bwd_smem_floats(p.d, p.hidden, MB);
    cudaError_t e = ensure_smem<mlp_bwd_kernel<IO, MB>>((int)smem);
    if (e != cudaSuccess) return e;
    mlp_bwd_kernel<IO, MB><<<chains, kNT, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mlpb
}  // namespace ttt
