// ttt_linear_tc.cu -- TTT-Linear inner loop on tensor cores (sm_103a).
//
// Method (cited by page title and equation):
//   "Test-Time Training(TTT)과 LLM 메모리" survey page, section "TTT layer":
//     Eq. 2 update, Eq. 4 loss ||f(k; W) - v||^2, Eq. 5 output z_t = f(q_t; W_t);
//     TTT-Linear f(x) = x + LN(W x + c) (residual form from the survey's
//     reproducibility section); mini-batch b; per-token eta.
//   "End-to-End Test-Time Training for Long Context" review, section 2.3,
//     Eq. 5: every gradient of mini-batch i is taken at W_{i-1}, weight 1/b.
//
// Work decomposition. One CTA runs one (sequence, head) chain through all its
// tokens in "super-steps" of 16 tokens (one mini-batch when b = 16, 16/b
// consecutive mini-batches when b < 16). Warp roles:
//   L (1 warp)  TMA loader: Q/K/V tiles [16 tok x d] bf16 (128B-swizzled) and
//               eta into a ring of kStages stages.
//   P (1 warp)  prep: fp16 copies of the K/Q tiles; Gram fragments: causal
//               Q K^T + 1 and (b < 16) K K^T + 1.
//   W (d/16)    warp w owns rows 16w..16w+15 of W and c as fp32 mma
//               accumulators in registers for the whole sequence, and runs the
//               serial chain for those rows:
//                 Y^T = W K^T + c,  Rq^T = W Q^T + c        (mma, fp16 operands)
//                 LayerNorm statistics of every token's column of Y^T, summed
//                 over the W warps through shared memory + a named barrier
//                 G = dl/dY (LN backward, a second barrier round)
//                 A~ = -(eta/b) G^T (its own rows), then W += A~ K, c += A~ 1
//                 Yq^T = Rq^T + A~ Mq   (Mq = causal Q K^T + 1: in-batch prefix)
//   O (2)       output: Z = Q + LN(Yq), L_t = ||z_t - v_t||^2, Z stores.
//
// Per super-step the W warps synchronise with each other twice per mini-batch
// (LayerNorm forward statistics, then backward sums); everything else moves
// through mbarriers between roles, all of them bounded waits.
//
// Precision. MMA operands are fp16 (10-bit mantissa) with fp32 accumulation;
// W, c, LayerNorm statistics and gradients stay fp32. Inputs and W must stay
// inside the fp16 range (|x| < 65504); an input outside it sets TTT_ERR_RANGE.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kSS = 16;       // tokens per super-step
constexpr int kStages = 6;    // input ring depth
constexpr unsigned kFull = 0xffffffffu;
constexpr int kBarStats = 1;  // named barrier ids (0 is __syncthreads)
constexpr int kBarBwd = 2;

template <int D>
struct Cfg {
    static constexpr int MT = D / 16;                // W warps (16 rows each)
    static constexpr int NO = 2;                     // output warps
    static constexpr int TPO = kSS / NO;             // tokens per output warp
    static constexpr int LPT = 32 / TPO;             // lanes per token in an output warp
    static constexpr int FPL = D / LPT;              // features per output lane (16 or 32)
    static constexpr int kWarpL = 0, kWarpP = 1, kWarpW = 2;
    static constexpr int kWarpO = kWarpW + MT;
    static constexpr int kWarps = kWarpO + NO;
    static constexpr int kThreads = kWarps * 32;
    // stage layout (bytes); tiles first so they stay 1024-aligned
    static constexpr int kTile = 32 * D;             // 16 rows x D x 2 B
    static constexpr int kOffK = 0, kOffQ = kTile, kOffV = 2 * kTile;  // bf16, as loaded
    static constexpr int kOffKh = 3 * kTile, kOffQh = 4 * kTile;      // fp16 copies (same layout)
    static constexpr int kOffMq = 5 * kTile;
    static constexpr int kOffGk = kOffMq + 512;
    static constexpr int kOffEta = kOffGk + 512;     // 16 floats
    static constexpr int kStageBytes = ((kOffEta + 64 + 1023) / 1024) * 1024;
    static constexpr int YS = D + 4;                 // row stride (floats) of the Yq^T hand-off
    static constexpr int kOffStages = 0;
    static constexpr int kOffY = kStages * kStageBytes;            // 2 slots x [16][YS] fp32
    static constexpr int kOffRedA = kOffY + 2 * kSS * YS * 4;     // [MT][16] float2
    static constexpr int kOffRedB = kOffRedA + MT * kSS * 8;      // [MT][16] float4
    static constexpr int kOffBar = kOffRedB + MT * kSS * 16;
    static constexpr int kNumBars = 3 * kStages + 4;
    static constexpr int kSmem = kOffBar + kNumBars * 8 + 16;
    static constexpr int kSmemAlloc = kSmem + 1024;                // slack for alignment
    static_assert(FPL % 4 == 0, "output lanes hold whole 4-feature chunks");
};

// Barrier map (all in shared memory):
//   full[s]   TMA Q/K/V + cp.async eta landed in stage s      (L -> P, W, O)
//   prep[s]   P finished stage s (fp16 tiles, Grams)           (P -> W, O)
//   empty[s]  every consumer is done with stage s              (P, W, O -> L)
//   yfull/yempty[2]  Yq^T hand-off                            (W <-> O)
struct Ring {
    uint64_t *full, *prep, *empty, *yfull, *yempty;
    volatile int *flags;  // [0] abort, [1] fp16 range violation seen
};

__device__ __forceinline__ uint32_t parity_of(int use) { return (uint32_t)(use & 1); }

// Byte offset of the 16-byte chunk (row r, chunk j) of a [16 x D] 2-byte tile
// loaded by TMA with 128-byte swizzle as D/64 boxes of 64 columns.
__device__ __forceinline__ uint32_t swz(int r, int j)
{
    return (uint32_t)((j >> 3) * 2048 + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void record(int *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// Bounded wait that also gives up as soon as another warp has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *flags)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (flags[0]) return false;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void abort_chain(volatile int *flags, int *status)
{
    flags[0] = 1;
    record(status, TTT_ERR_TIMEOUT);
}

__device__ __forceinline__ void warp_arrive(uint64_t *bar, int lane)
{
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// Sum over the 8 lanes that share (lane & 3): the row axis of an mma
// accumulator tile, i.e. the feature axis of a transposed activation.
__device__ __forceinline__ float col_sum(float v)
{
    v += __shfl_xor_sync(kFull, v, 4);
    v += __shfl_xor_sync(kFull, v, 8);
    v += __shfl_xor_sync(kFull, v, 16);
    return v;
}

__device__ __forceinline__ float round_h(float v) { return __half2float(__float2half_rn(v)); }

template <int D>
__device__ __forceinline__ uint8_t *stage_ptr(uint8_t *sm, int st)
{
    return sm + Cfg<D>::kOffStages + st * Cfg<D>::kStageBytes;
}

// ------------------------------------------------------------------ L: loader
template <int D>
__device__ void role_loader(const CUtensorMap *tmQ, const CUtensorMap *tmK, const CUtensorMap *tmV,
                            const LinearParams &p, uint8_t *sm, const Ring &R, int chain, int lane,
                            int nsteps)
{
    using C = Cfg<D>;
    const int T = p.T;
    const float *eta = p.eta + (size_t)chain * T;
    if (lane == 0) {
        prefetch_tmap(tmQ);
        prefetch_tmap(tmK);
        prefetch_tmap(tmV);
    }
    int issued = 0;
    for (int i = 0; i < nsteps; ++i) {
        const int st = i % kStages;
        if (!wait_bar(&R.empty[st], parity_of(i / kStages) ^ 1u, R.flags)) {
            abort_chain(R.flags, p.status);
            break;
        }
        TTT_TRACE_AT(p, i, 14);
        uint8_t *stg = stage_ptr<D>(sm, st);
        const int t0 = i * kSS;
        float *se = reinterpret_cast<float *>(stg + C::kOffEta);
        if (lane < kSS) {
            const int t = t0 + lane;
            cp_async_4(se + lane, eta + (t < T ? t : 0), t < T ? 4u : 0u);  // zero-fill past T
        }
        cp_async_mbar_arrive_noinc(&R.full[st]);
        if (lane == 0) {
            mbar_arrive_expect_tx(&R.full[st], 3 * C::kTile);
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                tma_load_3d(stg + C::kOffK + h * 2048, tmK, &R.full[st], h * 64, t0, chain);
                tma_load_3d(stg + C::kOffQ + h * 2048, tmQ, &R.full[st], h * 64, t0, chain);
                tma_load_3d(stg + C::kOffV + h * 2048, tmV, &R.full[st], h * 64, t0, chain);
            }
        }
        issued = i + 1;
    }
    // Never leave while a copy issued here may still be landing in shared memory.
    for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        (void)mbar_wait(&R.full[i % kStages], parity_of(i / kStages));
}

// ------------------------------------------------------------------ P: prep
// Two bf16 values (one 32-bit word) -> fp16x2, round to nearest even.
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w)
{
    return pack_h2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <int D, int SUBB>
__device__ void role_prep(const LinearParams &p, uint8_t *sm, const Ring &R, int lane, int nsteps)
{
    using C = Cfg<D>;
    const int g = lane >> 2, c4 = lane & 3;
    uint32_t mag = 0;  // per-halfword max of |bf16 bits|: >= 0x4780 means |x| >= 2^16 (or inf/nan)
    const int ra = (lane & 7) + ((lane >> 3) & 1) * 8;  // A-fragment row (ldmatrix x4)
    const int rb = (lane & 7) + (lane >> 4) * 8;        // B-fragment row
    for (int i = 0; i < nsteps; ++i) {
        const int st = i % kStages;
        if (!wait_bar(&R.full[st], parity_of(i / kStages), R.flags)) {
            abort_chain(R.flags, p.status);
            return;
        }
        TTT_TRACE_AT(p, i, 12);
        uint8_t *stg = stage_ptr<D>(sm, st);
        // (1) fp16 copies of the K and Q tiles (same swizzled byte layout).
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
            const uint4 *src = reinterpret_cast<const uint4 *>(stg + (tile == 0 ? C::kOffK : C::kOffQ));
            uint4 *dst = reinterpret_cast<uint4 *>(stg + (tile == 0 ? C::kOffKh : C::kOffQh));
#pragma unroll
            for (int ch = lane; ch < 2 * D; ch += 32) {
                const uint4 x = src[ch];
                mag = __vmaxu2(mag, __vmaxu2(__vmaxu2(x.x & 0x7fff7fffu, x.y & 0x7fff7fffu),
                                             __vmaxu2(x.z & 0x7fff7fffu, x.w & 0x7fff7fffu)));
                dst[ch] = make_uint4(bf2_to_h2(x.x), bf2_to_h2(x.y), bf2_to_h2(x.z), bf2_to_h2(x.w));
            }
        }
        __syncwarp();
        // (2) Gram fragments. d*[j][r] holds (t = g + 8(r>>1), s = 8j + 2c4 + (r&1)).
        const uint32_t sK = smem_u32(stg + C::kOffKh), sQ = smem_u32(stg + C::kOffQh);
        float dq[2][4] = {}, dk[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t aq[4], bk[4];
            ldsm_x4(aq, sQ + swz(ra, 2 * ks + (lane >> 4)));
            ldsm_x4(bk, sK + swz(rb, 2 * ks + ((lane >> 3) & 1)));
            mma16816(dq[0], aq, bk[0], bk[1]);
            mma16816(dq[1], aq, bk[2], bk[3]);
            if (SUBB < 16) {
                uint32_t ak[4];
                ldsm_x4(ak, sK + swz(ra, 2 * ks + (lane >> 4)));
                mma16816(dk[0], ak, bk[0], bk[1]);
                mma16816(dk[1], ak, bk[2], bk[3]);
            }
        }
        // Causal Q K^T + 1 as B fragments (k = s, n = t) for the W warps.
        auto mq = [&](int j, int r) {
            const int t = g + 8 * (r >> 1), s = 8 * j + 2 * c4 + (r & 1);
            return s <= t ? dq[j][r] + 1.f : 0.f;
        };
        reinterpret_cast<uint4 *>(stg + C::kOffMq)[lane] =
            make_uint4(pack_h2(mq(0, 0), mq(0, 1)), pack_h2(mq(1, 0), mq(1, 1)),
                       pack_h2(mq(0, 2), mq(0, 3)), pack_h2(mq(1, 2), mq(1, 3)));
        if (SUBB < 16) {
            reinterpret_cast<uint4 *>(stg + C::kOffGk)[lane] = make_uint4(
                pack_h2(dk[0][0] + 1.f, dk[0][1] + 1.f), pack_h2(dk[1][0] + 1.f, dk[1][1] + 1.f),
                pack_h2(dk[0][2] + 1.f, dk[0][3] + 1.f), pack_h2(dk[1][2] + 1.f, dk[1][3] + 1.f));
        }
        warp_arrive(&R.prep[st], lane);
        TTT_TRACE_AT(p, i, 13);
        if (lane == 0) mbar_arrive(&R.empty[st]);
    }
    const bool range_bad = (mag & 0xffffu) >= 0x4780u || (mag >> 16) >= 0x4780u;
    if (__any_sync(kFull, range_bad) && lane == 0) {
        R.flags[1] = 1;
        record(p.status, TTT_ERR_RANGE);
    }
}

// ------------------------------------------------------------------ W: weight + chain warps
template <int D, int SUBB>
__device__ void role_weights(const LinearParams &p, uint8_t *sm, const Ring &R, int w, int chain, int bi,
                             int hi, size_t tok0, int lane, int nsteps)
{
    using C = Cfg<D>;
    constexpr int MT = C::MT, NTW = D / 8, NSUB = kSS / SUBB;
    constexpr int kNThr = MT * 32;
    const int g = lane >> 2, c4 = lane & 3;
    const int r0 = 16 * w + g, r1 = r0 + 8;
    const float *W0 = p.W0 + bi * p.w0_bstride + (long long)hi * D * D;
    const float *c0 = p.c0 + bi * p.c0_bstride + (long long)hi * D;
    float Wa[NTW][4];  // W rows r0/r1, columns 8nt + 2c4 + {0,1}
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
        const float2 a = *reinterpret_cast<const float2 *>(W0 + r0 * D + 8 * nt + 2 * c4);
        const float2 b = *reinterpret_cast<const float2 *>(W0 + r1 * D + 8 * nt + 2 * c4);
        Wa[nt][0] = a.x;
        Wa[nt][1] = a.y;
        Wa[nt][2] = b.x;
        Wa[nt][3] = b.y;
    }
    float cb[2] = {c0[r0], c0[r1]};
    const float gam[2] = {p.ln_g[hi * D + r0], p.ln_g[hi * D + r1]};
    const float bet[2] = {p.ln_b[hi * D + r0], p.ln_b[hi * D + r1]};
    const int rb = (lane & 7) + (lane >> 4) * 8;        // ldmatrix row, non-transposed B
    const int cb16 = (lane >> 3) & 1;
    const int rt = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row, transposed B
    const int ct = lane >> 4;
    const float invD = 1.f / (float)D, eps = p.eps;
    float2 *redA = reinterpret_cast<float2 *>(sm + C::kOffRedA);
    float4 *redB = reinterpret_cast<float4 *>(sm + C::kOffRedB);
    const int T = p.T;

    for (int i = 0; i < nsteps; ++i) {
        const int st = i % kStages, slot = i & 1;
        uint8_t *stg = stage_ptr<D>(sm, st);
        if (w == 0) TTT_TRACE_AT(p, i, 0);
        bool bad = !wait_bar(&R.full[st], parity_of(i / kStages), R.flags) ||
                   !wait_bar(&R.prep[st], parity_of(i / kStages), R.flags) ||
                   !wait_bar(&R.yempty[slot], parity_of(i >> 1) ^ 1u, R.flags);
        if (bad) abort_chain(R.flags, p.status);
        if (w == 0) TTT_TRACE_AT(p, i, 1);
        // Y^T = W_{i-1} K_i^T + c and Rq^T = W_{i-1} Q_i^T + c (this warp's 16 rows).
        float yk[2][4], yq[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) yk[nt][r] = yq[nt][r] = cb[r >> 1];
        if (!bad) {
            const uint32_t sK = smem_u32(stg + C::kOffKh), sQ = smem_u32(stg + C::kOffQh);
#pragma unroll
            for (int ks = 0; ks < MT; ++ks) {
                const uint32_t af[4] = {pack_h2(Wa[2 * ks][0], Wa[2 * ks][1]), pack_h2(Wa[2 * ks][2], Wa[2 * ks][3]),
                                        pack_h2(Wa[2 * ks + 1][0], Wa[2 * ks + 1][1]),
                                        pack_h2(Wa[2 * ks + 1][2], Wa[2 * ks + 1][3])};
                uint32_t bk[4], bq[4];
                ldsm_x4(bk, sK + swz(rb, 2 * ks + cb16));
                ldsm_x4(bq, sQ + swz(rb, 2 * ks + cb16));
                mma16816(yk[0], af, bk[0], bk[1]);
                mma16816(yk[1], af, bk[2], bk[3]);
                mma16816(yq[0], af, bq[0], bq[1]);
                mma16816(yq[1], af, bq[2], bq[3]);
            }
        }
        if (w == 0) TTT_TRACE_AT(p, i, 2);
        const float *se = reinterpret_cast<const float *>(stg + C::kOffEta);
        float escale[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) escale[nt][e] = -se[8 * nt + 2 * c4 + e] * (1.f / (float)SUBB);
        // K - V + beta in this warp's accumulator order: ldmatrix.trans of the
        // bf16 tiles hands each lane tokens (2c4, 2c4+1) of features g, g+8.
        float kv[2][4];
        {
            uint32_t kr[4], vr[4];
            ldsm_x4_t(kr, smem_u32(stg + C::kOffK) + swz(rb, 2 * w + cb16));
            ldsm_x4_t(vr, smem_u32(stg + C::kOffV) + swz(rb, 2 * w + cb16));
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t a = kr[2 * nt + u], b = vr[2 * nt + u];
                    kv[nt][2 * u] = bf16_bits_to_f32(a & 0xffffu) - bf16_bits_to_f32(b & 0xffffu) + bet[u];
                    kv[nt][2 * u + 1] = bf16_bits_to_f32(a >> 16) - bf16_bits_to_f32(b >> 16) + bet[u];
                }
        }
        float at[2][4] = {};   // A~ = -(eta/b) G, fp16-rounded, every column once set
        float lin[2][2] = {};  // inner loss of each column
#pragma unroll
        for (int m = 0; m < NSUB; ++m) {
            // --- LayerNorm statistics: this warp's 16 rows, then all W warps (parallel variance).
            float mw[2][2], m2w[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float mloc = col_sum(yk[nt][e] + yk[nt][e + 2]) * (1.f / 16.f);
                    const float a = yk[nt][e] - mloc, b2 = yk[nt][e + 2] - mloc;
                    mw[nt][e] = mloc;
                    m2w[nt][e] = col_sum(a * a + b2 * b2);
                }
            if (g == 0) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) redA[w * kSS + 8 * nt + 2 * c4 + e] = make_float2(mw[nt][e], m2w[nt][e]);
            }
            if (named_bar_or(kBarStats, kNThr, bad || R.flags[0] != 0)) {
                abort_chain(R.flags, p.status);
                return;  // every W warp takes this branch together
            }
            float mu[2][2], rs[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = 8 * nt + 2 * c4 + e;
                    float2 part[MT];
                    float s = 0.f;
#pragma unroll
                    for (int u = 0; u < MT; ++u) {
                        part[u] = redA[u * kSS + t];
                        s += part[u].x;
                    }
                    const float mean = s * (1.f / (float)MT);
                    float m2 = 0.f;
#pragma unroll
                    for (int u = 0; u < MT; ++u) {
                        const float dm = part[u].x - mean;
                        m2 += part[u].y + 16.f * dm * dm;
                    }
                    mu[nt][e] = mean;
                    rs[nt][e] = rsqrtf(m2 * invD + eps);
                }
            // --- LayerNorm backward sums: m1 = sum dh, m2 = sum dh*yh, l = sum E^2, dh = 2 gamma E.
            float s1[2][2], s2[2][2], sl[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float a1 = 0.f, a2 = 0.f, al = 0.f;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float yh = (yk[nt][e + 2 * u] - mu[nt][e]) * rs[nt][e];
                        const float E = gam[u] * yh + kv[nt][e + 2 * u];
                        const float dh = 2.f * gam[u] * E;
                        a1 += dh;
                        a2 += dh * yh;
                        al += E * E;
                    }
                    s1[nt][e] = col_sum(a1);
                    s2[nt][e] = col_sum(a2);
                    sl[nt][e] = col_sum(al);
                }
            if (g == 0) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        redB[w * kSS + 8 * nt + 2 * c4 + e] = make_float4(s1[nt][e], s2[nt][e], sl[nt][e], 0.f);
            }
            named_bar_sync(kBarBwd, kNThr);
            float ad[2][4];  // this mini-batch's A~ columns (zero elsewhere)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = 8 * nt + 2 * c4 + e;
                    float M1 = 0.f, M2 = 0.f, LE = 0.f;
#pragma unroll
                    for (int u = 0; u < MT; ++u) {
                        const float4 q = redB[u * kSS + t];
                        M1 += q.x;
                        M2 += q.y;
                        LE += q.z;
                    }
                    M1 *= invD;
                    M2 *= invD;
                    const bool in_m = NSUB == 1 || t / SUBB == m;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float yh = (yk[nt][e + 2 * u] - mu[nt][e]) * rs[nt][e];
                        const float E = gam[u] * yh + kv[nt][e + 2 * u];
                        const float G = rs[nt][e] * (2.f * gam[u] * E - M1 - yh * M2);
                        const float a = round_h(escale[nt][e] * G);
                        ad[nt][e + 2 * u] = in_m ? a : 0.f;
                        if (in_m) at[nt][e + 2 * u] = a;
                    }
                    if (in_m) lin[nt][e] = LE;
                }
            // Later mini-batches of this super-step see this one's update:
            // Y^T[:, t] += A~[:, s] (k_s . k_t + 1) for s in mini-batch m
            // (columns already used receive it too, harmlessly).
            if (NSUB > 1 && m + 1 < NSUB) {
                const uint4 gk = reinterpret_cast<const uint4 *>(stg + C::kOffGk)[lane];
                const uint32_t adf[4] = {pack_h2(ad[0][0], ad[0][1]), pack_h2(ad[0][2], ad[0][3]),
                                         pack_h2(ad[1][0], ad[1][1]), pack_h2(ad[1][2], ad[1][3])};
                mma16816(yk[0], adf, gk.x, gk.y);
                mma16816(yk[1], adf, gk.z, gk.w);
            }
        }
        if (w == 0) TTT_TRACE_AT(p, i, 3);
        // W += A~ K_i, c += A~ 1   (W_{i-1} -> W_i for this warp's rows)
        const uint32_t af[4] = {pack_h2(at[0][0], at[0][1]), pack_h2(at[0][2], at[0][3]),
                                pack_h2(at[1][0], at[1][1]), pack_h2(at[1][2], at[1][3])};
        {
            const uint32_t sK = smem_u32(stg + C::kOffKh);
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                uint32_t bt[4];
                ldsm_x4_t(bt, sK + swz(rt, 2 * j + ct));
                mma16816(Wa[2 * j], af, bt[0], bt[1]);
                mma16816(Wa[2 * j + 1], af, bt[2], bt[3]);
            }
        }
        float s0 = at[0][0] + at[0][1] + at[1][0] + at[1][1];
        float s1r = at[0][2] + at[0][3] + at[1][2] + at[1][3];
        s0 += __shfl_xor_sync(kFull, s0, 1);
        s0 += __shfl_xor_sync(kFull, s0, 2);
        s1r += __shfl_xor_sync(kFull, s1r, 1);
        s1r += __shfl_xor_sync(kFull, s1r, 2);
        cb[0] += s0;
        cb[1] += s1r;
        // Yq^T = Rq^T + A~ Mq (in-batch prefix of every query) -> output warps.
        {
            const uint4 mq = reinterpret_cast<const uint4 *>(stg + C::kOffMq)[lane];
            mma16816(yq[0], af, mq.x, mq.y);
            mma16816(yq[1], af, mq.z, mq.w);
        }
        float *ys = reinterpret_cast<float *>(sm + C::kOffY + slot * kSS * C::YS * 4);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r)
                ys[(8 * nt + 2 * c4 + (r & 1)) * C::YS + 16 * w + g + 8 * (r >> 1)] = yq[nt][r];
        warp_arrive(&R.yfull[slot], lane);
        if (w == 0) TTT_TRACE_AT(p, i, 4);
        if (p.inner_loss && w == 0 && g == 0) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = i * kSS + 8 * nt + 2 * c4 + e;
                    if (t < T) p.inner_loss[tok0 + t] = lin[nt][e];
                }
        }
        warp_arrive(&R.empty[st], lane);
    }
    bool badv = !isfinite(cb[0]) || !isfinite(cb[1]);
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) badv |= !isfinite(Wa[nt][r]);
    if (p.W_out) {
        float *Wo = p.W_out + (size_t)chain * D * D;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            *reinterpret_cast<float2 *>(Wo + r0 * D + 8 * nt + 2 * c4) = make_float2(Wa[nt][0], Wa[nt][1]);
            *reinterpret_cast<float2 *>(Wo + r1 * D + 8 * nt + 2 * c4) = make_float2(Wa[nt][2], Wa[nt][3]);
        }
    }
    if (p.c_out && c4 == 0) {
        p.c_out[(size_t)chain * D + r0] = cb[0];
        p.c_out[(size_t)chain * D + r1] = cb[1];
    }
    if (__any_sync(kFull, badv) && lane == 0) record(p.status, TTT_ERR_NONFINITE);
}

// ------------------------------------------------------------------ O: output warps
template <int D>
__device__ void role_output(const LinearParams &p, uint8_t *sm, const Ring &R, int o, int chain, int hi,
                            size_t tok0, int lane, int nsteps)
{
    using C = Cfg<D>;
    constexpr int LPT = C::LPT, NCH = C::FPL / 4;  // chunks of 4 features per lane
    const int tl = lane / LPT, j = lane % LPT;
    const int tloc = o * C::TPO + tl;             // token of the super-step this lane serves
    const float invD = 1.f / (float)D, eps = p.eps;
    const int T = p.T;
    float gam[NCH][4], bet[NCH][4];
#pragma unroll
    for (int k = 0; k < NCH; ++k)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int f = 4 * j + 4 * LPT * k + q;
            gam[k][q] = p.ln_g[hi * D + f];
            bet[k][q] = p.ln_b[hi * D + f];
        }
    for (int i = 0; i < nsteps; ++i) {
        const int slot = i & 1, st = i % kStages;
        uint8_t *stg = stage_ptr<D>(sm, st);
        if (o == 0) TTT_TRACE_AT(p, i, 8);
        if (!wait_bar(&R.yfull[slot], parity_of(i >> 1), R.flags) ||
            !wait_bar(&R.prep[st], parity_of(i / kStages), R.flags) ||
            !wait_bar(&R.full[st], parity_of(i / kStages), R.flags)) {
            abort_chain(R.flags, p.status);
            break;
        }
        if (o == 0) TTT_TRACE_AT(p, i, 9);
        float y[NCH][4];
        const float *ys = reinterpret_cast<const float *>(sm + C::kOffY + slot * kSS * C::YS * 4) + tloc * C::YS;
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
            const float4 v = *reinterpret_cast<const float4 *>(ys + 4 * j + 4 * LPT * k);
            y[k][0] = v.x;
            y[k][1] = v.y;
            y[k][2] = v.z;
            y[k][3] = v.w;
        }
        warp_arrive(&R.yempty[slot], lane);
        // z = q + LN(yq); L_t = ||z_t - v_t||^2
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NCH; ++k) s += (y[k][0] + y[k][1]) + (y[k][2] + y[k][3]);
#pragma unroll
        for (int x = 1; x < LPT; x <<= 1) s += __shfl_xor_sync(kFull, s, x);
        const float mu = s * invD;
        float v2 = 0.f;
#pragma unroll
        for (int k = 0; k < NCH; ++k)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float a = y[k][q] - mu;
                v2 += a * a;
            }
#pragma unroll
        for (int x = 1; x < LPT; x <<= 1) v2 += __shfl_xor_sync(kFull, v2, x);
        const float rs = rsqrtf(v2 * invD + eps);
        float l = 0.f;
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
            const int f = 4 * j + 4 * LPT * k;
            const uint32_t off = swz(tloc, f >> 3) + (f & 7) * 2;
            const uint2 qb = *reinterpret_cast<const uint2 *>(stg + C::kOffQ + off);  // bf16
            const uint2 vb = *reinterpret_cast<const uint2 *>(stg + C::kOffV + off);  // bf16
            const float qv[4] = {bf16_bits_to_f32(qb.x & 0xffffu), bf16_bits_to_f32(qb.x >> 16),
                                 bf16_bits_to_f32(qb.y & 0xffffu), bf16_bits_to_f32(qb.y >> 16)};
            const float vv[4] = {bf16_bits_to_f32(vb.x & 0xffffu), bf16_bits_to_f32(vb.x >> 16),
                                 bf16_bits_to_f32(vb.y & 0xffffu), bf16_bits_to_f32(vb.y >> 16)};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float z = qv[q] + gam[k][q] * (y[k][q] - mu) * rs + bet[k][q];
                y[k][q] = z;
                l += (z - vv[q]) * (z - vv[q]);
            }
        }
#pragma unroll
        for (int x = 1; x < LPT; x <<= 1) l += __shfl_xor_sync(kFull, l, x);
        const int t = i * kSS + tloc;
        if (t < T) {
            if (p.z_f32) {
                float *Zr = static_cast<float *>(p.Z) + (tok0 + t) * D;
#pragma unroll
                for (int k = 0; k < NCH; ++k)
                    *reinterpret_cast<float4 *>(Zr + 4 * j + 4 * LPT * k) = make_float4(y[k][0], y[k][1], y[k][2], y[k][3]);
            } else {
                __nv_bfloat16 *Zr = static_cast<__nv_bfloat16 *>(p.Z) + (tok0 + t) * D;
#pragma unroll
                for (int k = 0; k < NCH; ++k)
                    *reinterpret_cast<uint2 *>(Zr + 4 * j + 4 * LPT * k) =
                        make_uint2(pack_bf2(y[k][0], y[k][1]), pack_bf2(y[k][2], y[k][3]));
            }
            if (p.loss && j == 0) p.loss[tok0 + t] = l;
        }
        if (o == 0) TTT_TRACE_AT(p, i, 10);
        warp_arrive(&R.empty[st], lane);
    }
}

// ------------------------------------------------------------------ kernel
template <int D, int SUBB>
__global__ void __launch_bounds__(Cfg<D>::kThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const LinearParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chain = blockIdx.x;
    const int bi = chain / p.H, hi = chain % p.H;
    const int nsteps = (p.T + kSS - 1) / kSS;
    const size_t tok0 = (size_t)chain * p.T;

    Ring R;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + C::kOffBar);
    R.full = bar;
    R.prep = bar + kStages;
    R.empty = bar + 2 * kStages;
    R.yfull = bar + 3 * kStages;
    R.yempty = R.yfull + 2;
    R.flags = reinterpret_cast<volatile int *>(bar + C::kNumBars);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&R.full[s], 33);                  // expect_tx arrive + 32 cp.async arrivals
            mbar_init(&R.prep[s], 1);
            mbar_init(&R.empty[s], C::MT + C::NO + 1);  // W warps, O warps, P
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&R.yfull[j], C::MT);
            mbar_init(&R.yempty[j], C::NO);
        }
        R.flags[0] = 0;
        R.flags[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (nsteps == 0) return;

    if (warp == C::kWarpL) {
        role_loader<D>(&tmQ, &tmK, &tmV, p, sm, R, chain, lane, nsteps);
    } else if (warp == C::kWarpP) {
        role_prep<D, SUBB>(p, sm, R, lane, nsteps);
    } else if (warp < C::kWarpO) {
        role_weights<D, SUBB>(p, sm, R, warp - C::kWarpW, chain, bi, hi, tok0, lane, nsteps);
    } else {
        role_output<D>(p, sm, R, warp - C::kWarpO, chain, hi, tok0, lane, nsteps);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// [chains][T][D] bf16 viewed as a 3-D tensor; box {64, rows, 1}, 128B swizzle.
bool make_map(CUtensorMap *m, const void *base, int D, int T, int chains, int rows)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)chains};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, int SUBB>
cudaError_t launch_dsub(const LinearParams &p, int chains, cudaStream_t s)
{
    CUtensorMap mQ, mK, mV;
    if (!make_map(&mQ, p.Q, D, p.T, chains, 16) || !make_map(&mK, p.K, D, p.T, chains, 16) ||
        !make_map(&mV, p.V, D, p.T, chains, 16))
        return cudaErrorInvalidValue;
    constexpr int smem = Cfg<D>::kSmemAlloc;
    cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel<D, SUBB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    linear_tc_kernel<D, SUBB><<<chains, Cfg<D>::kThreads, smem, s>>>(mQ, mK, mV, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const LinearParams &p, int chains, cudaStream_t s)
{
    switch (p.mb) {
    case 1: return launch_dsub<D, 1>(p, chains, s);
    case 2: return launch_dsub<D, 2>(p, chains, s);
    case 4: return launch_dsub<D, 4>(p, chains, s);
    case 8: return launch_dsub<D, 8>(p, chains, s);
    case 16: return launch_dsub<D, 16>(p, chains, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool linear_tc_supported(int io, int d, int mb)
{
    return io == TTT_BF16 && (d == 64 || d == 128) && (mb == 1 || mb == 2 || mb == 4 || mb == 8 || mb == 16);
}

cudaError_t launch_linear_tc(const LinearParams &p, int chains, cudaStream_t s)
{
    if (p.d == 64) return launch_d<64>(p, chains, s);
    if (p.d == 128) return launch_d<128>(p, chains, s);
    return cudaErrorInvalidValue;
}

}  // namespace ttt
