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
//   P (1 warp)  prep: K-V+beta in the C warp's fragment order; converts the
//               K/Q tiles to fp16 in place; Gram fragments K_{i-1}K_i^T + 1,
//               causal Q_i K_i^T + 1 and (b < 16) K_i K_i^T + 1.
//   C (1 warp)  the serial chain: Y_i^T, LayerNorm forward/backward, and
//               A~_i = -(eta/b) G_i^T as an fp16 mma A-fragment.
//   T (d/16)    each owns 16 rows of W (and c) as fp32 mma accumulators in
//               registers for the whole sequence: W += A~_i K_i and the next
//               products W [K_{i+1}; Q_i]^T + c.
//   O (d/64)    output: Yq^T = W Q_i^T + c + A~_i Mq_i, Z = Q + LN(Yq),
//               L_t = ||z_t - v_t||^2, Z stored by TMA.
//
// Lookahead. Y_i = K_i W_{i-1}^T + c_{i-1} is split as
//   Y_i^T = (W_{i-2} K_i^T + c_{i-2}) + A~_{i-1} (K_{i-1} K_i^T + 1)
// so the serial chain per super-step is one 16x16xd mma group plus the
// LayerNorm, while the d x d products run one step ahead on the T warps.
// Exact in real arithmetic; it reorders rounding only.
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

template <int D>
struct Cfg {
    static constexpr int MT = D / 16;                // 16-row tiles of W / features
    static constexpr int NO = D / 64;                // output warps
    static constexpr int kWarpL = 0, kWarpP = 1, kWarpC = 2, kWarpT = 3;
    static constexpr int kWarpO = kWarpT + MT;
    static constexpr int kWarps = kWarpO + NO;
    static constexpr int kThreads = kWarps * 32;
    // stage layout (bytes); tiles first so they stay 1024-aligned
    static constexpr int kTile = 32 * D;             // 16 rows x D x 2 B
    static constexpr int kOffK = 0, kOffQ = kTile, kOffV = 2 * kTile;
    static constexpr int kOffKVD = 3 * kTile;        // MT*2 x 32 lanes x float4
    static constexpr int kOffGp = kOffKVD + MT * 2 * 512;
    static constexpr int kOffMq = kOffGp + 512;
    static constexpr int kOffGs = kOffMq + 512;      // fp32 [16][16]
    static constexpr int kOffEta = kOffGs + 1024;    // 16 floats
    static constexpr int kStageBytes = ((kOffEta + 64 + 1023) / 1024) * 1024;
    // per-step rings (2 slots)
    static constexpr int kFragF32 = MT * 2 * 512;    // S or Rq: MT x 2 ntiles x 32 lanes x 16 B
    static constexpr int kFragA = MT * 512;          // A~: MT x 32 lanes x 16 B
    static constexpr int kZStage = 32 * D;           // 2 ntiles x D/64 halves x 1 KB
    static constexpr int kOffStages = 0;
    static constexpr int kOffS = kStages * kStageBytes;
    static constexpr int kOffRq = kOffS + 2 * kFragF32;
    static constexpr int kOffA = kOffRq + 2 * kFragF32;
    static constexpr int kOffZ = kOffA + 2 * kFragA;                  // 1024-aligned
    static constexpr int kOffBar = kOffZ + 2 * kZStage;
    static constexpr int kNumBars = 3 * kStages + 12;
    static constexpr int kSmem = kOffBar + kNumBars * 8 + 16;
    static constexpr int kSmemAlloc = kSmem + 1024;                   // slack for alignment
};


// Barrier map (all in shared memory):
//   full[s]   TMA Q/K/V + cp.async eta landed in stage s      (L -> P, C, O)
//   prep[s]   P finished stage s (fp16 tiles, Grams, K-V+beta) (P -> C, T, O)
//   empty[s]  every consumer is done with stage s              (C, T, O, P -> L)
//   sfull/sempty[2]  W_{i-2} K_i^T + c for the chain warp       (T <-> C)
//   qfull/qempty[2]  W_{i-1} Q_i^T + c for the output warps     (T <-> O)
//   afull/aempty[2]  A~_i fragments                             (C <-> T, O)
struct Ring {
    uint64_t *full, *prep, *empty, *sfull, *sempty, *qfull, *qempty, *afull, *aempty;
    volatile int *flags;  // [0] abort, [1] fp16 range violation seen
};

__device__ __forceinline__ uint32_t parity_of(int use) { return (uint32_t)(use & 1); }

// Byte offset of the 16-byte chunk (row r, chunk j) of a [16 x D] 2-byte tile
// loaded by TMA with 128-byte swizzle as D/64 boxes of 64 columns.
__device__ __forceinline__ uint32_t swz(int r, int j)
{
    return (uint32_t)((j >> 3) * 2048 + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

// Byte offset inside a Z staging buffer made of (ntile, half) boxes of
// 8 rows x 128 B each (the TMA store box), 128-byte swizzled.
template <int D>
__device__ __forceinline__ uint32_t zswz(int t, int j)
{
    const int rr = t & 7;
    return (uint32_t)((((t >> 3) * (D / 64)) + (j >> 3)) * 1024 + rr * 128 + (((j & 7) ^ rr) << 4));
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

__device__ __forceinline__ float h_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu))); }
__device__ __forceinline__ float h_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }
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
template <int D, int SUBB>
__device__ void role_prep(const LinearParams &p, uint8_t *sm, const Ring &R, int hi, int lane, int nsteps)
{
    using C = Cfg<D>;
    constexpr int MT = C::MT;
    const int g = lane >> 2, c4 = lane & 3;
    float beta[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        beta[mt][0] = p.ln_b[hi * D + 16 * mt + g];
        beta[mt][1] = p.ln_b[hi * D + 16 * mt + g + 8];
    }
    bool range_bad = false;
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
        // (1) K - V + beta in the chain warp's accumulator order (from bf16).
        float4 *kvd = reinterpret_cast<float4 *>(stg + C::kOffKVD);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                float v[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int f = 16 * mt + g + 8 * (r >> 1), t = 8 * nt + 2 * c4 + (r & 1);
                    const uint32_t off = swz(t, f >> 3) + (f & 7) * 2;
                    const uint32_t kb = *reinterpret_cast<const uint16_t *>(stg + C::kOffK + off);
                    const uint32_t vb = *reinterpret_cast<const uint16_t *>(stg + C::kOffV + off);
                    v[r] = bf16_bits_to_f32(kb) - bf16_bits_to_f32(vb) + beta[mt][r >> 1];
                }
                kvd[(mt * 2 + nt) * 32 + lane] = make_float4(v[0], v[1], v[2], v[3]);
            }
        }
        __syncwarp();
        // (2) K and Q tiles: bf16 -> fp16 in place (same byte layout).
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
            uint4 *base = reinterpret_cast<uint4 *>(stg + (tile == 0 ? C::kOffK : C::kOffQ));
            for (int ch = lane; ch < 2 * D; ch += 32) {
                uint4 x = base[ch];
                uint32_t *w = reinterpret_cast<uint32_t *>(&x);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float lo = bf16_bits_to_f32(w[k] & 0xffffu), hi2 = bf16_bits_to_f32(w[k] >> 16);
                    range_bad |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi2) <= 65504.f);
                    w[k] = pack_h2(lo, hi2);
                }
                base[ch] = x;
            }
        }
        __syncwarp();
        // (3) Gram fragments. d*[j][r] holds (t = g + 8(r>>1), s = 8j + 2c4 + (r&1)).
        const uint32_t sK = smem_u32(stg + C::kOffK), sQ = smem_u32(stg + C::kOffQ);
        const uint32_t sKp = smem_u32(stage_ptr<D>(sm, (i + kStages - 1) % kStages) + C::kOffK);
        const bool has_prev = i > 0;
        float dq[2][4] = {}, dk[2][4] = {}, dp[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t aq[4], ak[4], bk[4], bp[4];
            ldsm_x4(aq, sQ + swz(ra, 2 * ks + (lane >> 4)));
            ldsm_x4(ak, sK + swz(ra, 2 * ks + (lane >> 4)));
            ldsm_x4(bk, sK + swz(rb, 2 * ks + ((lane >> 3) & 1)));
            mma16816(dq[0], aq, bk[0], bk[1]);
            mma16816(dq[1], aq, bk[2], bk[3]);
            if (SUBB < 16) {
                mma16816(dk[0], ak, bk[0], bk[1]);
                mma16816(dk[1], ak, bk[2], bk[3]);
            }
            if (has_prev) {
                ldsm_x4(bp, sKp + swz(rb, 2 * ks + ((lane >> 3) & 1)));
                mma16816(dp[0], ak, bp[0], bp[1]);
                mma16816(dp[1], ak, bp[2], bp[3]);
            }
        }
        // Causal Q K^T + 1 as B fragments (k = s, n = t) for the output warps.
        auto mq = [&](int j, int r) {
            const int t = g + 8 * (r >> 1), s = 8 * j + 2 * c4 + (r & 1);
            return s <= t ? dq[j][r] + 1.f : 0.f;
        };
        reinterpret_cast<uint4 *>(stg + C::kOffMq)[lane] =
            make_uint4(pack_h2(mq(0, 0), mq(0, 1)), pack_h2(mq(1, 0), mq(1, 1)),
                       pack_h2(mq(0, 2), mq(0, 3)), pack_h2(mq(1, 2), mq(1, 3)));
        if (has_prev) {
            reinterpret_cast<uint4 *>(stg + C::kOffGp)[lane] = make_uint4(
                pack_h2(dp[0][0] + 1.f, dp[0][1] + 1.f), pack_h2(dp[1][0] + 1.f, dp[1][1] + 1.f),
                pack_h2(dp[0][2] + 1.f, dp[0][3] + 1.f), pack_h2(dp[1][2] + 1.f, dp[1][3] + 1.f));
        }
        if (SUBB < 16) {
            float *gs = reinterpret_cast<float *>(stg + C::kOffGs);  // [s][t]
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    gs[(8 * j + 2 * c4 + (r & 1)) * 16 + g + 8 * (r >> 1)] = dk[j][r] + 1.f;
        }
        warp_arrive(&R.prep[st], lane);
        TTT_TRACE_AT(p, i, 13);
        if (has_prev) {
            fence_proxy_async();  // in-place generic writes before the next TMA refill
            warp_arrive(&R.empty[(i + kStages - 1) % kStages], lane);
        }
    }
    if (nsteps > 0) {
        fence_proxy_async();
        warp_arrive(&R.empty[(nsteps - 1) % kStages], lane);
    }
    if (__any_sync(kFull, range_bad) && lane == 0) {
        R.flags[1] = 1;
        record(p.status, TTT_ERR_RANGE);
    }
}

// ------------------------------------------------------------------ C: the serial chain
template <int D, int SUBB>
__device__ void role_chain(const LinearParams &p, uint8_t *sm, const Ring &R, int hi, size_t tok0,
                           int lane, int nsteps)
{
    using C = Cfg<D>;
    constexpr int MT = C::MT;
    constexpr int NSUB = kSS / SUBB;
    const int g = lane >> 2, c4 = lane & 3;
    const float invD = 1.f / (float)D, eps = p.eps;
    float gam[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        gam[mt][0] = p.ln_g[hi * D + 16 * mt + g];
        gam[mt][1] = p.ln_g[hi * D + 16 * mt + g + 8];
    }
    const int T = p.T;
    for (int i = 0; i < nsteps; ++i) {
        const int slot = i & 1, st = i % kStages;
        uint8_t *stg = stage_ptr<D>(sm, st);
        if (!wait_bar(&R.sfull[slot], parity_of(i >> 1), R.flags) ||
            !wait_bar(&R.prep[st], parity_of(i / kStages), R.flags) ||
            !wait_bar(&R.full[st], parity_of(i / kStages), R.flags)) {
            abort_chain(R.flags, p.status);
            return;
        }
        TTT_TRACE_AT(p, i, 0);
        // y = W_{i-2} K_i^T + c_{i-2}  (+ A~_{i-1} (K_{i-1} K_i^T + 1) below)
        float y[MT][2][4];
        const float4 *S = reinterpret_cast<const float4 *>(sm + C::kOffS + slot * C::kFragF32);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float4 v = S[(mt * 2 + nt) * 32 + lane];
                y[mt][nt][0] = v.x;
                y[mt][nt][1] = v.y;
                y[mt][nt][2] = v.z;
                y[mt][nt][3] = v.w;
            }
        if (i > 0) {
            const uint4 gp = reinterpret_cast<const uint4 *>(stg + C::kOffGp)[lane];
            const uint4 *Ap = reinterpret_cast<const uint4 *>(sm + C::kOffA + (slot ^ 1) * C::kFragA);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const uint4 a = Ap[mt * 32 + lane];
                const uint32_t af[4] = {a.x, a.y, a.z, a.w};
                mma16816(y[mt][0], af, gp.x, gp.y);
                mma16816(y[mt][1], af, gp.z, gp.w);
            }
        }
        warp_arrive(&R.sempty[slot], lane);
        const float *se = reinterpret_cast<const float *>(stg + C::kOffEta);
        float escale[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) escale[nt][e] = -se[8 * nt + 2 * c4 + e] * (1.f / (float)SUBB);
        const float4 *kvd = reinterpret_cast<const float4 *>(stg + C::kOffKVD);
        const float *gs = reinterpret_cast<const float *>(stg + C::kOffGs);
        float lin[2][2] = {};
#pragma unroll
        for (int m = 0; m < NSUB; ++m) {
            // LayerNorm statistics of every column held (only sub-step m's are used).
            float mu[2][2], rs[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float s = 0.f;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) s += y[mt][nt][e] + y[mt][nt][e + 2];
                    mu[nt][e] = col_sum(s) * invD;
                }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float s = 0.f;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        const float a = y[mt][nt][e] - mu[nt][e], b2 = y[mt][nt][e + 2] - mu[nt][e];
                        s += a * a + b2 * b2;
                    }
                    rs[nt][e] = rsqrtf(col_sum(s) * invD + eps);
                }
            // Backward sums: m1 = sum dh, m2 = sum dh*yh, l = sum E^2, dh = 2 gamma E.
            float m1[2][2] = {}, m2[2][2] = {}, le[2][2] = {};
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float4 kv = kvd[(mt * 2 + nt) * 32 + lane];
                    const float kvv[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int e = r & 1;
                        const float gm = gam[mt][r >> 1];
                        const float yh = (y[mt][nt][r] - mu[nt][e]) * rs[nt][e];
                        const float E = gm * yh + kvv[r];
                        const float dh = 2.f * gm * E;
                        m1[nt][e] += dh;
                        m2[nt][e] += dh * yh;
                        le[nt][e] += E * E;
                    }
                }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    m1[nt][e] = col_sum(m1[nt][e]) * invD;
                    m2[nt][e] = col_sum(m2[nt][e]) * invD;
                    le[nt][e] = col_sum(le[nt][e]);
                }
            // G and A~ = -(eta/b) G (rounded to fp16 once) for sub-step m's columns.
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float4 kv = kvd[(mt * 2 + nt) * 32 + lane];
                    const float kvv[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int e = r & 1;
                        const int t = 8 * nt + 2 * c4 + e;
                        if (NSUB == 1 || t / SUBB == m) {
                            const float gm = gam[mt][r >> 1];
                            const float yh = (y[mt][nt][r] - mu[nt][e]) * rs[nt][e];
                            const float E = gm * yh + kvv[r];
                            const float G = rs[nt][e] * (2.f * gm * E - m1[nt][e] - yh * m2[nt][e]);
                            y[mt][nt][r] = round_h(escale[nt][e] * G);
                        }
                    }
                }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    if (NSUB == 1 || (8 * nt + 2 * c4 + e) / SUBB == m) lin[nt][e] = le[nt][e];
            // Later mini-batches of this super-step see the update of sub-step m:
            // y[:, t] += A~[:, s] (k_s . k_t + 1) for s in sub-step m, t after it.
            if (NSUB > 1 && m + 1 < NSUB) {
#pragma unroll
                for (int ss = 0; ss < SUBB; ++ss) {
                    const int s = m * SUBB + ss;
                    const int cs = (s & 7) >> 1, nts = s >> 3, es = s & 1;
                    const float2 g0 = *reinterpret_cast<const float2 *>(gs + s * 16 + 2 * c4);
                    const float2 g1 = *reinterpret_cast<const float2 *>(gs + s * 16 + 8 + 2 * c4);
                    const float gv[2][2] = {{g0.x, g0.y}, {g1.x, g1.y}};
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const float a = __shfl_sync(kFull, y[mt][nts][es + 2 * rr], (g << 2) | cs);
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                                for (int e = 0; e < 2; ++e)
                                    if ((8 * nt + 2 * c4 + e) / SUBB > m)
                                        y[mt][nt][e + 2 * rr] = fmaf(a, gv[nt][e], y[mt][nt][e + 2 * rr]);
                        }
                }
            }
        }
        TTT_TRACE_AT(p, i, 1);
        // Publish A~_i (fp16 A-fragments: rows f, columns s).
        if (!wait_bar(&R.aempty[slot], parity_of(i >> 1) ^ 1u, R.flags)) {
            abort_chain(R.flags, p.status);
            return;
        }
        uint4 *Ab = reinterpret_cast<uint4 *>(sm + C::kOffA + slot * C::kFragA);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            Ab[mt * 32 + lane] = make_uint4(pack_h2(y[mt][0][0], y[mt][0][1]), pack_h2(y[mt][0][2], y[mt][0][3]),
                                            pack_h2(y[mt][1][0], y[mt][1][1]), pack_h2(y[mt][1][2], y[mt][1][3]));
        warp_arrive(&R.afull[slot], lane);
        TTT_TRACE_AT(p, i, 2);
        if (p.inner_loss && g == 0) {
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
}

// ------------------------------------------------------------------ T: weight warps
template <int D>
__device__ void role_weights(const LinearParams &p, uint8_t *sm, const Ring &R, int w, int chain, int bi,
                             int hi, int lane, int nsteps)
{
    using C = Cfg<D>;
    constexpr int MT = C::MT, NTW = D / 8;
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
    float cb0 = c0[r0], cb1 = c0[r1];
    const int rb = (lane & 7) + (lane >> 4) * 8;        // ldmatrix row, non-transposed B
    const int cb = (lane >> 3) & 1;
    const int rt = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row, transposed B
    const int ct = lane >> 4;

    uint32_t Af[MT][4];
    auto pack_w = [&]() {
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
            Af[ks][0] = pack_h2(Wa[2 * ks][0], Wa[2 * ks][1]);
            Af[ks][1] = pack_h2(Wa[2 * ks][2], Wa[2 * ks][3]);
            Af[ks][2] = pack_h2(Wa[2 * ks + 1][0], Wa[2 * ks + 1][1]);
            Af[ks][3] = pack_h2(Wa[2 * ks + 1][2], Wa[2 * ks + 1][3]);
        }
    };
    // out[nt] = W rows (r0, r1) x 8 tokens + c, fragment order of the chain warp
    auto rgemm = [&](uint32_t tile, float4 *dst) {
        float o[2][4] = {{cb0, cb0, cb1, cb1}, {cb0, cb0, cb1, cb1}};
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
            uint32_t bq[4];
            ldsm_x4(bq, tile + swz(rb, 2 * ks + cb));
            mma16816(o[0], Af[ks], bq[0], bq[1]);
            mma16816(o[1], Af[ks], bq[2], bq[3]);
        }
        dst[(w * 2 + 0) * 32 + lane] = make_float4(o[0][0], o[0][1], o[0][2], o[0][3]);
        dst[(w * 2 + 1) * 32 + lane] = make_float4(o[1][0], o[1][1], o[1][2], o[1][3]);
    };

    // Prologue: S_0 = W_0 K_0^T + c_0.
    if (!wait_bar(&R.prep[0], 0u, R.flags)) {
        abort_chain(R.flags, p.status);
        return;
    }
    pack_w();
    rgemm(smem_u32(stage_ptr<D>(sm, 0) + C::kOffK), reinterpret_cast<float4 *>(sm + C::kOffS));
    warp_arrive(&R.sfull[0], lane);

    for (int i = 0; i < nsteps; ++i) {
        const int st = i % kStages, slot = i & 1;
        const bool has_next = i + 1 < nsteps;
        uint8_t *stg = stage_ptr<D>(sm, st);
        if (w == 0) TTT_TRACE_AT(p, i, 3);
        bool ok = true;
        if (has_next) {
            ok = wait_bar(&R.prep[(i + 1) % kStages], parity_of((i + 1) / kStages), R.flags) &&
                 wait_bar(&R.sempty[slot ^ 1], parity_of((i + 1) >> 1) ^ 1u, R.flags);
        }
        ok = ok && wait_bar(&R.qempty[slot], parity_of(i >> 1) ^ 1u, R.flags);
        if (!ok) {
            abort_chain(R.flags, p.status);
            return;
        }
        if (w == 0) TTT_TRACE_AT(p, i, 4);
        pack_w();  // W_{start of i} as fp16 A-fragments
        if (has_next)
            rgemm(smem_u32(stage_ptr<D>(sm, (i + 1) % kStages) + C::kOffK),
                  reinterpret_cast<float4 *>(sm + C::kOffS + (slot ^ 1) * C::kFragF32));
        rgemm(smem_u32(stg + C::kOffQ), reinterpret_cast<float4 *>(sm + C::kOffRq + slot * C::kFragF32));
        __syncwarp();
        if (lane == 0) {
            if (has_next) mbar_arrive(&R.sfull[slot ^ 1]);
            mbar_arrive(&R.qfull[slot]);
        }
        if (w == 0) TTT_TRACE_AT(p, i, 5);
        // W += A~_i K_i, c += A~_i 1
        if (!wait_bar(&R.afull[slot], parity_of(i >> 1), R.flags)) {
            abort_chain(R.flags, p.status);
            return;
        }
        if (w == 0) TTT_TRACE_AT(p, i, 6);
        const uint4 a = reinterpret_cast<const uint4 *>(sm + C::kOffA + slot * C::kFragA)[w * 32 + lane];
        warp_arrive(&R.aempty[slot], lane);
        const uint32_t at[4] = {a.x, a.y, a.z, a.w};
        const uint32_t sK = smem_u32(stg + C::kOffK);
#pragma unroll
        for (int j = 0; j < MT; ++j) {
            uint32_t bt[4];
            ldsm_x4_t(bt, sK + swz(rt, 2 * j + ct));
            mma16816(Wa[2 * j], at, bt[0], bt[1]);
            mma16816(Wa[2 * j + 1], at, bt[2], bt[3]);
        }
        float s0 = h_lo(a.x) + h_hi(a.x) + h_lo(a.z) + h_hi(a.z);
        float s1 = h_lo(a.y) + h_hi(a.y) + h_lo(a.w) + h_hi(a.w);
        s0 += __shfl_xor_sync(kFull, s0, 1);
        s0 += __shfl_xor_sync(kFull, s0, 2);
        s1 += __shfl_xor_sync(kFull, s1, 1);
        s1 += __shfl_xor_sync(kFull, s1, 2);
        cb0 += s0;
        cb1 += s1;
        if (w == 0) TTT_TRACE_AT(p, i, 7);
        warp_arrive(&R.empty[st], lane);
    }
    bool bad = !isfinite(cb0) || !isfinite(cb1);
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) bad |= !isfinite(Wa[nt][r]);
    if (p.W_out) {
        float *Wo = p.W_out + (size_t)chain * D * D;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            *reinterpret_cast<float2 *>(Wo + r0 * D + 8 * nt + 2 * c4) = make_float2(Wa[nt][0], Wa[nt][1]);
            *reinterpret_cast<float2 *>(Wo + r1 * D + 8 * nt + 2 * c4) = make_float2(Wa[nt][2], Wa[nt][3]);
        }
    }
    if (p.c_out && c4 == 0) {
        p.c_out[(size_t)chain * D + r0] = cb0;
        p.c_out[(size_t)chain * D + r1] = cb1;
    }
    if (__any_sync(kFull, bad) && lane == 0) record(p.status, TTT_ERR_NONFINITE);
}

// ------------------------------------------------------------------ O: output warps
template <int D>
__device__ void role_output(const CUtensorMap *tmZ, const LinearParams &p, uint8_t *sm, const Ring &R, int o,
                            int chain, int hi, size_t tok0, int lane, int nsteps)
{
    using C = Cfg<D>;
    constexpr int MT = C::MT, NTO = 2 / C::NO;  // n-tiles (8 tokens) per output warp
    const int g = lane >> 2, c4 = lane & 3;
    const float invD = 1.f / (float)D, eps = p.eps;
    const int T = p.T;
    float gam[MT][2], bet[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            gam[mt][u] = p.ln_g[hi * D + 16 * mt + g + 8 * u];
            bet[mt][u] = p.ln_b[hi * D + 16 * mt + g + 8 * u];
        }
    if (lane == 0) prefetch_tmap(tmZ);
    for (int i = 0; i < nsteps; ++i) {
        const int slot = i & 1, st = i % kStages;
        uint8_t *stg = stage_ptr<D>(sm, st);
        float yq[MT][NTO][4];
        if (o == 0) TTT_TRACE_AT(p, i, 8);
        if (!wait_bar(&R.qfull[slot], parity_of(i >> 1), R.flags)) {
            abort_chain(R.flags, p.status);
            break;
        }
        const float4 *Rq = reinterpret_cast<const float4 *>(sm + C::kOffRq + slot * C::kFragF32);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int k = 0; k < NTO; ++k) {
                const float4 v = Rq[(mt * 2 + o * NTO + k) * 32 + lane];
                yq[mt][k][0] = v.x;
                yq[mt][k][1] = v.y;
                yq[mt][k][2] = v.z;
                yq[mt][k][3] = v.w;
            }
        warp_arrive(&R.qempty[slot], lane);
        if (o == 0) TTT_TRACE_AT(p, i, 9);
        if (!wait_bar(&R.afull[slot], parity_of(i >> 1), R.flags) ||
            !wait_bar(&R.prep[st], parity_of(i / kStages), R.flags) ||
            !wait_bar(&R.full[st], parity_of(i / kStages), R.flags)) {
            abort_chain(R.flags, p.status);
            break;
        }
        {
            const uint4 mq = reinterpret_cast<const uint4 *>(stg + C::kOffMq)[lane];
            const uint4 *Ab = reinterpret_cast<const uint4 *>(sm + C::kOffA + slot * C::kFragA);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const uint4 a = Ab[mt * 32 + lane];
                const uint32_t af[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int k = 0; k < NTO; ++k) {
                    const int nt = o * NTO + k;
                    mma16816(yq[mt][k], af, nt == 0 ? mq.x : mq.z, nt == 0 ? mq.y : mq.w);
                }
            }
        }
        warp_arrive(&R.aempty[slot], lane);
        if (o == 0) TTT_TRACE_AT(p, i, 10);
        // z = q + LN(yq); L_t = ||z_t - v_t||^2
        float L[NTO][2];
#pragma unroll
        for (int k = 0; k < NTO; ++k)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float s = 0.f;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) s += yq[mt][k][e] + yq[mt][k][e + 2];
                const float mu = col_sum(s) * invD;
                float v2 = 0.f;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const float a = yq[mt][k][e] - mu, b2 = yq[mt][k][e + 2] - mu;
                    v2 += a * a + b2 * b2;
                }
                const float rs = rsqrtf(col_sum(v2) * invD + eps);
                const int t = 8 * (o * NTO + k) + 2 * c4 + e;
                float l = 0.f;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int f = 16 * mt + g + 8 * u;
                        const uint32_t off = swz(t, f >> 3) + (f & 7) * 2;
                        const float q = __half2float(*reinterpret_cast<const __half *>(stg + C::kOffQ + off));
                        const float v = bf16_bits_to_f32(*reinterpret_cast<const uint16_t *>(stg + C::kOffV + off));
                        const float z = q + gam[mt][u] * (yq[mt][k][e + 2 * u] - mu) * rs + bet[mt][u];
                        yq[mt][k][e + 2 * u] = z;
                        l += (z - v) * (z - v);
                    }
                L[k][e] = col_sum(l);
            }
        if (p.z_f32) {
            // fp32 Z: each group of 8 lanes writes 8 consecutive features (one
            // 32-byte sector) of a token.
            float *Zf = static_cast<float *>(p.Z) + tok0 * D;
#pragma unroll
            for (int k = 0; k < NTO; ++k)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = i * kSS + 8 * (o * NTO + k) + 2 * c4 + e;
                    if (t < T) {
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                            for (int u = 0; u < 2; ++u) Zf[(size_t)t * D + 16 * mt + g + 8 * u] = yq[mt][k][e + 2 * u];
                    }
                }
        } else {
            // bf16 Z tile -> staging (transposed by stmatrix) -> TMA store.
            uint8_t *zb = sm + C::kOffZ + slot * C::kZStage;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
#pragma unroll
            for (int k = 0; k < NTO; ++k) {
                const int nt = o * NTO + k;
#pragma unroll
                for (int mp = 0; mp < MT; mp += 2) {
                    const int jm = lane >> 3;
                    const int t = 8 * nt + (lane & 7);
                    const int chunk = 2 * (mp + (jm >> 1)) + (jm & 1);
                    stsm_x4_t(smem_u32(zb + zswz<D>(t, chunk)),
                              pack_bf2(yq[mp][k][0], yq[mp][k][1]), pack_bf2(yq[mp][k][2], yq[mp][k][3]),
                              pack_bf2(yq[mp + 1][k][0], yq[mp + 1][k][1]),
                              pack_bf2(yq[mp + 1][k][2], yq[mp + 1][k][3]));
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < NTO; ++k) {
                    const int nt = o * NTO + k;
                    if (i * kSS + 8 * nt < T) {
#pragma unroll
                        for (int h = 0; h < D / 64; ++h)
                            tma_store_3d(tmZ, zb + (nt * (D / 64) + h) * 1024, h * 64, i * kSS + 8 * nt, chain);
                    }
                }
                bulk_commit();
            }
        }
        if (p.loss && g == 0) {
#pragma unroll
            for (int k = 0; k < NTO; ++k)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = i * kSS + 8 * (o * NTO + k) + 2 * c4 + e;
                    if (t < T) p.loss[tok0 + t] = L[k][e];
                }
        }
        if (o == 0) TTT_TRACE_AT(p, i, 11);
        warp_arrive(&R.empty[st], lane);
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
}

// ------------------------------------------------------------------ kernel
template <int D, int SUBB>
__global__ void __launch_bounds__(Cfg<D>::kThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmZ,
                 const LinearParams p)
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
    R.sfull = bar + 3 * kStages;
    R.sempty = R.sfull + 2;
    R.qfull = R.sfull + 4;
    R.qempty = R.sfull + 6;
    R.afull = R.sfull + 8;
    R.aempty = R.sfull + 10;
    R.flags = reinterpret_cast<volatile int *>(bar + C::kNumBars);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&R.full[s], 33);               // expect_tx arrive + 32 cp.async arrivals
            mbar_init(&R.prep[s], 1);
            mbar_init(&R.empty[s], C::MT + C::NO + 2);  // T warps, O warps, C, P
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&R.sfull[j], C::MT);
            mbar_init(&R.sempty[j], 1);
            mbar_init(&R.qfull[j], C::MT);
            mbar_init(&R.qempty[j], C::NO);
            mbar_init(&R.afull[j], 1);
            mbar_init(&R.aempty[j], C::MT + C::NO);
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
        role_prep<D, SUBB>(p, sm, R, hi, lane, nsteps);
    } else if (warp == C::kWarpC) {
        role_chain<D, SUBB>(p, sm, R, hi, tok0, lane, nsteps);
    } else if (warp < C::kWarpO) {
        role_weights<D>(p, sm, R, warp - C::kWarpT, chain, bi, hi, lane, nsteps);
    } else {
        role_output<D>(&tmZ, p, sm, R, warp - C::kWarpO, chain, hi, tok0, lane, nsteps);
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
    CUtensorMap mQ, mK, mV, mZ;
    if (!make_map(&mQ, p.Q, D, p.T, chains, 16) || !make_map(&mK, p.K, D, p.T, chains, 16) ||
        !make_map(&mV, p.V, D, p.T, chains, 16))
        return cudaErrorInvalidValue;
    if (p.z_f32)
        mZ = mQ;  // not used: fp32 Z is written with plain stores
    else if (!make_map(&mZ, p.Z, D, p.T, chains, 8))
        return cudaErrorInvalidValue;
    constexpr int smem = Cfg<D>::kSmemAlloc;
    cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel<D, SUBB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    linear_tc_kernel<D, SUBB><<<chains, Cfg<D>::kThreads, smem, s>>>(mQ, mK, mV, mZ, p);
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
