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
// consecutive mini-batches when b < 16, a share of one mini-batch when b is
// 32 to 1024: see role_weights_mb2 / role_weights_mb). Warp roles:
//   L (1 warp)  TMA loader: Q/K/V tiles [16 tok x d] bf16 (128B-swizzled) and
//               eta into a ring of 6 stages.
//               Two stages behind its loads it also applies the learning-rate
//               gate (eta_gate) and writes, for d = 64, the per-token scalars
//               (the LayerNorm shift u0.k + mean(c0) and the sums
//               sum_f gamma_f kv_f, sum_f kv_f^2 with kv = k - v + beta), for
//               d = 128 the fp16 copies of the K/Q tiles.
//   P (1 warp)  prep: for d = 64 the fp16 copies of the K/Q tiles, for d = 128
//               the per-token scalars; Gram fragments (causal Q_i K_i^T + 1,
//               K_{i-1} K_i^T + 1 and, for b < 16, K_i K_i^T + 1).
//   W (d/16)    warp w owns rows 16w..16w+15 of W and c as fp32 mma
//               accumulators in registers for the whole sequence, and runs the
//               serial chain for those rows.
//   O (2)       output: Z = Q + LN(Yq), L_t = ||z_t - v_t||^2, Z stores.
//
// The serial chain of one super-step i (W warps) is
//   LayerNorm forward + backward of Y_i^T (one cross-warp reduction round per
//   mini-batch) -> A~_i = -(eta/b) G_i^T -> Y_{i+1}^T = S_{i+1} + A~_i Kx_i
// where S_{i+1} = W_{i-1} K_{i+1}^T + c_{i-1} and Rq_i = W_{i-1} Q_i^T + c_{i-1}
// are computed while the reduction round is in flight, and Kx_i = K_i K_{i+1}^T
// + 1. Exact in real arithmetic (W_i = W_{i-1} + A~_i K_i); it reorders rounding
// only. Off the chain: W += A~_i K_i, c += A~_i 1, Yq_i^T = Rq_i + A~_i Mq_i.
//
// One reduction round. The feature mean of Y is invariant under the update
// (the LayerNorm gradient sums to zero over features, so the column sums of W
// and the sum of c never change), so sh_t = u0.k_t + mean(c0), with u0 the
// feature mean of W_0's rows, is the token's LN mean up to rounding drift. Each
// W warp sums, over its rows, d = y - sh: d, d^2, gamma^2 d, gamma^2 d^2 and
// gamma kv d; the five sums of the W warps add up (split-phase mbarrier) and give
// the mean, variance and the two LayerNorm-backward means in closed form.
//
// Chain/weight split (d = 64; d = 128 with b < 16). The chain above runs on its own warps (C, d/16
// of them, rows 16w..16w+15 of Y^T) that do nothing else: partial sums, one
// named-barrier reduction round, G and A~, the 16-wide correction. Separate
// weight warps (T) hold W and c, apply W += A~ K, and compute S_{i+2},
// Rq_{i+1} and Yq_i. A~ and S cross between the two groups through shared
// memory and alternating producer/consumer named barriers, so the chain warps
// never wait on an mbarrier. No warp of either group leaves early: after a
// failed wait a T warp keeps running in step (results discarded, status set).
// At d = 128 the split form has 20 warps at 96 registers a thread (some
// spilled). It runs for b < 16, where a super-step holds 16/b LayerNorm rounds
// and the chain warps, free of the weight products, shorten each round. At
// b = 16 (one round per super-step) the W warps of the merged kernel do both
// jobs, which measured faster.
//
// Precision. MMA operands are fp16 (10-bit mantissa) with fp32 accumulation;
// W, c, LayerNorm statistics and gradients stay fp32. Inputs and W must stay
// inside the fp16 range (|x| < 65504); an input outside it sets TTT_ERR_RANGE.
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace ttt {
namespace {

using namespace tc;

template <int D>
struct Cfg {
    static constexpr int kStages = 6;  // input ring depth (eight measured slower at d = 64)
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
    // The query tiles; the key tiles stand in for them when the queries are the keys.
    __device__ static int offQ(const LinearParams &p) { return p.q_is_k ? kOffK : kOffQ; }
    __device__ static int offQh(const LinearParams &p) { return p.q_is_k ? kOffKh : kOffQh; }
    static constexpr int kOffMq = 5 * kTile;         // fp16 B fragments, 32 lanes x 16 B each
    static constexpr int kOffGk = kOffMq + 512;
    static constexpr int kOffKx = kOffGk + 512;
    static constexpr int kOffEta = kOffKx + 512;     // 16 floats each:
    static constexpr int kOffSh = kOffEta + 64;      //   LayerNorm shift
    static constexpr int kOffPk = kOffSh + 64;       //   sum_f gamma_f kv_f
    static constexpr int kOffQk = kOffPk + 64;       //   sum_f kv_f^2
    static constexpr int kOffKxA = kOffQk + 64;      // K_{i-1} K_i^T + 1 and K_i K_i^T + 1 as fp16
    static constexpr int kOffGkA = kOffKxA + 512;    //   A fragments (rows t of step i)
    static constexpr int kStageBytes = ((kOffGkA + 512 + 1023) / 1024) * 1024;
    static constexpr int YS = D + 4;                 // row stride (floats) of the Yq^T hand-off
    static constexpr int kOffStages = 0;
    static constexpr int kOffY = kStages * kStageBytes;            // 2 slots x [16][YS] fp32
    static constexpr int kOffRedX = kOffY + 2 * kSS * YS * 4;     // 2 bufs x [MT][16] float4
    static constexpr int kOffRedY = kOffRedX + 2 * MT * kSS * 16; // 2 bufs x [MT][16] float
    static constexpr int kOffCst = kOffRedY + 2 * MT * kSS * 4;   // u0, gamma, beta: 3 x D floats
    // chain/weight split (D = 64): hand-off rings between the chain (C) and weight (T) warps
    static constexpr int kOffAR = kOffCst + 3 * D * 4;            // 2 slots x [MT][32 lanes] A~ fragments
    static constexpr int SRS = 20;                                // row stride (floats) of an S block [16 t][16 f]
    static constexpr int kOffSR = kOffAR + 2 * MT * 512;          // 2 slots x [MT][16][SRS] S blocks
    // cluster kernel: ring of A~ blocks the chain CTA sends to the output CTA
    static constexpr int kNA = 4;                                 // ring slots
    static constexpr int kOffAR1 = kOffSR + 2 * MT * 16 * SRS * 4;  // kNA slots x [MT][32 lanes] uint4
    static constexpr int kOffBar = kOffAR1 + kNA * MT * 512;
    static constexpr int kSplitWarpC = 2, kSplitWarpT = 2 + MT, kSplitWarpO = 2 + 2 * MT;
    static constexpr int kSplitWarps = kSplitWarpO + NO;
    static constexpr int kSplitThreads = kSplitWarps * 32;
    static constexpr int kNumBars = 3 * kStages + 6 + 2 * kNA;  // + afull[kNA], aempty[kNA] (cluster kernel)
    static constexpr int kSmem = kOffBar + kNumBars * 8 + 16;
    static constexpr int kSmemAlloc = kSmem + 1024;                // slack for alignment
    static_assert(FPL % 4 == 0, "output lanes hold whole 4-feature chunks");
};

// Barrier map (all in shared memory):
//   full[s]   TMA Q/K/V + cp.async eta landed in stage s      (L -> P, W, O)
//   prep[s]   P finished stage s (fp16 tiles, Grams, sums)     (P -> W, O)
//   empty[s]  every consumer is done with stage s              (P, W, O -> L)
//   yfull/yempty[2]  Yq^T hand-off                            (W <-> O)
//   red[2]    the W warps' partial LayerNorm sums of one round (W -> W)
//   afull[k]  A~ of a step landed in ring slot k (cluster kernel, output CTA)
//   aempty[k] the output CTA is done with slot k     (cluster kernel, chain CTA)
struct Ring {
    uint64_t *full, *prep, *empty, *yfull, *yempty, *red;
    uint64_t *afull, *aempty;
    volatile int *flags;  // [0] abort, [1] fp16 range violation seen
};

template <int D>
__device__ __forceinline__ uint8_t *stage_ptr(uint8_t *sm, int st)
{
    return sm + Cfg<D>::kOffStages + st * Cfg<D>::kStageBytes;
}

// ------------------------------------------------------------------ per-token LayerNorm scalars
// For d = 64 the loader warp computes them (two stages behind its loads);
// for d = 128 the prep warp does, because a loader with 64 features per lane
// to sum would fall behind on the loads.
template <int D>
constexpr bool kSumsInLoader = D == 64;
// For d = 128 the loader makes the fp16 copies of the K/Q tiles instead (two
// stages behind its loads), and the prep warp forms its Grams from the bf16
// tiles, which bf16 represents exactly.
template <int D>
constexpr bool kCopiesInLoader = D == 128;
template <int D>
constexpr bool kLoaderPrep = kSumsInLoader<D> || kCopiesInLoader<D>;  // the loader also arrives on prep[]
static_assert(kLoaderPrep<64> && kLoaderPrep<128>, "the loader applies the learning-rate gate");

// fp16 copies of a stage's K and Q tiles (same swizzled byte layout; no Q copy
// when the queries are the keys). All loads are issued before any store.
template <int D>
__device__ __forceinline__ void fp16_copies(uint8_t *stg, bool q_is_k, int lane, uint32_t &mag)
{
    using C = Cfg<D>;
    constexpr int NCH = 2 * D / 32;  // 16-byte chunks per lane per tile
    const uint4 *sk = reinterpret_cast<const uint4 *>(stg + C::kOffK);
    const uint4 *sq = reinterpret_cast<const uint4 *>(stg + C::kOffQ);
    uint4 xk[NCH], xq[NCH];
#pragma unroll
    for (int k = 0; k < NCH; ++k) xk[k] = sk[lane + 32 * k];
    if (!q_is_k) {
#pragma unroll
        for (int k = 0; k < NCH; ++k) xq[k] = sq[lane + 32 * k];
    }
    auto conv = [&](const uint4 &x) {
        mag = __vmaxu2(mag, __vmaxu2(__vmaxu2(x.x & 0x7fff7fffu, x.y & 0x7fff7fffu),
                                     __vmaxu2(x.z & 0x7fff7fffu, x.w & 0x7fff7fffu)));
        return make_uint4(bf2_to_h2(x.x), bf2_to_h2(x.y), bf2_to_h2(x.z), bf2_to_h2(x.w));
    };
    uint4 *dk = reinterpret_cast<uint4 *>(stg + C::kOffKh);
    uint4 *dq = reinterpret_cast<uint4 *>(stg + C::kOffQh);
#pragma unroll
    for (int k = 0; k < NCH; ++k) dk[lane + 32 * k] = conv(xk[k]);
    if (!q_is_k) {
#pragma unroll
        for (int k = 0; k < NCH; ++k) dq[lane + 32 * k] = conv(xq[k]);
    }
}

// Chain constants into shared memory: u0 = feature mean of W_0's rows, gamma,
// beta; returns mean(c0) (all lanes). W_0 is read row-contiguously in float4s
// with every load of a lane independent, so the whole matrix is in flight at
// once instead of one dependent round trip per row.
template <int D>
__device__ float chain_consts(const LinearParams &p, uint8_t *sm, int bi, int hi, int lane)
{
    using C = Cfg<D>;
    constexpr int Q4 = D / 4;              // float4s per row
    constexpr int RSTEP = 32 / Q4;         // rows covered by one pass of the warp (2 for d = 64, 1 for 128)
    float *cu = reinterpret_cast<float *>(sm + C::kOffCst), *cg = cu + D, *cbt = cg + D;
    const float4 *W4 = reinterpret_cast<const float4 *>(p.W0 + bi * p.w0_bstride + (long long)hi * D * D);
    const float *c0 = p.c0 + bi * p.c0_bstride + (long long)hi * D;
    const int q = lane % Q4, r0 = lane / Q4;  // this lane's column group and first row
    float4 acc[4] = {};
#pragma unroll 16
    for (int f = r0, k = 0; f < D; f += RSTEP, ++k) {
        const float4 v = W4[f * Q4 + q];
        acc[k & 3].x += v.x;
        acc[k & 3].y += v.y;
        acc[k & 3].z += v.z;
        acc[k & 3].w += v.w;
    }
    float4 t = make_float4((acc[0].x + acc[1].x) + (acc[2].x + acc[3].x), (acc[0].y + acc[1].y) + (acc[2].y + acc[3].y),
                           (acc[0].z + acc[1].z) + (acc[2].z + acc[3].z), (acc[0].w + acc[1].w) + (acc[2].w + acc[3].w));
    if (RSTEP == 2) {  // lanes q and q + 16 summed alternate rows
        t.x += __shfl_xor_sync(kFull, t.x, 16);
        t.y += __shfl_xor_sync(kFull, t.y, 16);
        t.z += __shfl_xor_sync(kFull, t.z, 16);
        t.w += __shfl_xor_sync(kFull, t.w, 16);
    }
    if (r0 == 0) {
        const float s = 1.f / (float)D;
        reinterpret_cast<float4 *>(cu)[q] = make_float4(t.x * s, t.y * s, t.z * s, t.w * s);
    }
    float cmean = 0.f;
#pragma unroll
    for (int qq = 0; qq < D / 32; ++qq) {
        const int j = lane + 32 * qq;
        cg[j] = p.ln_g[hi * D + j];
        cbt[j] = p.ln_b[hi * D + j];
        cmean += c0[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cmean += __shfl_xor_sync(kFull, cmean, o);
    __syncwarp();
    return cmean * (1.f / (float)D);
}

// Per-token scalars of one stage (16 tokens; lane pair per token, half the
// features each): the LayerNorm shift sh_t = u0 . k_t + mean(c0),
// sum_f gamma_f kv_f and sum_f kv_f^2 with kv = k - v + beta.
template <int D>
__device__ void token_sums(uint8_t *stg, const uint8_t *sm, float cmean, int lane)
{
    using C = Cfg<D>;
    const float *cu = reinterpret_cast<const float *>(sm + C::kOffCst), *cg = cu + D, *cbt = cg + D;
    const int tt = lane & 15, half = lane >> 4;
    float shs = 0.f, ps = 0.f, qs = 0.f;
    // Partly rolled for d = 128: the kernel's hot code must fit the SM's instruction cache.
    constexpr int kUnroll = D == 128 ? 2 : D / 16;
#pragma unroll(kUnroll)
    for (int ch = 0; ch < D / 16; ++ch) {
        const int jj = half * (D / 16) + ch;  // 16-byte chunk (8 features)
        const uint4 kb = *reinterpret_cast<const uint4 *>(stg + C::kOffK + swz(tt, jj));
        const uint4 vb = *reinterpret_cast<const uint4 *>(stg + C::kOffV + swz(tt, jj));
        const uint32_t kw[4] = {kb.x, kb.y, kb.z, kb.w}, vw[4] = {vb.x, vb.y, vb.z, vb.w};
        const float4 *u4 = reinterpret_cast<const float4 *>(cu + 8 * jj);
        const float4 *g4 = reinterpret_cast<const float4 *>(cg + 8 * jj);
        const float4 *b4 = reinterpret_cast<const float4 *>(cbt + 8 * jj);
        const float4 uu[2] = {u4[0], u4[1]}, gg[2] = {g4[0], g4[1]}, bb[2] = {b4[0], b4[1]};
        const float uf[8] = {uu[0].x, uu[0].y, uu[0].z, uu[0].w, uu[1].x, uu[1].y, uu[1].z, uu[1].w};
        const float gf[8] = {gg[0].x, gg[0].y, gg[0].z, gg[0].w, gg[1].x, gg[1].y, gg[1].z, gg[1].w};
        const float bf[8] = {bb[0].x, bb[0].y, bb[0].z, bb[0].w, bb[1].x, bb[1].y, bb[1].z, bb[1].w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t kbits = q & 1 ? kw[q >> 1] >> 16 : kw[q >> 1] & 0xffffu;
            const uint32_t vbits = q & 1 ? vw[q >> 1] >> 16 : vw[q >> 1] & 0xffffu;
            const float kf = bf16_bits_to_f32(kbits), vf = bf16_bits_to_f32(vbits);
            const float kv = kf - vf + bf[q];
            shs = fmaf(uf[q], kf, shs);
            ps = fmaf(gf[q], kv, ps);
            qs = fmaf(kv, kv, qs);
        }
    }
    shs += __shfl_xor_sync(kFull, shs, 16);
    ps += __shfl_xor_sync(kFull, ps, 16);
    qs += __shfl_xor_sync(kFull, qs, 16);
    if (half == 0) {
        reinterpret_cast<float *>(stg + C::kOffSh)[tt] = shs + cmean;
        reinterpret_cast<float *>(stg + C::kOffPk)[tt] = ps;
        reinterpret_cast<float *>(stg + C::kOffQk)[tt] = qs;
    }
}

// ------------------------------------------------------------------ L: loader + per-token sums
// The loader warp issues the TMA loads of stage i, and kLag stages behind,
// once stage j has landed, writes the per-token scalars of the LayerNorm
// reduction into it: the shift sh_t = u0 . k_t + mean(c0) (u0 = feature mean
// of W_0's rows), sum_f gamma_f kv_f and sum_f kv_f^2 (kv = k - v + beta). Its
// arrival on prep[j] joins the prep warp's.
constexpr int kLag = 2;

// LOADQ: the query tiles are loaded (unless the queries are the keys); SUMS: the
// per-token scalars of the chain are written (d = 64). The cluster kernel's
// chain CTA loads no queries, its output CTA forms no per-token scalars.
template <int D, bool LOADQ = true, bool SUMS = kSumsInLoader<D>>
__device__ void role_loader_sums(const CUtensorMap *tmQ, const CUtensorMap *tmK, const CUtensorMap *tmV,
                                 const LinearParams &p, uint8_t *sm, const Ring &R, int chain, int bi, int hi, int lane,
                                 int nsteps)
{
    using C = Cfg<D>;
    static_assert(!SUMS || kSumsInLoader<D>, "per-token scalars in the loader for d = 64 only");
    const int T = p.T;
    const float *eta = p.eta + (size_t)chain * T;
    const bool no_q = !LOADQ || p.q_is_k;
    const float cmean = SUMS ? chain_consts<D>(p, sm, bi, hi, lane) : 0.f;
    uint32_t mag = 0;  // range check of the tiles this warp converts
    if (lane == 0) {
        prefetch_tmap(tmQ);
        prefetch_tmap(tmK);
        prefetch_tmap(tmV);
    }
    int issued = 0;
    const int lag = kLoaderPrep<D> ? kLag : 0;
    for (int i = 0; i < nsteps + lag; ++i) {
        // The lagged work on stage i - kLag first: it needs only that stage's own
        // loads, while the load of stage i waits for the consumers to release it
        // (about two super-steps behind the chain); done the other way round, the
        // weight warps would wait for this work.
        if (kLoaderPrep<D> && i >= kLag) {
            const int j = i - kLag, sj = j % C::kStages;
            if (!wait_bar(&R.full[sj], parity_of(j / C::kStages), R.flags)) {
                abort_chain(R.flags, p.status);
                break;
            }
            if (p.eta_gate && lane < kSS) {  // eta = eta_base * sigmoid(logit) in place; 0 past T
                float *se = reinterpret_cast<float *>(stage_ptr<D>(sm, sj) + C::kOffEta);
                const int t = j * kSS + lane;
                se[lane] = t < T ? __fdividef(p.eta_base, 1.f + __expf(-se[lane])) : 0.f;
            }
            if (SUMS) token_sums<D>(stage_ptr<D>(sm, sj), sm, cmean, lane);
            if (kCopiesInLoader<D>) fp16_copies<D>(stage_ptr<D>(sm, sj), p.q_is_k != 0, lane, mag);
            warp_arrive(&R.prep[sj], lane);
        }
        if (i < nsteps) {
            const int st = i % C::kStages;
            if (!wait_bar(&R.empty[st], parity_of(i / C::kStages) ^ 1u, R.flags)) {
                abort_chain(R.flags, p.status);
                break;
            }
            TTT_TRACE_AT(p, i, 14);
            uint8_t *stg = stage_ptr<D>(sm, st);
            const int t0 = i * kSS;
            float *se = reinterpret_cast<float *>(stg + C::kOffEta);
#ifdef TTT_FAULT_HOOKS
            const bool drop = i == p.drop_step;  // failure-detection tests: this stage never lands
#else
            constexpr bool drop = false;
#endif
            if (!drop && lane < kSS) {
                const int t = t0 + lane;
                cp_async_4(se + lane, eta + (t < T ? t : 0), t < T ? 4u : 0u);  // zero-fill past T
            }
            if (!drop) cp_async_mbar_arrive_noinc(&R.full[st]);
            if (!drop && lane == 0) {
                mbar_arrive_expect_tx(&R.full[st], (no_q ? 2 : 3) * C::kTile);
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    tma_load_3d(stg + C::kOffK + h * 2048, tmK, &R.full[st], h * 64, t0, chain);
                    if (!no_q) tma_load_3d(stg + C::kOffQ + h * 2048, tmQ, &R.full[st], h * 64, t0, chain);
                    tma_load_3d(stg + C::kOffV + h * 2048, tmV, &R.full[st], h * 64, t0, chain);
                }
            }
            issued = i + 1;
        }
    }
    if (kCopiesInLoader<D>) {
        const bool range_bad = (mag & 0xffffu) >= 0x4780u || (mag >> 16) >= 0x4780u;
        if (__any_sync(kFull, range_bad) && lane == 0) {
            R.flags[1] = 1;
            record(p.status, TTT_ERR_RANGE);
        }
    }
    // Never leave while a copy issued here may still be landing in shared memory.
    for (int i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i)
        (void)mbar_wait(&R.full[i % C::kStages], parity_of(i / C::kStages));
}

// ------------------------------------------------------------------ P: prep
// What the prep warp forms (the one-CTA kernels: all of it; the cluster
// kernel's chain CTA only the K copy and K_{i-1} K_i^T, its output CTA the K and
// Q copies and Q K^T).
constexpr int kPrepQ = 1, kPrepMq = 2, kPrepKx = 4, kPrepAll = 7;

template <int D, int SUBB, int PREP = kPrepAll>
__device__ void role_prep(const LinearParams &p, uint8_t *sm, const Ring &R, int bi, int hi, int lane, int nsteps)
{
    using C = Cfg<D>;
    const int g = lane >> 2, c4 = lane & 3;
    const bool prefix = p.prefix != 0;
    uint32_t mag = 0;  // per-halfword max of |bf16 bits|: >= 0x4780 means |x| >= 2^16 (or inf/nan)
    const int ra = (lane & 7) + ((lane >> 3) & 1) * 8;  // A-fragment row (ldmatrix x4)
    const int rb = (lane & 7) + (lane >> 4) * 8;        // B-fragment row
    const float cmean = kSumsInLoader<D> ? 0.f : chain_consts<D>(p, sm, bi, hi, lane);
    for (int i = 0; i < nsteps; ++i) {
        const int st = i % C::kStages;
        if (!wait_bar(&R.full[st], parity_of(i / C::kStages), R.flags)) {
            abort_chain(R.flags, p.status);
            return;
        }
        TTT_TRACE_AT(p, i, 12);
        uint8_t *stg = stage_ptr<D>(sm, st);
        // (1) fp16 copies of the K and Q tiles (the loader makes them for d = 128).
        if (!kCopiesInLoader<D>) fp16_copies<D>(stg, p.q_is_k != 0 || !(PREP & kPrepQ), lane, mag);
        if (D == 128) TTT_TRACE_AT(p, i, 14);
        if (!kSumsInLoader<D>) token_sums<D>(stg, sm, cmean, lane);
        if (D == 128) TTT_TRACE_AT(p, i, 15);
        __syncwarp();
        // (3) Gram fragments. d*[j][r] holds (t = g + 8(r>>1), s = 8j + 2c4 + (r&1)):
        //     dq = Q_i K_i^T, dk = K_i K_i^T, dx = K_i K_{i-1}^T (t in step i, s in step i-1),
        //     from the fp16 copies, or (copies in the loader) from the bf16 tiles.
        constexpr bool kBf = kCopiesInLoader<D>;
        auto gmma = [](float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
            if constexpr (kBf)
                mma16816_bf16(d, a, b0, b1);
            else
                mma16816(d, a, b0, b1);
        };
        const int offK = kBf ? C::kOffK : C::kOffKh, offQ = kBf ? C::offQ(p) : C::offQh(p);
        const uint32_t sK = smem_u32(stg + offK), sQ = smem_u32(stg + offQ);
        const uint32_t sKp = smem_u32(stage_ptr<D>(sm, (i + C::kStages - 1) % C::kStages) + offK);
        const bool has_prev = (PREP & kPrepKx) && i > 0;
        float dq[2][4] = {}, dk[2][4] = {}, dx[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t aq[4], ak[4], bk[4];
            ldsm_x4(bk, sK + swz(rb, 2 * ks + ((lane >> 3) & 1)));
            if (PREP & kPrepMq) {
                ldsm_x4(aq, sQ + swz(ra, 2 * ks + (lane >> 4)));
                gmma(dq[0], aq, bk[0], bk[1]);
                gmma(dq[1], aq, bk[2], bk[3]);
            }
            if (SUBB < 16 || has_prev) ldsm_x4(ak, sK + swz(ra, 2 * ks + (lane >> 4)));
            if (SUBB < 16) {
                gmma(dk[0], ak, bk[0], bk[1]);
                gmma(dk[1], ak, bk[2], bk[3]);
            }
            if (has_prev) {
                uint32_t bp[4];
                ldsm_x4(bp, sKp + swz(rb, 2 * ks + ((lane >> 3) & 1)));
                gmma(dx[0], ak, bp[0], bp[1]);
                gmma(dx[1], ak, bp[2], bp[3]);
            }
        }
        // As B fragments (k = s, n = t) for the W warps. The mask selects which
        // tokens' updates the output of token t sees: s <= t (in-batch prefix), or
        // under the anchor rule only the mini-batches before t's own (none when
        // b >= 16: the outputs use the anchor alone).
        auto mq = [&](int j, int r) {
            const int t = g + 8 * (r >> 1), s = 8 * j + 2 * c4 + (r & 1);
            const bool seen = prefix ? s <= t : s / SUBB < t / SUBB;
            return seen ? dq[j][r] + 1.f : 0.f;
        };
        if (PREP & kPrepMq)
            reinterpret_cast<uint4 *>(stg + C::kOffMq)[lane] =
                make_uint4(pack_h2(mq(0, 0), mq(0, 1)), pack_h2(mq(1, 0), mq(1, 1)),
                           pack_h2(mq(0, 2), mq(0, 3)), pack_h2(mq(1, 2), mq(1, 3)));
        if (SUBB < 16) {
            const uint32_t k0 = pack_h2(dk[0][0] + 1.f, dk[0][1] + 1.f), k1 = pack_h2(dk[1][0] + 1.f, dk[1][1] + 1.f);
            const uint32_t k2 = pack_h2(dk[0][2] + 1.f, dk[0][3] + 1.f), k3 = pack_h2(dk[1][2] + 1.f, dk[1][3] + 1.f);
            reinterpret_cast<uint4 *>(stg + C::kOffGk)[lane] = make_uint4(k0, k1, k2, k3);   // B (k = s, n = t)
            reinterpret_cast<uint4 *>(stg + C::kOffGkA)[lane] = make_uint4(k0, k2, k1, k3);  // A (m = t, k = s)
        }
        if (has_prev) {
            const uint32_t x0 = pack_h2(dx[0][0] + 1.f, dx[0][1] + 1.f), x1 = pack_h2(dx[1][0] + 1.f, dx[1][1] + 1.f);
            const uint32_t x2 = pack_h2(dx[0][2] + 1.f, dx[0][3] + 1.f), x3 = pack_h2(dx[1][2] + 1.f, dx[1][3] + 1.f);
            reinterpret_cast<uint4 *>(stg + C::kOffKx)[lane] = make_uint4(x0, x1, x2, x3);   // B (k = s_{i-1}, n = t_i)
            reinterpret_cast<uint4 *>(stg + C::kOffKxA)[lane] = make_uint4(x0, x2, x1, x3);  // A (m = t_i, k = s_{i-1})
        }
        warp_arrive(&R.prep[st], lane);
        TTT_TRACE_AT(p, i, 13);
        if (PREP & kPrepKx) {
            if (has_prev && lane == 0) mbar_arrive(&R.empty[(i + C::kStages - 1) % C::kStages]);  // K_{i-1} no longer read
        } else if (lane == 0) {
            mbar_arrive(&R.empty[st]);  // no Gram reads this stage again
        }
    }
    if ((PREP & kPrepKx) && nsteps > 0 && lane == 0) mbar_arrive(&R.empty[(nsteps - 1) % C::kStages]);
    const bool range_bad = (mag & 0xffffu) >= 0x4780u || (mag >> 16) >= 0x4780u;
    if (__any_sync(kFull, range_bad) && lane == 0) {
        R.flags[1] = 1;
        record(p.status, TTT_ERR_RANGE);
    }
}

// ------------------------------------------------------------------ W: weight + chain warps
// acc (this warp's 16 rows x 16 tokens) = c + W tile^T, W packed to fp16 on the fly.
template <int D>
__device__ __forceinline__ void rows_gemm(const float (&Wa)[D / 8][4], const float (&cb)[2], uint32_t tile, int lane,
                                          float (&acc)[2][4])
{
    const int rb = (lane & 7) + (lane >> 4) * 8, cb16 = (lane >> 3) & 1;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[nt][r] = cb[r >> 1];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t af[4] = {pack_h2(Wa[2 * ks][0], Wa[2 * ks][1]), pack_h2(Wa[2 * ks][2], Wa[2 * ks][3]),
                                pack_h2(Wa[2 * ks + 1][0], Wa[2 * ks + 1][1]),
                                pack_h2(Wa[2 * ks + 1][2], Wa[2 * ks + 1][3])};
        uint32_t bk[4];
        ldsm_x4(bk, tile + swz(rb, 2 * ks + cb16));
        mma16816(acc[0], af, bk[0], bk[1]);
        mma16816(acc[1], af, bk[2], bk[3]);
    }
}

// rows_gemm with W already packed as fp16 A fragments (one set per k-step).
template <int D>
__device__ __forceinline__ void rows_gemm_h(const uint32_t (&Wh)[D / 16][4], const float (&cb)[2], uint32_t tile,
                                            int lane, float (&acc)[2][4])
{
    const int rb = (lane & 7) + (lane >> 4) * 8, cb16 = (lane >> 3) & 1;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[nt][r] = cb[r >> 1];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t bk[4];
        ldsm_x4(bk, tile + swz(rb, 2 * ks + cb16));
        mma16816(acc[0], Wh[ks], bk[0], bk[1]);
        mma16816(acc[1], Wh[ks], bk[2], bk[3]);
    }
}

// Two products of the same rows with one fp16 packing of W: acc0 from tile0 and
// acc1 from tile1 (four independent accumulator chains).
template <int D>
__device__ __forceinline__ void rows_gemm2(const float (&Wa)[D / 8][4], const float (&cb)[2], uint32_t tile0,
                                           uint32_t tile1, int lane, float (&acc0)[2][4], float (&acc1)[2][4])
{
    const int rb = (lane & 7) + (lane >> 4) * 8, cb16 = (lane >> 3) & 1;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc0[nt][r] = acc1[nt][r] = cb[r >> 1];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t b0[4], b1[4];
        ldsm_x4(b0, tile0 + swz(rb, 2 * ks + cb16));
        ldsm_x4(b1, tile1 + swz(rb, 2 * ks + cb16));
        const uint32_t af[4] = {pack_h2(Wa[2 * ks][0], Wa[2 * ks][1]), pack_h2(Wa[2 * ks][2], Wa[2 * ks][3]),
                                pack_h2(Wa[2 * ks + 1][0], Wa[2 * ks + 1][1]),
                                pack_h2(Wa[2 * ks + 1][2], Wa[2 * ks + 1][3])};
        mma16816(acc0[0], af, b0[0], b0[1]);
        mma16816(acc0[1], af, b0[2], b0[3]);
        mma16816(acc1[0], af, b1[0], b1[1]);
        mma16816(acc1[1], af, b1[2], b1[3]);
    }
}

// A weight warp's entry of a reduction round: its twenty per-column moments
// (five moments x the lane's four columns 8nt + 2c4 + e), summed over the
// warp's rows, i.e. over the eight lanes g that share c4, stored as
// redX[w][t] = moments 0-3 and redY[w][t] = moment 4. The lanes split the
// values as they reduce them (g bit 2 picks the column tile nt, bit 1 the
// column e, bit 0 moments 0-2 or 3-4): eighteen shuffles where summing each
// value over all eight lanes takes sixty.
__device__ __forceinline__ void store_moments(const float (&q5)[5][2][2], float4 *redX, float *redY, int w, int g,
                                              int c4)
{
    const int bA = (g >> 2) & 1, bB = (g >> 1) & 1, bC = g & 1;
    float hA[5][2], hB[5];
#pragma unroll
    for (int k = 0; k < 5; ++k)
#pragma unroll
        for (int e = 0; e < 2; ++e)
            hA[k][e] = (bA ? q5[k][1][e] : q5[k][0][e]) + __shfl_xor_sync(kFull, bA ? q5[k][0][e] : q5[k][1][e], 16);
#pragma unroll
    for (int k = 0; k < 5; ++k)
        hB[k] = (bB ? hA[k][1] : hA[k][0]) + __shfl_xor_sync(kFull, bB ? hA[k][0] : hA[k][1], 8);
    const float x0 = __shfl_xor_sync(kFull, bC ? hB[0] : hB[3], 4);
    const float x1 = __shfl_xor_sync(kFull, bC ? hB[1] : hB[4], 4);
    const float x2 = __shfl_xor_sync(kFull, hB[2], 4);
    const int t = 8 * bA + 2 * c4 + bB;
    float *rx = reinterpret_cast<float *>(redX + w * kSS + t);
    if (bC == 0) {  // moments 0, 1, 2
        rx[0] = hB[0] + x0;
        rx[1] = hB[1] + x1;
        rx[2] = hB[2] + x2;
    } else {        // moments 3, 4
        rx[3] = hB[3] + x0;
        redY[w * kSS + t] = hB[4] + x1;
    }
}

template <int D, int SUBB>
__device__ void role_weights(const LinearParams &p, uint8_t *sm, const Ring &R, int w, int chain, int bi,
                             int hi, size_t tok0, int lane, int nsteps)
{
    using C = Cfg<D>;
    constexpr int MT = C::MT, NTW = D / 8, NSUB = kSS / SUBB;
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
    float gam2all = 0.f;  // sum of gamma^2 over all features
#pragma unroll
    for (int q = 0; q < D / 32; ++q) gam2all = fmaf(p.ln_g[hi * D + lane + 32 * q], p.ln_g[hi * D + lane + 32 * q], gam2all);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gam2all += __shfl_xor_sync(kFull, gam2all, o);
    const int rb = (lane & 7) + (lane >> 4) * 8;        // ldmatrix row, non-transposed B
    const int cb16 = (lane >> 3) & 1;
    const int rt = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row, transposed B
    const int ct = lane >> 4;
    const float invD = 1.f / (float)D, eps = p.eps;
    const int T = p.T;

    // Prologue: Y_0^T = W_0 K_0^T + c_0.
    float yk[2][4];
    if (!wait_bar(&R.full[0], 0u, R.flags) || !wait_bar(&R.prep[0], 0u, R.flags)) {
        abort_chain(R.flags, p.status);
        return;
    }
    rows_gemm<D>(Wa, cb, smem_u32(stage_ptr<D>(sm, 0) + C::kOffKh), lane, yk);

    int rnd = 0;  // reduction rounds so far (buffer rnd & 1, phase (rnd >> 1) & 1)
    for (int i = 0; i < nsteps; ++i) {
        const int st = i % C::kStages, slot = i & 1, stn = (i + 1) % C::kStages;
        const bool has_next = i + 1 < nsteps;
        uint8_t *stg = stage_ptr<D>(sm, st);
        uint8_t *stgn = stage_ptr<D>(sm, stn);
        if (w == 0) TTT_TRACE_AT(p, i, 0);
        bool ok = true;  // stage i's full/prep were waited for as "next" (or in the prologue)
        if (has_next)
            ok = ok && wait_bar(&R.full[stn], parity_of((i + 1) / C::kStages), R.flags) &&
                 wait_bar(&R.prep[stn], parity_of((i + 1) / C::kStages), R.flags);
        ok = ok && wait_bar(&R.yempty[slot], parity_of(i >> 1) ^ 1u, R.flags);
        if (!ok) {
            abort_chain(R.flags, p.status);
            return;
        }
        if (w == 0) TTT_TRACE_AT(p, i, 1);
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
        // Per-column (token) scalars of this lane's four columns t = 8nt + 2c4 + e.
        const float *ssh = reinterpret_cast<const float *>(stg + C::kOffSh);
        float escale[2][2], shv[2][2];
        {
            const float *se = reinterpret_cast<const float *>(stg + C::kOffEta);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 e2 = *reinterpret_cast<const float2 *>(se + 8 * nt + 2 * c4);
                const float2 s2 = *reinterpret_cast<const float2 *>(ssh + 8 * nt + 2 * c4);
                escale[nt][0] = -e2.x * (1.f / (float)SUBB);
                escale[nt][1] = -e2.y * (1.f / (float)SUBB);
                shv[nt][0] = s2.x;
                shv[nt][1] = s2.y;
            }
        }
        // The column this lane combines across the W warps (lanes g and g + 4
        // duplicate); its results reach the lanes that hold it by shuffles.
        const int tc = 8 * (g & 1) + 2 * c4 + ((g >> 1) & 1);
        const float sh_c = ssh[tc];
        const float pk_c = reinterpret_cast<const float *>(stg + C::kOffPk)[tc];
        const float qk_c = reinterpret_cast<const float *>(stg + C::kOffQk)[tc];
        float at[2][4] = {};   // A~ = -(eta/b) G, fp16-rounded, every column once set
        float lin[2][2] = {};  // inner loss of each column
        float Sn[2][4], Rq[2][4];
#pragma unroll
        for (int m = 0; m < NSUB; ++m) {
            // --- this warp's shifted sums over its 16 rows, for every column.
            float q5[5][2][2];  // [moment][nt][e]
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float a1 = 0.f, a2 = 0.f, ab = 0.f, ac = 0.f, ad = 0.f;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float dv = yk[nt][e + 2 * u] - shv[nt][e];
                        const float g2d = gam[u] * gam[u] * dv;
                        a1 += dv;
                        a2 = fmaf(dv, dv, a2);
                        ab += g2d;
                        ac = fmaf(g2d, dv, ac);
                        ad = fmaf(gam[u] * kv[nt][e + 2 * u], dv, ad);
                    }
                    q5[0][nt][e] = a1;
                    q5[1][nt][e] = a2;
                    q5[2][nt][e] = ab;
                    q5[3][nt][e] = ac;
                    q5[4][nt][e] = ad;
                }
            if (w == 0 && m == 0) TTT_TRACE_AT(p, i, 5);
            const int buf = rnd & 1;
            float4 *redX = reinterpret_cast<float4 *>(sm + C::kOffRedX) + buf * MT * kSS;
            float *redY = reinterpret_cast<float *>(sm + C::kOffRedY) + buf * MT * kSS;
            store_moments(q5, redX, redY, w, g, c4);
            warp_arrive(&R.red[buf], lane);
            if (w == 0 && m == 0) TTT_TRACE_AT(p, i, 6);
            if (m == 0) {
                // Independent tensor-core work while the other W warps finish their sums:
                // S_{i+1} = W_{i-1} K_{i+1}^T + c_{i-1}, Rq_i = W_{i-1} Q_i^T + c_{i-1}, in one
                // pass (one copy of the code; on the last step the unused S reads the Q tile).
                const uint32_t sQi = smem_u32(stg + C::offQh(p));
                rows_gemm2<D>(Wa, cb, has_next ? smem_u32(stgn + C::kOffKh) : sQi, sQi, lane, Sn, Rq);
                if (w == 0) TTT_TRACE_AT(p, i, 2);
            }
            if (!wait_bar(&R.red[buf], parity_of(rnd >> 1), R.flags)) {
                abort_chain(R.flags, p.status);
                return;
            }
            ++rnd;
            if (w == 0 && m == 0) TTT_TRACE_AT(p, i, 7);
            // Combine column tc over the W warps: moments about mu = sh + ee.
            float mu_c, rs_c, M1_c, M2_c, LE_c;
            {
                float S1 = 0.f, S2 = 0.f, SB = 0.f, SC = 0.f, SD = 0.f;
#pragma unroll
                for (int u = 0; u < MT; ++u) {
                    const float4 x = redX[u * kSS + tc];
                    S1 += x.x;
                    S2 += x.y;
                    SB += x.z;
                    SC += x.w;
                    SD += redY[u * kSS + tc];
                }
                const float ee = S1 * invD;
                const float syy = fmaxf(fmaf(-ee, S1, S2), 0.f);                    // sum (y - mu)^2
                rs_c = rsqrtf(syy * invD + eps);
                const float sg1 = fmaf(-ee, gam2all, SB);                             // sum g^2 (y - mu)
                const float sg2 = fmaf(ee * ee, gam2all, fmaf(-2.f * ee, SB, SC));   // sum g^2 (y - mu)^2
                const float sgk = fmaf(-ee, pk_c, SD);                                // sum g kv (y - mu)
                M1_c = 2.f * invD * fmaf(rs_c, sg1, pk_c);                            // mean of dh
                M2_c = 2.f * invD * rs_c * fmaf(rs_c, sg2, sgk);                      // mean of dh * yh
                LE_c = fmaf(rs_c, fmaf(rs_c, sg2, 2.f * sgk), qk_c);                 // sum E^2
                mu_c = sh_c + ee;
            }
            float ad[2][4];  // this mini-batch's A~ columns (zero elsewhere)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = 8 * nt + 2 * c4 + e;
                    const int src = (nt + 2 * e) * 4 + c4;
                    const float mu = __shfl_sync(kFull, mu_c, src);
                    const float rs = __shfl_sync(kFull, rs_c, src);
                    const float M1 = __shfl_sync(kFull, M1_c, src);
                    const float M2 = __shfl_sync(kFull, M2_c, src);
                    const float LE = __shfl_sync(kFull, LE_c, src);
                    const bool in_m = NSUB == 1 || t / SUBB == m;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float yh = (yk[nt][e + 2 * u] - mu) * rs;
                        const float E = fmaf(gam[u], yh, kv[nt][e + 2 * u]);
                        const float G = rs * (2.f * gam[u] * E - M1 - yh * M2);
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
        const uint32_t af[4] = {pack_h2(at[0][0], at[0][1]), pack_h2(at[0][2], at[0][3]),
                                pack_h2(at[1][0], at[1][1]), pack_h2(at[1][2], at[1][3])};
        // The chain: Y_{i+1}^T = S_{i+1} + A~_i (K_i K_{i+1}^T + 1).
        if (has_next) {
            const uint4 kx = reinterpret_cast<const uint4 *>(stgn + C::kOffKx)[lane];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) yk[nt][r] = Sn[nt][r];
            mma16816(yk[0], af, kx.x, kx.y);
            mma16816(yk[1], af, kx.z, kx.w);
        }
        // W += A~ K_i, c += A~ 1   (W_{i-1} -> W_i for this warp's rows), over the
        // committed tokens (all of them unless a partial last mini-batch ends here).
        const int tcm = committed_in_step(p.t_commit, i);
        {
            uint32_t au[4] = {af[0], af[1], af[2], af[3]};
            mask_tokens(au, tcm, lane);
            const uint32_t sK = smem_u32(stg + C::kOffKh);
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                uint32_t bt[4];
                ldsm_x4_t(bt, sK + swz(rt, 2 * j + ct));
                mma16816(Wa[2 * j], au, bt[0], bt[1]);
                mma16816(Wa[2 * j + 1], au, bt[2], bt[3]);
            }
        }
        auto atc = [&](int nt, int r) { return 8 * nt + 2 * c4 + (r & 1) < tcm ? at[nt][r] : 0.f; };
        float s0 = atc(0, 0) + atc(0, 1) + atc(1, 0) + atc(1, 1);
        float s1r = atc(0, 2) + atc(0, 3) + atc(1, 2) + atc(1, 3);
        s0 += __shfl_xor_sync(kFull, s0, 1);
        s0 += __shfl_xor_sync(kFull, s0, 2);
        s1r += __shfl_xor_sync(kFull, s1r, 1);
        s1r += __shfl_xor_sync(kFull, s1r, 2);
        cb[0] += s0;
        cb[1] += s1r;
        // Yq^T = Rq^T + A~ Mq (in-batch prefix of every query) -> output warps.
        {
            const uint4 mq = reinterpret_cast<const uint4 *>(stg + C::kOffMq)[lane];
            mma16816(Rq[0], af, mq.x, mq.y);
            mma16816(Rq[1], af, mq.z, mq.w);
        }
        if (w == 0) TTT_TRACE_AT(p, i, 11);
        float *ys = reinterpret_cast<float *>(sm + C::kOffY + slot * kSS * C::YS * 4);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r)
                ys[(8 * nt + 2 * c4 + (r & 1)) * C::YS + 16 * w + g + 8 * (r >> 1)] = Rq[nt][r];
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

// ------------------------------------------------------------------ W: mini-batches of 32 / 64 tokens
// The two-phase form for NB <= 4 (the mini-batch's stages stay in the ring):
// phase 1 takes Y, the LayerNorm backward and A~ of every block at the anchor,
// back to back; phase 2 emits each block's outputs with the running in-batch
// prefix (Wa = W_{i-1} + sum of the earlier blocks' A~ K) and applies the
// block's update, ending at W_i. Measured faster than the one-pass form below
// at b = 64.
template <int D, int NB>
__device__ void role_weights_mb2(const LinearParams &p, uint8_t *sm, const Ring &R, int w, int chain, int bi, int hi,
                                 size_t tok0, int lane, int nsteps)
{
    static_assert(NB <= 4, "phase 1 keeps every block of the mini-batch in the stage ring");
    using C = Cfg<D>;
    constexpr int MT = C::MT, NTW = D / 8, BSZ = kSS * NB;
    const int g = lane >> 2, c4 = lane & 3;
    const int r0 = 16 * w + g, r1 = r0 + 8;
    const float *W0 = p.W0 + bi * p.w0_bstride + (long long)hi * D * D;
    const float *c0 = p.c0 + bi * p.c0_bstride + (long long)hi * D;
    float Wa[NTW][4];
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
    float gam2all = 0.f;
#pragma unroll
    for (int q = 0; q < D / 32; ++q) gam2all = fmaf(p.ln_g[hi * D + lane + 32 * q], p.ln_g[hi * D + lane + 32 * q], gam2all);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gam2all += __shfl_xor_sync(kFull, gam2all, o);
    const int rb = (lane & 7) + (lane >> 4) * 8, cb16 = (lane >> 3) & 1;
    const int rt = (lane & 7) + ((lane >> 3) & 1) * 8, ct = lane >> 4;
    const float invD = 1.f / (float)D, eps = p.eps;
    const int T = p.T;
    // Final state: written once, after the last committed mini-batch (a partial
    // last mini-batch still runs its blocks' updates for its own outputs).
    auto write_state = [&]() {
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
    };
    bool state_written = false;
    const int nmb = (nsteps + NB - 1) / NB;
    int rnd = 0;
    for (int mbi = 0; mbi < nmb; ++mbi) {
        uint32_t afs[NB][4];
        const int nbk = nsteps - mbi * NB < NB ? nsteps - mbi * NB : NB;  // blocks with tokens
        if ((mbi + 1) * BSZ > p.t_commit && !state_written) {  // the uncommitted partial mini-batch
            write_state();
            state_written = true;
        }
        // Phase 1: every block's A~ at the anchor.
#pragma unroll 1
        for (int pb = 0; pb < NB; ++pb) {
            if (pb >= nbk) break;
            const int i = mbi * NB + pb, st = i % C::kStages;
            uint8_t *stg = stage_ptr<D>(sm, st);
            if (!wait_bar(&R.full[st], parity_of(i / C::kStages), R.flags) ||
                !wait_bar(&R.prep[st], parity_of(i / C::kStages), R.flags)) {
                abort_chain(R.flags, p.status);
                return;
            }
            float yk[2][4];
            rows_gemm<D>(Wa, cb, smem_u32(stg + C::kOffKh), lane, yk);
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
            const float *ssh = reinterpret_cast<const float *>(stg + C::kOffSh);
            const float *se = reinterpret_cast<const float *>(stg + C::kOffEta);
            float escale[2][2], shv[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 e2 = *reinterpret_cast<const float2 *>(se + 8 * nt + 2 * c4);
                const float2 s2 = *reinterpret_cast<const float2 *>(ssh + 8 * nt + 2 * c4);
                escale[nt][0] = -e2.x * (1.f / (float)BSZ);
                escale[nt][1] = -e2.y * (1.f / (float)BSZ);
                shv[nt][0] = s2.x;
                shv[nt][1] = s2.y;
            }
            const int tc = 8 * (g & 1) + 2 * c4 + ((g >> 1) & 1);
            const float sh_c = ssh[tc];
            const float pk_c = reinterpret_cast<const float *>(stg + C::kOffPk)[tc];
            const float qk_c = reinterpret_cast<const float *>(stg + C::kOffQk)[tc];
            float q5[5][2][2];  // [moment][nt][e]
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float a1 = 0.f, a2 = 0.f, ab = 0.f, ac = 0.f, ad = 0.f;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float dv = yk[nt][e + 2 * u] - shv[nt][e];
                        const float g2d = gam[u] * gam[u] * dv;
                        a1 += dv;
                        a2 = fmaf(dv, dv, a2);
                        ab += g2d;
                        ac = fmaf(g2d, dv, ac);
                        ad = fmaf(gam[u] * kv[nt][e + 2 * u], dv, ad);
                    }
                    q5[0][nt][e] = a1;
                    q5[1][nt][e] = a2;
                    q5[2][nt][e] = ab;
                    q5[3][nt][e] = ac;
                    q5[4][nt][e] = ad;
                }
            const int buf = rnd & 1;
            float4 *redX = reinterpret_cast<float4 *>(sm + C::kOffRedX) + buf * MT * kSS;
            float *redY = reinterpret_cast<float *>(sm + C::kOffRedY) + buf * MT * kSS;
            store_moments(q5, redX, redY, w, g, c4);
            warp_arrive(&R.red[buf], lane);
            if (!wait_bar(&R.red[buf], parity_of(rnd >> 1), R.flags)) {
                abort_chain(R.flags, p.status);
                return;
            }
            ++rnd;
            float mu_c, rs_c, M1_c, M2_c, LE_c;
            {
                float S1 = 0.f, S2 = 0.f, SB = 0.f, SC = 0.f, SD = 0.f;
#pragma unroll
                for (int u = 0; u < MT; ++u) {
                    const float4 x = redX[u * kSS + tc];
                    S1 += x.x;
                    S2 += x.y;
                    SB += x.z;
                    SC += x.w;
                    SD += redY[u * kSS + tc];
                }
                const float ee = S1 * invD;
                const float syy = fmaxf(fmaf(-ee, S1, S2), 0.f);
                rs_c = rsqrtf(syy * invD + eps);
                const float sg1 = fmaf(-ee, gam2all, SB);
                const float sg2 = fmaf(ee * ee, gam2all, fmaf(-2.f * ee, SB, SC));
                const float sgk = fmaf(-ee, pk_c, SD);
                M1_c = 2.f * invD * fmaf(rs_c, sg1, pk_c);
                M2_c = 2.f * invD * rs_c * fmaf(rs_c, sg2, sgk);
                LE_c = fmaf(rs_c, fmaf(rs_c, sg2, 2.f * sgk), qk_c);
                mu_c = sh_c + ee;
            }
            float at[2][4], lin[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int src = (nt + 2 * e) * 4 + c4;
                    const float mu = __shfl_sync(kFull, mu_c, src);
                    const float rs = __shfl_sync(kFull, rs_c, src);
                    const float M1 = __shfl_sync(kFull, M1_c, src);
                    const float M2 = __shfl_sync(kFull, M2_c, src);
                    lin[nt][e] = __shfl_sync(kFull, LE_c, src);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float yh = (yk[nt][e + 2 * u] - mu) * rs;
                        const float E = fmaf(gam[u], yh, kv[nt][e + 2 * u]);
                        const float G = rs * (2.f * gam[u] * E - M1 - yh * M2);
                        at[nt][e + 2 * u] = round_h(escale[nt][e] * G);
                    }
                }
            afs[pb][0] = pack_h2(at[0][0], at[0][1]);
            afs[pb][1] = pack_h2(at[0][2], at[0][3]);
            afs[pb][2] = pack_h2(at[1][0], at[1][1]);
            afs[pb][3] = pack_h2(at[1][2], at[1][3]);
            if (p.inner_loss && w == 0 && g == 0) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int t = i * kSS + 8 * nt + 2 * c4 + e;
                        if (t < T) p.inner_loss[tok0 + t] = lin[nt][e];
                    }
            }
        }
        // Phase 2: each block's outputs, then its update. With the in-batch prefix the
        // outputs see the running weights (W_{i-1} plus the earlier blocks' updates);
        // under the anchor rule every block's outputs come first, all at W_{i-1}.
        auto block_update = [&](int pb) {
            const int i = mbi * NB + pb, st = i % C::kStages;
            uint8_t *stg = stage_ptr<D>(sm, st);
            {
                const uint32_t sK = smem_u32(stg + C::kOffKh);
#pragma unroll
                for (int j = 0; j < MT; ++j) {
                    uint32_t bt[4];
                    ldsm_x4_t(bt, sK + swz(rt, 2 * j + ct));
                    mma16816(Wa[2 * j], afs[pb], bt[0], bt[1]);
                    mma16816(Wa[2 * j + 1], afs[pb], bt[2], bt[3]);
                }
            }
            auto hsum = [](uint32_t v) {
                return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu))) +
                       __half2float(__ushort_as_half((unsigned short)(v >> 16)));
            };
            float s0 = hsum(afs[pb][0]) + hsum(afs[pb][2]), s1r = hsum(afs[pb][1]) + hsum(afs[pb][3]);
            s0 += __shfl_xor_sync(kFull, s0, 1);
            s0 += __shfl_xor_sync(kFull, s0, 2);
            s1r += __shfl_xor_sync(kFull, s1r, 1);
            s1r += __shfl_xor_sync(kFull, s1r, 2);
            cb[0] += s0;
            cb[1] += s1r;
            warp_arrive(&R.empty[st], lane);
        };
#pragma unroll
        for (int pb = 0; pb < NB; ++pb) {
            if (pb >= nbk) break;
            const int i = mbi * NB + pb, st = i % C::kStages, slot = i & 1;
            uint8_t *stg = stage_ptr<D>(sm, st);
            float rq[2][4];
            rows_gemm<D>(Wa, cb, smem_u32(stg + C::offQh(p)), lane, rq);
            {
                const uint4 mq = reinterpret_cast<const uint4 *>(stg + C::kOffMq)[lane];
                mma16816(rq[0], afs[pb], mq.x, mq.y);
                mma16816(rq[1], afs[pb], mq.z, mq.w);
            }
            if (!wait_bar(&R.yempty[slot], parity_of(i >> 1) ^ 1u, R.flags)) {
                abort_chain(R.flags, p.status);
                return;
            }
            float *ys = reinterpret_cast<float *>(sm + C::kOffY + slot * kSS * C::YS * 4);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    ys[(8 * nt + 2 * c4 + (r & 1)) * C::YS + 16 * w + g + 8 * (r >> 1)] = rq[nt][r];
            warp_arrive(&R.yfull[slot], lane);
            if (p.prefix) block_update(pb);
        }
        if (!p.prefix) {
#pragma unroll
            for (int pb = 0; pb < NB; ++pb)
                if (pb < nbk) block_update(pb);
        }
    }
    if (!state_written) write_state();
}

// ------------------------------------------------------------------ W: mini-batches of 128 to 1024 tokens
// b = 16 NB: a mini-batch spans NB super-steps (blocks) that share the anchor
// W_{i-1}, so their gradients have no chain between them. One pass over the
// blocks: Y, the LayerNorm backward and A~ of a block come from the anchor (kept
// as the fp16 A fragments of that product); its outputs come from the running
// weights Wa = W_{i-1} + the earlier blocks' A~ K (the in-batch prefix) plus the
// block's own prefix (Mq); then the block's update goes into Wa and its stage is
// released. At the end of the mini-batch Wa = W_i becomes the next anchor.
template <int D, int NB>
__device__ void role_weights_mb(const LinearParams &p, uint8_t *sm, const Ring &R, int w, int chain, int bi, int hi,
                                size_t tok0, int lane, int nsteps)
{
    using C = Cfg<D>;
    constexpr int MT = C::MT, NTW = D / 8, BSZ = kSS * NB;
    const int g = lane >> 2, c4 = lane & 3;
    const int r0 = 16 * w + g, r1 = r0 + 8;
    const float *W0 = p.W0 + bi * p.w0_bstride + (long long)hi * D * D;
    const float *c0 = p.c0 + bi * p.c0_bstride + (long long)hi * D;
    float Wa[NTW][4];
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
    uint32_t Wh[D / 16][4];  // the anchor W_{i-1} as fp16 A fragments (what rows_gemm would pack)
    float ca[2];
    auto set_anchor = [&]() {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            Wh[ks][0] = pack_h2(Wa[2 * ks][0], Wa[2 * ks][1]);
            Wh[ks][1] = pack_h2(Wa[2 * ks][2], Wa[2 * ks][3]);
            Wh[ks][2] = pack_h2(Wa[2 * ks + 1][0], Wa[2 * ks + 1][1]);
            Wh[ks][3] = pack_h2(Wa[2 * ks + 1][2], Wa[2 * ks + 1][3]);
        }
        ca[0] = cb[0];
        ca[1] = cb[1];
    };
    set_anchor();
    const float gam[2] = {p.ln_g[hi * D + r0], p.ln_g[hi * D + r1]};
    const float bet[2] = {p.ln_b[hi * D + r0], p.ln_b[hi * D + r1]};
    float gam2all = 0.f;
#pragma unroll
    for (int q = 0; q < D / 32; ++q) gam2all = fmaf(p.ln_g[hi * D + lane + 32 * q], p.ln_g[hi * D + lane + 32 * q], gam2all);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gam2all += __shfl_xor_sync(kFull, gam2all, o);
    const int rb = (lane & 7) + (lane >> 4) * 8, cb16 = (lane >> 3) & 1;
    const int rt = (lane & 7) + ((lane >> 3) & 1) * 8, ct = lane >> 4;
    const float invD = 1.f / (float)D, eps = p.eps;
    const int T = p.T;
    // Final state: written once, after the last committed mini-batch (a partial
    // last mini-batch still runs its blocks' updates for its own outputs).
    auto write_state = [&]() {
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
    };
    bool state_written = false;
    const int nmb = (nsteps + NB - 1) / NB;
    int rnd = 0;
    for (int mbi = 0; mbi < nmb; ++mbi) {
        const int nbk = nsteps - mbi * NB < NB ? nsteps - mbi * NB : NB;  // blocks with tokens
        if ((mbi + 1) * BSZ > p.t_commit && !state_written) {  // the uncommitted partial mini-batch
            write_state();
            state_written = true;
        }
#pragma unroll 1
        for (int pb = 0; pb < NB; ++pb) {
            if (pb >= nbk) break;
            const int i = mbi * NB + pb, st = i % C::kStages;
            uint8_t *stg = stage_ptr<D>(sm, st);
            if (!wait_bar(&R.full[st], parity_of(i / C::kStages), R.flags) ||
                !wait_bar(&R.prep[st], parity_of(i / C::kStages), R.flags)) {
                abort_chain(R.flags, p.status);
                return;
            }
            float yk[2][4];
            rows_gemm_h<D>(Wh, ca, smem_u32(stg + C::kOffKh), lane, yk);  // Y at the anchor
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
            const float *ssh = reinterpret_cast<const float *>(stg + C::kOffSh);
            const float *se = reinterpret_cast<const float *>(stg + C::kOffEta);
            float escale[2][2], shv[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 e2 = *reinterpret_cast<const float2 *>(se + 8 * nt + 2 * c4);
                const float2 s2 = *reinterpret_cast<const float2 *>(ssh + 8 * nt + 2 * c4);
                escale[nt][0] = -e2.x * (1.f / (float)BSZ);
                escale[nt][1] = -e2.y * (1.f / (float)BSZ);
                shv[nt][0] = s2.x;
                shv[nt][1] = s2.y;
            }
            const int tc = 8 * (g & 1) + 2 * c4 + ((g >> 1) & 1);
            const float sh_c = ssh[tc];
            const float pk_c = reinterpret_cast<const float *>(stg + C::kOffPk)[tc];
            const float qk_c = reinterpret_cast<const float *>(stg + C::kOffQk)[tc];
            float q5[5][2][2];  // [moment][nt][e]
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float a1 = 0.f, a2 = 0.f, ab = 0.f, ac = 0.f, ad = 0.f;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float dv = yk[nt][e + 2 * u] - shv[nt][e];
                        const float g2d = gam[u] * gam[u] * dv;
                        a1 += dv;
                        a2 = fmaf(dv, dv, a2);
                        ab += g2d;
                        ac = fmaf(g2d, dv, ac);
                        ad = fmaf(gam[u] * kv[nt][e + 2 * u], dv, ad);
                    }
                    q5[0][nt][e] = a1;
                    q5[1][nt][e] = a2;
                    q5[2][nt][e] = ab;
                    q5[3][nt][e] = ac;
                    q5[4][nt][e] = ad;
                }
            const int buf = rnd & 1;
            float4 *redX = reinterpret_cast<float4 *>(sm + C::kOffRedX) + buf * MT * kSS;
            float *redY = reinterpret_cast<float *>(sm + C::kOffRedY) + buf * MT * kSS;
            store_moments(q5, redX, redY, w, g, c4);
            warp_arrive(&R.red[buf], lane);
            if (!wait_bar(&R.red[buf], parity_of(rnd >> 1), R.flags)) {
                abort_chain(R.flags, p.status);
                return;
            }
            ++rnd;
            float mu_c, rs_c, M1_c, M2_c, LE_c;
            {
                float S1 = 0.f, S2 = 0.f, SB = 0.f, SC = 0.f, SD = 0.f;
#pragma unroll
                for (int u = 0; u < MT; ++u) {
                    const float4 x = redX[u * kSS + tc];
                    S1 += x.x;
                    S2 += x.y;
                    SB += x.z;
                    SC += x.w;
                    SD += redY[u * kSS + tc];
                }
                const float ee = S1 * invD;
                const float syy = fmaxf(fmaf(-ee, S1, S2), 0.f);
                rs_c = rsqrtf(syy * invD + eps);
                const float sg1 = fmaf(-ee, gam2all, SB);
                const float sg2 = fmaf(ee * ee, gam2all, fmaf(-2.f * ee, SB, SC));
                const float sgk = fmaf(-ee, pk_c, SD);
                M1_c = 2.f * invD * fmaf(rs_c, sg1, pk_c);
                M2_c = 2.f * invD * rs_c * fmaf(rs_c, sg2, sgk);
                LE_c = fmaf(rs_c, fmaf(rs_c, sg2, 2.f * sgk), qk_c);
                mu_c = sh_c + ee;
            }
            float at[2][4], lin[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int src = (nt + 2 * e) * 4 + c4;
                    const float mu = __shfl_sync(kFull, mu_c, src);
                    const float rs = __shfl_sync(kFull, rs_c, src);
                    const float M1 = __shfl_sync(kFull, M1_c, src);
                    const float M2 = __shfl_sync(kFull, M2_c, src);
                    lin[nt][e] = __shfl_sync(kFull, LE_c, src);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float yh = (yk[nt][e + 2 * u] - mu) * rs;
                        const float E = fmaf(gam[u], yh, kv[nt][e + 2 * u]);
                        const float G = rs * (2.f * gam[u] * E - M1 - yh * M2);
                        at[nt][e + 2 * u] = round_h(escale[nt][e] * G);
                    }
                }
            const uint32_t af[4] = {pack_h2(at[0][0], at[0][1]), pack_h2(at[0][2], at[0][3]),
                                    pack_h2(at[1][0], at[1][1]), pack_h2(at[1][2], at[1][3])};
            if (p.inner_loss && w == 0 && g == 0) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int t = i * kSS + 8 * nt + 2 * c4 + e;
                        if (t < T) p.inner_loss[tok0 + t] = lin[nt][e];
                    }
            }
            // Outputs: the running weights (in-batch prefix of the earlier blocks) or,
            // under the anchor rule, the anchor; plus this block's own prefix (Mq).
            {
                const int slot = i & 1;
                float rq[2][4];
                if (p.prefix)
                    rows_gemm<D>(Wa, cb, smem_u32(stg + C::offQh(p)), lane, rq);
                else
                    rows_gemm_h<D>(Wh, ca, smem_u32(stg + C::offQh(p)), lane, rq);
                const uint4 mq = reinterpret_cast<const uint4 *>(stg + C::kOffMq)[lane];
                mma16816(rq[0], af, mq.x, mq.y);
                mma16816(rq[1], af, mq.z, mq.w);
                if (!wait_bar(&R.yempty[slot], parity_of(i >> 1) ^ 1u, R.flags)) {
                    abort_chain(R.flags, p.status);
                    return;
                }
                float *ys = reinterpret_cast<float *>(sm + C::kOffY + slot * kSS * C::YS * 4);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        ys[(8 * nt + 2 * c4 + (r & 1)) * C::YS + 16 * w + g + 8 * (r >> 1)] = rq[nt][r];
                warp_arrive(&R.yfull[slot], lane);
            }
            // This block's update into the running weights; then the stage is free.
            {
                const uint32_t sK = smem_u32(stg + C::kOffKh);
#pragma unroll
                for (int j = 0; j < MT; ++j) {
                    uint32_t bt[4];
                    ldsm_x4_t(bt, sK + swz(rt, 2 * j + ct));
                    mma16816(Wa[2 * j], af, bt[0], bt[1]);
                    mma16816(Wa[2 * j + 1], af, bt[2], bt[3]);
                }
                auto hsum = [](uint32_t v) {
                    return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu))) +
                           __half2float(__ushort_as_half((unsigned short)(v >> 16)));
                };
                float s0 = hsum(af[0]) + hsum(af[2]), s1r = hsum(af[1]) + hsum(af[3]);
                s0 += __shfl_xor_sync(kFull, s0, 1);
                s0 += __shfl_xor_sync(kFull, s0, 2);
                s1r += __shfl_xor_sync(kFull, s1r, 1);
                s1r += __shfl_xor_sync(kFull, s1r, 2);
                cb[0] += s0;
                cb[1] += s1r;
            }
            warp_arrive(&R.empty[st], lane);
        }
        set_anchor();  // W_i: the next mini-batch's anchor
    }
    if (!state_written) write_state();
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
        const int slot = i & 1, st = i % C::kStages;
        uint8_t *stg = stage_ptr<D>(sm, st);
        if (o == 0) TTT_TRACE_AT(p, i, 8);
        if (!wait_bar(&R.yfull[slot], parity_of(i >> 1), R.flags) ||
            !wait_bar(&R.prep[st], parity_of(i / C::kStages), R.flags) ||
            !wait_bar(&R.full[st], parity_of(i / C::kStages), R.flags)) {
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
            const uint2 qb = *reinterpret_cast<const uint2 *>(stg + C::offQ(p) + off);  // bf16
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

// ------------------------------------------------------------------ chain/weight split (D = 64)
constexpr int kBarRed = 1;  // C warps: one reduction round
constexpr int kBarA0 = 2;   // A~_i ready (C -> T), ids 2 and 3 by i & 1
constexpr int kBarS0 = 4;   // S_k ready (T -> C), ids 4 and 5 by k & 1

// The chain runs on NC warps (4 in the one-CTA kernel, 2 in the chain CTA of
// the cluster kernel). Chain warp c holds Y_i for output features
// 16 CB c .. 16 CB (c + 1) - 1 as CB = MT / NC blocks of 16 (block w = CB c + bk
// in the weight warps' numbering) with the tokens on the mma M axis: lane
// (g, c4) has tokens g, g+8 and features 16w + 8nt + 2c4 + e, so a token's sums
// over the warp's features need 4 CB in-register terms and two shuffle levels
// (which also split the ten sums of a lane's two tokens over the four lanes of
// its quad: eight shuffles), and one exchange through shared memory completes
// them. Every lane then reads every chain warp's totals of both its tokens, in
// the same order in every warp, and forms their statistics itself.
// SEND (cluster kernel): every step's A~ also goes to the output CTA (rank 1)
// through its ring of kNA slots, each 16-byte piece by st.async completing on
// that CTA's afull[slot]; a slot is written again only after the output CTA
// has released it (aempty[slot] here).
template <int D, int SUBB, int NC, bool SEND = false>
__device__ void role_chain_split(const LinearParams &p, uint8_t *sm, const Ring &R, int c, int hi, size_t tok0,
                                 int lane, int nsteps)
{
    using C = Cfg<D>;
    constexpr int MT = C::MT, NSUB = kSS / SUBB;
    constexpr int CB = MT / NC;
    constexpr int kNAS = (NC + MT) * 32;  // chain and weight warps
    static_assert(CB * NC == MT, "the chain warps cover the weight warps' row blocks");
    const int g = lane >> 2, c4 = lane & 3;
    float gam[CB][2][2], bet[CB][2][2], gg2[CB][2][2];
#pragma unroll
    for (int bk = 0; bk < CB; ++bk)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int f = 16 * (CB * c + bk) + 8 * nt + 2 * c4 + e;
                gam[bk][nt][e] = p.ln_g[hi * D + f];
                bet[bk][nt][e] = p.ln_b[hi * D + f];
                gg2[bk][nt][e] = gam[bk][nt][e] * gam[bk][nt][e];
            }
    float gam2all = 0.f;  // sum of gamma^2 over all features
#pragma unroll
    for (int q = 0; q < D / 32; ++q) gam2all = fmaf(p.ln_g[hi * D + lane + 32 * q], p.ln_g[hi * D + lane + 32 * q], gam2all);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gam2all += __shfl_xor_sync(kFull, gam2all, o);
    const float invD = 1.f / (float)D, eps = p.eps;
    const int T = p.T;
    const float *SR = reinterpret_cast<const float *>(sm + C::kOffSR);
    uint4 *AR = reinterpret_cast<uint4 *>(sm + C::kOffAR);
    float yk[CB][2][4];  // [bk][nt][r]: token g + 8(r>>1), feature 16(CB c + bk) + 8nt + 2c4 + (r&1)
    auto load_s = [&](int slot) {
#pragma unroll
        for (int bk = 0; bk < CB; ++bk) {
            const float *blk = SR + (slot * MT + CB * c + bk) * 16 * C::SRS;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float2 v = *reinterpret_cast<const float2 *>(blk + (g + 8 * u) * C::SRS + 8 * nt + 2 * c4);
                    yk[bk][nt][2 * u] = v.x;
                    yk[bk][nt][2 * u + 1] = v.y;
                }
        }
    };
    // The per-step inputs of the chain (k - v + beta, the learning rates, the
    // per-token scalars of the loader). Stage i is read only after the weight
    // warps have handed S_i over (they waited for the stage first), so these
    // loads for step i + 1 are issued while the chain waits for S_{i+1}.
    float kv[CB][2][4], escale[2], shv[2], pkv[2], qkv[2];
    auto load_in = [&](const uint8_t *stg) {
#pragma unroll
        for (int bk = 0; bk < CB; ++bk)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int t = g + 8 * u, f = 16 * (CB * c + bk) + 8 * nt + 2 * c4;
                    const uint32_t off = swz(t, f >> 3) + (f & 7) * 2;
                    const uint32_t kb = *reinterpret_cast<const uint32_t *>(stg + C::kOffK + off);
                    const uint32_t vb = *reinterpret_cast<const uint32_t *>(stg + C::kOffV + off);
                    kv[bk][nt][2 * u] = bf16_bits_to_f32(kb & 0xffffu) - bf16_bits_to_f32(vb & 0xffffu) + bet[bk][nt][0];
                    kv[bk][nt][2 * u + 1] = bf16_bits_to_f32(kb >> 16) - bf16_bits_to_f32(vb >> 16) + bet[bk][nt][1];
                }
        const float *ssh = reinterpret_cast<const float *>(stg + C::kOffSh);
        const float *se = reinterpret_cast<const float *>(stg + C::kOffEta);
        const float *spk = reinterpret_cast<const float *>(stg + C::kOffPk);
        const float *sqk = reinterpret_cast<const float *>(stg + C::kOffQk);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            escale[u] = -se[g + 8 * u] * (1.f / (float)SUBB);
            shv[u] = ssh[g + 8 * u];
            pkv[u] = spk[g + 8 * u];
            qkv[u] = sqk[g + 8 * u];
        }
    };
    int rnd = 0;
    named_bar_sync(kBarS0, kNAS);  // Y_0 = W_0 K_0^T + c_0 from the T warps
    load_s(0);
    load_in(stage_ptr<D>(sm, 0));
    for (int i = 0; i < nsteps; ++i) {
        const int st = i % C::kStages, stn = (i + 1) % C::kStages;
        const bool has_next = i + 1 < nsteps;
        uint8_t *stg = stage_ptr<D>(sm, st);
        uint8_t *stgn = stage_ptr<D>(sm, stn);
        if (c == 0) TTT_TRACE_AT(p, i, 0);
        float at[CB][2][4] = {}, lin[2] = {};
#pragma unroll
        for (int m = 0; m < NSUB; ++m) {
            // this warp's shifted sums over its 32 features, per token (u)
            float q[2][5];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float a1 = 0.f, a2 = 0.f, ab = 0.f, ac = 0.f, ad = 0.f;
#pragma unroll
                for (int bk = 0; bk < CB; ++bk)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float dv = yk[bk][nt][2 * u + e] - shv[u];
                            const float g2d = gg2[bk][nt][e] * dv;
                            a1 += dv;
                            a2 = fmaf(dv, dv, a2);
                            ab += g2d;
                            ac = fmaf(g2d, dv, ac);
                            ad = fmaf(gam[bk][nt][e] * kv[bk][nt][2 * u + e], dv, ad);
                        }
                q[u][0] = a1;
                q[u][1] = a2;
                q[u][2] = ab;
                q[u][3] = ac;
                q[u][4] = ad;
            }
            if (c == 0 && m == 0) TTT_TRACE_AT(p, i, 1);
            // Sum the ten values over the four lanes (c4) that share g, the lanes splitting
            // the work as they go: at the first level lane bit 0 picks the token (u = c4 & 1),
            // at the second lane bit 1 picks sums 0-2 or 3-4. Eight shuffles instead of twenty;
            // each lane then holds two or three of the warp's ten totals.
            const int b0 = c4 & 1, b1 = c4 >> 1;
            float hq[5];
#pragma unroll
            for (int k = 0; k < 5; ++k)
                hq[k] = (b0 ? q[1][k] : q[0][k]) + __shfl_xor_sync(kFull, b0 ? q[0][k] : q[1][k], 1);
            const float x0 = __shfl_xor_sync(kFull, b1 ? hq[0] : hq[3], 2);
            const float x1 = __shfl_xor_sync(kFull, b1 ? hq[1] : hq[4], 2);
            const float x2 = __shfl_xor_sync(kFull, hq[2], 2);
            const float r0 = (b1 ? hq[3] : hq[0]) + x0;  // sum 0 (b1 = 0) or 3 (b1 = 1) of token g + 8 b0
            const float r1 = (b1 ? hq[4] : hq[1]) + x1;  // sum 1 or 4
            const float r2 = hq[2] + x2;                 // sum 2 (b1 = 0 lanes)
            if (c == 0 && m == 0) TTT_TRACE_AT(p, i, 15);
            const int buf = rnd & 1;
            float4 *redX = reinterpret_cast<float4 *>(sm + C::kOffRedX) + buf * NC * kSS;
            float *redY = reinterpret_cast<float *>(sm + C::kOffRedY) + buf * NC * kSS;
            {
                const int t = g + 8 * b0;
                float *rx = reinterpret_cast<float *>(redX + c * kSS + t);
                if (b1 == 0) {
                    rx[0] = r0;
                    rx[1] = r1;
                    rx[2] = r2;
                } else {
                    rx[3] = r0;
                    redY[c * kSS + t] = r1;
                }
            }
            named_bar_sync(kBarRed, NC * 32);
            ++rnd;
            if (c == 0 && m == 0) TTT_TRACE_AT(p, i, 2);
            float mu[2], rsv[2], rsE[2], cst[2], M2v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                // every chain warp's sums of this token, added in the same order in every warp
                float S1 = 0.f, S2 = 0.f, SB = 0.f, SC = 0.f, SD = 0.f;
#pragma unroll
                for (int src = 0; src < NC; ++src) {
                    const float4 x = redX[src * kSS + g + 8 * u];
                    S1 += x.x;
                    S2 += x.y;
                    SB += x.z;
                    SC += x.w;
                    SD += redY[src * kSS + g + 8 * u];
                }
                const float ee = S1 * invD;
                const float syy = fmaxf(fmaf(-ee, S1, S2), 0.f);
                const float rs = rsqrtf(syy * invD + eps);
                const float sg1 = fmaf(-ee, gam2all, SB);
                const float sg2 = fmaf(ee * ee, gam2all, fmaf(-2.f * ee, SB, SC));
                const float sgk = fmaf(-ee, pkv[u], SD);
                const float M1 = 2.f * invD * fmaf(rs, sg1, pkv[u]);
                M2v[u] = 2.f * invD * rs * fmaf(rs, sg2, sgk);
                const bool in_m = NSUB == 1 || (g + 8 * u) / SUBB == m;
                if (in_m) lin[u] = fmaf(rs, fmaf(rs, sg2, 2.f * sgk), qkv[u]);
                mu[u] = shv[u] + ee;
                rsv[u] = rs;
                rsE[u] = rs * escale[u];   // a~ = rs escale (2 gamma E - M1 - yh M2)
                cst[u] = -rsE[u] * M1;
            }
            if (c == 0 && m == 0) TTT_TRACE_AT(p, i, 12);
            float ad[CB][2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const bool in_m = NSUB == 1 || (g + 8 * u) / SUBB == m;
#pragma unroll
                for (int bk = 0; bk < CB; ++bk)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int r = 2 * u + e;
                            const float yh = (yk[bk][nt][r] - mu[u]) * rsv[u];
                            const float E = fmaf(gam[bk][nt][e], yh, kv[bk][nt][r]);
                            const float t2 = fmaf(-M2v[u], yh, 2.f * gam[bk][nt][e] * E);
                            const float a = round_h(fmaf(rsE[u], t2, cst[u]));
                            ad[bk][nt][r] = in_m ? a : 0.f;
                            if (in_m) at[bk][nt][r] = a;
                        }
            }
            if (c == 0 && m == 0) TTT_TRACE_AT(p, i, 13);
            if (NSUB > 1 && m + 1 < NSUB) {
                // Later mini-batches of this super-step see this one's update:
                // Y[t][f] += sum_{s in mini-batch m} (k_s . k_t + 1) A~[f][s].
                const uint4 gk = reinterpret_cast<const uint4 *>(stg + C::kOffGkA)[lane];
                const uint32_t ga[4] = {gk.x, gk.y, gk.z, gk.w};
#pragma unroll
                for (int bk = 0; bk < CB; ++bk) {
                    const uint32_t d00 = movm_t(pack_h2(ad[bk][0][0], ad[bk][0][1]));
                    const uint32_t d01 = movm_t(pack_h2(ad[bk][0][2], ad[bk][0][3]));
                    const uint32_t d10 = movm_t(pack_h2(ad[bk][1][0], ad[bk][1][1]));
                    const uint32_t d11 = movm_t(pack_h2(ad[bk][1][2], ad[bk][1][3]));
                    mma16816(yk[bk][0], ga, d00, d01);
                    mma16816(yk[bk][1], ga, d10, d11);
                }
            }
        }
        // A~ in the T warps' layout (rows f, columns t): four 8x8 transposes per block.
        uint32_t af[CB][4];
#pragma unroll
        for (int bk = 0; bk < CB; ++bk) {
            af[bk][0] = movm_t(pack_h2(at[bk][0][0], at[bk][0][1]));
            af[bk][1] = movm_t(pack_h2(at[bk][1][0], at[bk][1][1]));
            af[bk][2] = movm_t(pack_h2(at[bk][0][2], at[bk][0][3]));
            af[bk][3] = movm_t(pack_h2(at[bk][1][2], at[bk][1][3]));
            AR[((i & 1) * MT + CB * c + bk) * 32 + lane] = make_uint4(af[bk][0], af[bk][1], af[bk][2], af[bk][3]);
        }
        named_bar_arrive(kBarA0 + (i & 1), kNAS);
        if constexpr (SEND) {
            const int k = i % C::kNA;
            if (i >= C::kNA && !wait_bar_cluster(&R.aempty[k], parity_of(i / C::kNA - 1), R.flags))
                abort_chain(R.flags, p.status);  // keep going in step (results discarded)
            const uint4 *ar1 = reinterpret_cast<const uint4 *>(sm + C::kOffAR1);
            const uint32_t rbar = map_shared(smem_u32(&R.afull[k]), 1);
#pragma unroll
            for (int bk = 0; bk < CB; ++bk)
                st_async_v4(map_shared(smem_u32(ar1 + (k * MT + CB * c + bk) * 32 + lane), 1),
                            make_uint4(af[bk][0], af[bk][1], af[bk][2], af[bk][3]), rbar);
        }
        if (c == 0) TTT_TRACE_AT(p, i, 3);
        warp_arrive(&R.empty[st], lane);  // before the global stores: a release need not wait for them
        if (p.inner_loss && c == 0 && c4 == 0) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = i * kSS + g + 8 * u;
                if (t < T) p.inner_loss[tok0 + t] = lin[u];
            }
        }
        if (has_next) {
            // Y_{i+1} = S_{i+1} + (K_{i+1} K_i^T + 1) A~_i^T
            named_bar_sync(kBarS0 + ((i + 1) & 1), kNAS);
            if (c == 0) TTT_TRACE_AT(p, i, 11);
            load_in(stgn);
            load_s((i + 1) & 1);
            const uint4 kx = reinterpret_cast<const uint4 *>(stgn + C::kOffKxA)[lane];
            const uint32_t xa[4] = {kx.x, kx.y, kx.z, kx.w};
#pragma unroll
            for (int bk = 0; bk < CB; ++bk) {
                mma16816(yk[bk][0], xa, af[bk][0], af[bk][2]);
                mma16816(yk[bk][1], xa, af[bk][1], af[bk][3]);
            }
            if (c == 0) TTT_TRACE_AT(p, i, 4);
        }
    }
}

// MODE kWFull: W, c, S and the output products Rq, Yq (one-CTA kernel).
// MODE kWChain: W, c and S only (cluster kernel, chain CTA).
// MODE kWOut: a copy of W, c (the same products on the same operands, so the
// two copies agree bit for bit) and Rq, Yq, with each step's A~ from the
// chain CTA's ring (cluster kernel, output CTA); writes no final state.
constexpr int kWFull = 0, kWChain = 1, kWOut = 2;

template <int D, int NC, int MODE = kWFull>
__device__ void role_weights_split(const LinearParams &p, uint8_t *sm, const Ring &R, int w, int chain, int bi, int hi,
                                   int lane, int nsteps)
{
    using C = Cfg<D>;
    constexpr int MT = C::MT, NTW = D / 8;
    constexpr int kNAS = (NC + MT) * 32;  // chain and weight warps
    const int g = lane >> 2, c4 = lane & 3;
    const int r0 = 16 * w + g, r1 = r0 + 8;
    const float *W0 = p.W0 + bi * p.w0_bstride + (long long)hi * D * D;
    const float *c0 = p.c0 + bi * p.c0_bstride + (long long)hi * D;
    float Wa[NTW][4];
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
    const int rt = (lane & 7) + ((lane >> 3) & 1) * 8, ct = lane >> 4;
    float *SR = reinterpret_cast<float *>(sm + C::kOffSR);
    const uint4 *AR = reinterpret_cast<const uint4 *>(sm + C::kOffAR);
    auto wait_stage = [&](int k) {
        if (!wait_bar(&R.full[k % C::kStages], parity_of(k / C::kStages), R.flags) ||
            !wait_bar(&R.prep[k % C::kStages], parity_of(k / C::kStages), R.flags))
            abort_chain(R.flags, p.status);  // keep going in step with the chain warps
    };
    auto store_s = [&](int k, const float (&acc)[2][4]) {  // S_k (this warp's rows) -> the chain warps
        float *blk = SR + ((k & 1) * MT + w) * 16 * C::SRS;  // [t][f - 16w], the chain warps' order
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) blk[(8 * nt + 2 * c4 + (r & 1)) * C::SRS + g + 8 * (r >> 1)] = acc[nt][r];
        named_bar_arrive(kBarS0 + (k & 1), kNAS);
    };
    auto publish_s = [&](int k) {  // S_k = W K_k^T + c
        float acc[2][4];
        rows_gemm<D>(Wa, cb, smem_u32(stage_ptr<D>(sm, k % C::kStages) + C::kOffKh), lane, acc);
        store_s(k, acc);
    };
    const uint4 *AR1 = reinterpret_cast<const uint4 *>(sm + C::kOffAR1);
    wait_stage(0);
    if (MODE != kWOut) {
        publish_s(0);
        if (nsteps > 1) {
            wait_stage(1);
            publish_s(1);
        }
    }
    float Rq[2][4];
    if (MODE != kWChain) rows_gemm<D>(Wa, cb, smem_u32(stage_ptr<D>(sm, 0) + C::offQh(p)), lane, Rq);
    for (int j = 0; j < nsteps; ++j) {
        const int st = j % C::kStages, slot = j & 1;
        uint8_t *stg = stage_ptr<D>(sm, st);
        uint4 a;
        if (MODE == kWOut) {
            // this step's A~ from the chain CTA: 2 KB of st.async into ring slot k
            const int k = j % C::kNA;
            if (w == 0 && lane == 0) mbar_arrive_expect_tx(&R.afull[k], C::MT * 512);
            if (!wait_bar_cluster(&R.afull[k], parity_of(j / C::kNA), R.flags)) abort_chain(R.flags, p.status);
            a = AR1[(k * MT + w) * 32 + lane];
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(map_shared(smem_u32(&R.aempty[k]), 0));  // slot k read
        } else {
            named_bar_sync(kBarA0 + slot, kNAS);
            a = AR[(slot * MT + w) * 32 + lane];
        }
        if (w == 0) TTT_TRACE_AT(p, j, 5);
        const uint32_t af[4] = {a.x, a.y, a.z, a.w};
        // W_{j-1} -> W_j, c_{j-1} -> c_j over the committed tokens of the super-step
        uint32_t au[4] = {a.x, a.y, a.z, a.w};
        mask_tokens(au, committed_in_step(p.t_commit, j), lane);
        {
            const uint32_t sK = smem_u32(stg + C::kOffKh);
#pragma unroll
            for (int jj = 0; jj < MT; ++jj) {
                uint32_t bt[4];
                ldsm_x4_t(bt, sK + swz(rt, 2 * jj + ct));
                mma16816(Wa[2 * jj], au, bt[0], bt[1]);
                mma16816(Wa[2 * jj + 1], au, bt[2], bt[3]);
            }
        }
        auto hsum = [](uint32_t v) {
            return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu))) +
                   __half2float(__ushort_as_half((unsigned short)(v >> 16)));
        };
        float s0 = hsum(au[0]) + hsum(au[2]), s1 = hsum(au[1]) + hsum(au[3]);
        s0 += __shfl_xor_sync(kFull, s0, 1);
        s0 += __shfl_xor_sync(kFull, s0, 2);
        s1 += __shfl_xor_sync(kFull, s1, 1);
        s1 += __shfl_xor_sync(kFull, s1, 2);
        cb[0] += s0;
        cb[1] += s1;
        if (MODE != kWChain) {
            // Yq_j^T = Rq_j^T + A~_j Mq_j -> output warps
            {
                const uint4 mq = reinterpret_cast<const uint4 *>(stg + C::kOffMq)[lane];
                mma16816(Rq[0], af, mq.x, mq.y);
                mma16816(Rq[1], af, mq.z, mq.w);
            }
            if (!wait_bar(&R.yempty[slot], parity_of(j >> 1) ^ 1u, R.flags)) abort_chain(R.flags, p.status);
            float *ys = reinterpret_cast<float *>(sm + C::kOffY + slot * kSS * C::YS * 4);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    ys[(8 * nt + 2 * c4 + (r & 1)) * C::YS + 16 * w + g + 8 * (r >> 1)] = Rq[nt][r];
            warp_arrive(&R.yfull[slot], lane);
        }
        if (w == 0) TTT_TRACE_AT(p, j, 6);
        if (MODE == kWFull) {
            // S_{j+2} = W_j K_{j+2}^T + c_j and Rq_{j+1} = W_j Q_{j+1}^T + c_j (stage j+1 was
            // waited for one step earlier), in one pass over W_j.
            if (j + 2 < nsteps) {
                wait_stage(j + 2);
                float acc[2][4];
                rows_gemm2<D>(Wa, cb, smem_u32(stage_ptr<D>(sm, (j + 2) % C::kStages) + C::kOffKh),
                              smem_u32(stage_ptr<D>(sm, (j + 1) % C::kStages) + C::offQh(p)), lane, acc, Rq);
                store_s(j + 2, acc);
            } else if (j + 1 < nsteps) {
                rows_gemm<D>(Wa, cb, smem_u32(stage_ptr<D>(sm, (j + 1) % C::kStages) + C::offQh(p)), lane, Rq);
            }
        } else if (MODE == kWChain) {
            if (j + 2 < nsteps) {  // S_{j+2} = W_j K_{j+2}^T + c_j
                wait_stage(j + 2);
                float acc[2][4];
                rows_gemm<D>(Wa, cb, smem_u32(stage_ptr<D>(sm, (j + 2) % C::kStages) + C::kOffKh), lane, acc);
                store_s(j + 2, acc);
            }
        } else {
            if (j + 1 < nsteps) {  // Rq_{j+1} = W_j Q_{j+1}^T + c_j
                wait_stage(j + 1);
                rows_gemm<D>(Wa, cb, smem_u32(stage_ptr<D>(sm, (j + 1) % C::kStages) + C::offQh(p)), lane, Rq);
            }
        }
        if (w == 0) TTT_TRACE_AT(p, j, 7);
        warp_arrive(&R.empty[st], lane);
    }
    if (MODE == kWOut) return;  // the chain CTA writes the final state
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

template <int D, int SUBB>
__global__ void __launch_bounds__(Cfg<D>::kSplitThreads, 1)
linear_tc_split_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const LinearParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chain = blockIdx.x;
    const int bi = chain / p.H, hi = chain % p.H;
    const int nsteps = (p.T + kSS - 1) / kSS;
    const size_t tok0 = (size_t)chain * p.T;

    Ring R;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + C::kOffBar);
    R.full = bar;
    R.prep = bar + C::kStages;
    R.empty = bar + 2 * C::kStages;
    R.yfull = bar + 3 * C::kStages;
    R.yempty = R.yfull + 2;
    R.red = R.yfull + 4;
    R.flags = reinterpret_cast<volatile int *>(bar + C::kNumBars);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&R.full[s], 33);                      // expect_tx arrive + 32 cp.async arrivals
            mbar_init(&R.prep[s], kLoaderPrep<D> ? 2 : 1);  // P (and L)
            mbar_init(&R.empty[s], 2 * C::MT + C::NO + 1);  // C warps, T warps, O warps, P
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&R.yfull[j], C::MT);
            mbar_init(&R.yempty[j], C::NO);
            mbar_init(&R.red[j], C::MT);
        }
        R.flags[0] = 0;
        R.flags[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (nsteps == 0) return;

    if (warp == C::kWarpL) {
        role_loader_sums<D>(&tmQ, &tmK, &tmV, p, sm, R, chain, bi, hi, lane, nsteps);
    } else if (warp == C::kWarpP) {
        role_prep<D, SUBB>(p, sm, R, bi, hi, lane, nsteps);
    } else if (warp < C::kSplitWarpT) {
        role_chain_split<D, SUBB, C::MT>(p, sm, R, warp - C::kSplitWarpC, hi, tok0, lane, nsteps);
    } else if (warp < C::kSplitWarpO) {
        role_weights_split<D, C::MT>(p, sm, R, warp - C::kSplitWarpT, chain, bi, hi, lane, nsteps);
    } else {
        role_output<D>(p, sm, R, warp - C::kSplitWarpO, chain, hi, tok0, lane, nsteps);
    }
}

// ------------------------------------------------------------------ cluster kernel (d = 64, b = 16)
// One chain over a cluster of two CTAs on two SMs, for workloads with fewer
// chains than half the SMs (few heads, long sequences). The chain's serial
// loop is latency-bound and slows down whenever other warps compete for its
// scheduler partitions, so the work is split by role:
//   rank 0, the chain CTA: the chain (2 warps, alone on partitions 0 and 1),
//     W and c with S_{i+2} (4 weight warps, partitions 2 and 3), the loader
//     of K, V, eta with the per-token scalars, and the prep warp (fp16 K copy,
//     K_{i-1} K_i^T); it writes inner_loss and the final state;
//   rank 1, the output CTA: a copy of W and c kept in step by each A~_i that
//     the chain CTA sends through distributed shared memory (one way, ahead of
//     its use, so off the chain's loop), Rq and Yq, the output LayerNorm,
//     Z and L_t, with its own loads of Q, K, V, eta and its own Q K^T.
// Warps 4, 5, 8, 9 of rank 0 and 8..11 of rank 1 have no role.
template <int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<D>::kSplitThreads, 1)
linear_tc_cluster_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const LinearParams p)
{
    using C = Cfg<D>;
    static_assert(C::kSplitWarps == 12, "warp map below");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_ctarank();
    const int chain = blockIdx.x >> 1;
    const int bi = chain / p.H, hi = chain % p.H;
    const int nsteps = (p.T + kSS - 1) / kSS;
    const size_t tok0 = (size_t)chain * p.T;

    Ring R;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + C::kOffBar);
    R.full = bar;
    R.prep = bar + C::kStages;
    R.empty = bar + 2 * C::kStages;
    R.yfull = bar + 3 * C::kStages;
    R.yempty = R.yfull + 2;
    R.red = R.yfull + 4;
    R.afull = R.yfull + 6;
    R.aempty = R.afull + C::kNA;
    R.flags = reinterpret_cast<volatile int *>(bar + C::kNumBars);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&R.full[s], 33);   // expect_tx arrive + 32 cp.async arrivals
            mbar_init(&R.prep[s], 2);    // P and L
            mbar_init(&R.empty[s], rank == 0 ? 2 + C::MT + 1 : C::MT + C::NO + 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&R.yfull[j], C::MT);
            mbar_init(&R.yempty[j], C::NO);
            mbar_init(&R.red[j], C::MT);
        }
        for (int k = 0; k < C::kNA; ++k) {
            mbar_init(&R.afull[k], 1);       // the expect_tx arrival; the bytes come from rank 0
            mbar_init(&R.aempty[k], C::MT);  // the four weight warps of rank 1, remotely
        }
        R.flags[0] = 0;
        R.flags[1] = 0;
        fence_mbar_init();
    }
    cluster_sync();  // both CTAs' barriers exist before either touches the other
    if (nsteps > 0) {
        if (rank == 0) {
            switch (warp) {
            case 0:
            case 1: role_chain_split<D, kSS, 2, true>(p, sm, R, warp, hi, tok0, lane, nsteps); break;
            case 2: role_weights_split<D, 2, kWChain>(p, sm, R, 0, chain, bi, hi, lane, nsteps); break;
            case 3: role_weights_split<D, 2, kWChain>(p, sm, R, 1, chain, bi, hi, lane, nsteps); break;
            case 6: role_weights_split<D, 2, kWChain>(p, sm, R, 2, chain, bi, hi, lane, nsteps); break;
            case 7: role_weights_split<D, 2, kWChain>(p, sm, R, 3, chain, bi, hi, lane, nsteps); break;
            case 10: role_loader_sums<D, false, true>(&tmQ, &tmK, &tmV, p, sm, R, chain, bi, hi, lane, nsteps); break;
            case 11: role_prep<D, kSS, kPrepKx>(p, sm, R, bi, hi, lane, nsteps); break;
            default: break;
            }
        } else {
            LinearParams po = p;  // the chain CTA writes inner_loss and the final state
            po.inner_loss = nullptr;
            po.W_out = nullptr;
            po.c_out = nullptr;
            switch (warp) {
            case 0:
            case 1:
            case 2:
            case 3: role_weights_split<D, 2, kWOut>(po, sm, R, warp, chain, bi, hi, lane, nsteps); break;
            case 4:
            case 5: role_output<D>(po, sm, R, warp - 4, chain, hi, tok0, lane, nsteps); break;
            case 6: role_loader_sums<D, true, false>(&tmQ, &tmK, &tmV, po, sm, R, chain, bi, hi, lane, nsteps); break;
            case 7: role_prep<D, kSS, kPrepQ | kPrepMq>(po, sm, R, bi, hi, lane, nsteps); break;
            default: break;
            }
        }
    }
    // Neither CTA leaves while the other may still write into its shared
    // memory (A~ pieces into rank 1, slot releases into rank 0).
    cluster_sync();
}

// ------------------------------------------------------------------ kernel
template <int D, int SUBB>
__global__ void __launch_bounds__(Cfg<D>::kThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const LinearParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chain = blockIdx.x;
    const int bi = chain / p.H, hi = chain % p.H;
    const int nsteps = (p.T + kSS - 1) / kSS;
    const size_t tok0 = (size_t)chain * p.T;

    Ring R;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + C::kOffBar);
    R.full = bar;
    R.prep = bar + C::kStages;
    R.empty = bar + 2 * C::kStages;
    R.yfull = bar + 3 * C::kStages;
    R.yempty = R.yfull + 2;
    R.red = R.yfull + 4;
    R.flags = reinterpret_cast<volatile int *>(bar + C::kNumBars);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&R.full[s], 33);                  // expect_tx arrive + 32 cp.async arrivals
            mbar_init(&R.prep[s], kLoaderPrep<D> ? 2 : 1);  // P (and L)
            mbar_init(&R.empty[s], C::MT + C::NO + 1);  // W warps, O warps, P
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&R.yfull[j], C::MT);
            mbar_init(&R.yempty[j], C::NO);
            mbar_init(&R.red[j], C::MT);
        }
        R.flags[0] = 0;
        R.flags[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (nsteps == 0) return;

    if (warp == C::kWarpL) {
        role_loader_sums<D>(&tmQ, &tmK, &tmV, p, sm, R, chain, bi, hi, lane, nsteps);
    } else if (warp == C::kWarpP) {
        role_prep<D, SUBB>(p, sm, R, bi, hi, lane, nsteps);
    } else if (warp < C::kWarpO) {
        if constexpr (SUBB > kSS && SUBB / kSS <= 4)
            role_weights_mb2<D, SUBB / kSS>(p, sm, R, warp - C::kWarpW, chain, bi, hi, tok0, lane, nsteps);
        else if constexpr (SUBB > kSS)
            role_weights_mb<D, SUBB / kSS>(p, sm, R, warp - C::kWarpW, chain, bi, hi, tok0, lane, nsteps);
        else
            role_weights<D, SUBB>(p, sm, R, warp - C::kWarpW, chain, bi, hi, tok0, lane, nsteps);
    } else {
        role_output<D>(p, sm, R, warp - C::kWarpO, chain, hi, tok0, lane, nsteps);
    }
}

// ------------------------------------------------------------------ host side
// 0: never (default: measured faster at every chain count), 1: when the
// chains fit half the SMs, 2: always.
std::atomic<int> g_cluster_mode{0};

// The two-CTA form of d = 64, b = 16 (mode 1) runs when every chain gets its
// pair of SMs in one wave (2 * chains <= SMs); otherwise the one-CTA kernel
// keeps a chain per SM.
bool use_cluster_form(int chains)
{
    const int mode = g_cluster_mode.load(std::memory_order_relaxed);
    if (mode == 0) return false;
    if (mode == 2) return true;
    static std::atomic<int> sms[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    int n = sms[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        sms[dev].store(n, std::memory_order_relaxed);
    }
    return 2 * chains <= n;
}

template <int D, int SUBB>
cudaError_t launch_dsub(const LinearParams &p, int chains, cudaStream_t s)
{
    CUtensorMap mQ, mK, mV;
    if (!make_map(&mQ, p.Q, D, p.T, chains, 16) || !make_map(&mK, p.K, D, p.T, chains, 16) ||
        !make_map(&mV, p.V, D, p.T, chains, 16))
        return cudaErrorInvalidValue;
    constexpr int smem = Cfg<D>::kSmemAlloc;
    if constexpr (D == 64 && SUBB == kSS) {
        if (use_cluster_form(chains)) {
            cudaError_t e = ensure_smem<linear_tc_cluster_kernel<D>>(smem);
            if (e != cudaSuccess) return e;
            linear_tc_cluster_kernel<D><<<2 * chains, Cfg<D>::kSplitThreads, smem, s>>>(mQ, mK, mV, p);
            return cudaGetLastError();
        }
    }
    // The chain/weight split: d = 64 for b <= 16; d = 128 for b < 16 only, where the
    // per-mini-batch LayerNorm rounds of a super-step dominate (at b = 16 the one
    // round per super-step runs faster on the merged kernel).
    if constexpr ((D == 64 && SUBB <= kSS) || (D == 128 && SUBB < kSS)) {
        cudaError_t e = ensure_smem<linear_tc_split_kernel<D, SUBB>>(smem);
        if (e != cudaSuccess) return e;
        linear_tc_split_kernel<D, SUBB><<<chains, Cfg<D>::kSplitThreads, smem, s>>>(mQ, mK, mV, p);
    } else {
        cudaError_t e = ensure_smem<linear_tc_kernel<D, SUBB>>(smem);
        if (e != cudaSuccess) return e;
        linear_tc_kernel<D, SUBB><<<chains, Cfg<D>::kThreads, smem, s>>>(mQ, mK, mV, p);
    }
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
    case 32: return launch_dsub<D, 32>(p, chains, s);
    case 64: return launch_dsub<D, 64>(p, chains, s);
    case 128: return launch_dsub<D, 128>(p, chains, s);
    case 256: return launch_dsub<D, 256>(p, chains, s);
    case 512: return launch_dsub<D, 512>(p, chains, s);
    case 1024: return launch_dsub<D, 1024>(p, chains, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool linear_tc_supported(int io, int d, int mb)
{
    // b = 1..16 divides the 16-token super-step; b = 32..1024 spans 2..64 of them
    return io == TTT_BF16 && (d == 64 || d == 128) && mb >= 1 && mb <= 1024 && (mb & (mb - 1)) == 0;
}

int linear_cluster_mode(int mode)
{
    if (mode >= 0 && mode <= 2) g_cluster_mode.store(mode, std::memory_order_relaxed);
    return g_cluster_mode.load(std::memory_order_relaxed);
}

cudaError_t launch_linear_tc(const LinearParams &p, int chains, cudaStream_t s)
{
    if (p.d == 64) return launch_d<64>(p, chains, s);
    if (p.d == 128) return launch_d<128>(p, chains, s);
    return cudaErrorInvalidValue;
}

}  // namespace ttt
