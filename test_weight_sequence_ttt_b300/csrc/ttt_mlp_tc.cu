// ttt_mlp_tc.cu -- TTT-MLP inner loop on tensor cores (sm_103a): d = 64,
// hidden = 256 (4d), mini-batch b = 16, bf16 Q/K/V.
//
// Method: the TTT-MLP of the "TTT layer" section of the "Test-Time
// Training(TTT)과 LLM 메모리" survey page (f_res(x) = W2 gelu_tanh(W1 x + c1)
// + c2, f(x) = x + LN(f_res(x)), Eq. 2 update, Eq. 4 loss, Eq. 5 output),
// trained by the mini-batch rule of Eq. 5 of the "End-to-End Test-Time Training
// for Long Context" review (section 2.3): every gradient of mini-batch i at the
// anchor (W1, W2) = (W1_{i-1}, W2_{i-1}), weight 1/b, and z_t read with the
// in-batch prefix of the updates. Per mini-batch (K, Q, V: 16 x d):
//   Z1 = K W1^T + c1, X2 = gelu(Z1), Y = X2 W2^T + c2               (anchor)
//   G = dl/dY through x + LN(y);  G1 = (G W2) * gelu'(Z1)
//   Z1q = Q W1^T + c1 + A~1^T Mq1,   A~1 = -(eta/b) G1, Mq1 = causal q.k + 1
//   Yq = gelu(Z1q) W2^T + c2 + A~2^T Mq2, A~2 = -(eta/b) G, Mq2 = causal x2q.x2k + 1
//   Z = Q + LN(Yq);  W1 += A~1^T K, c1 += A~1^T 1;  W2 += A~2^T X2, c2 += A~2^T 1
//
// One CTA per (sequence, head) chain. Warp roles:
//   L (1)  TMA loader of the Q/K/V tiles and eta (shared with TTT-Linear).
//   P (1)  the learning-rate gate (eta_gate); fp16 copies of the K/Q tiles;
//          causal Q K^T + 1 and K_{i-1} K_i^T + 1 fragments; two steps behind,
//          the output side: the X2q X2k^T Gram (causal + 1 fragments for the Y
//          warps) and Z = Q + LN(Yq), L_t with the Z stores.
//   H (8)  warp w owns hidden units 32w..32w+31: W1 rows and c1 in registers
//          (fp32 mma accumulators), W2 columns as an fp32 master in tensor
//          memory (tcgen05.ld / tcgen05.st around each update) plus the fp16
//          copy of W2 in shared memory that every product reads. Computes Z1,
//          gelu, G1, Z1q and the W1 / W2 updates.
//   Y (2)  warp y owns output features 32y..32y+31 and c2: Y, the LayerNorm
//          forward/backward (both Y warps, through shared memory), G and, one
//          step later, Yq = X2q W2^T + c2 + A~2^T Mq2, handed to P.
// Look-ahead. The recurrence of one step is A~1_i -> Z1 of step i+1 ->
// gelu -> Y of step i+1 -> LayerNorm backward -> G -> A~1_{i+1}. Neither
// weight update sits on it:
//   Z1_{i+1}^T = (W1_{i-1} K_{i+1}^T + c1_{i-1}) + A~1_i (K_i K_{i+1}^T + 1)
//   Y_{i+1}^T  = (W2_{i-1} X2_{i+1}^T + c2_{i-1}) + A~2_i (X2_i X2_{i+1}^T + 1)
// (exact in real arithmetic), so the H warps apply W1 += A~1 K and the
// tensor-memory W2 update while the Y warps already work on the next step;
// three fp16 copies of W2 (W2_j in buffer j % 3) keep every reader's version.
// H and Y hand activations over through shared memory with named barriers
// (producer bar.arrive, consumer bar.sync). No warp leaves early: after a
// failed wait a warp keeps running in step with the others (its results are
// discarded, the status word says why), so every barrier is always met.
//
// Cluster form (few chains): one chain over a cluster of two CTAs, CTA r owning
// hidden units 128r..128r+127 (W1 rows, c1, W2 columns; eight H warps of 16 units
// each, against 32 in the one-CTA form, so the issue slots still have three warps
// per partition to pick from). Every contraction over the hidden units is then
// a sum of the two CTAs' partials:
//   - Y of the recurrence: each CTA's Y warps send their partial (the A~2 Gram
//     term included) to the other CTA through distributed shared memory
//     (st.async, completion counted on the receiver's mbarrier) and add the
//     one they receive; both CTAs then run the same LayerNorm backward, so G,
//     A~2 and c2 are bitwise the same in both (fp32 addition commutes).
//   - Yq of the outputs: CTA 1 sends its partial (and its part of the X2q X2k^T
//     Gram, through A~2) to CTA 0, whose P warp adds it and writes Z; P releases
//     the slot with a remote arrive.
// The K/Q/V tiles are loaded by both CTAs; the d-wide Grams are built in both.
//
// Precision: fp16 MMA operands (W1, W2, K, Q, X2, G, A~) with fp32
// accumulation; W1, W2, c1, c2, LayerNorm statistics and gradients fp32. GELU
// uses the hardware tanh approximation.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_common.cuh"

namespace ttt {
namespace {

using namespace tc;

constexpr int kD = 64, kHid = 256, kB = 16;
constexpr int kNY = 2;  // Y warps, 32 output features each
constexpr int kWarpL = 0, kWarpP = 1, kWarpH = 2;
constexpr int kStages = 5;
// stage layout (bytes)
constexpr int kTile = 32 * kD;
constexpr int kOffK = 0, kOffQ = kTile, kOffV = 2 * kTile;  // bf16, as loaded
constexpr int kOffKh = 3 * kTile, kOffQh = 4 * kTile;      // fp16 copies (same swizzled layout)
constexpr int kOffMq = 5 * kTile;                          // causal q.k + 1, fp16 B fragments
constexpr int kOffKx = kOffMq + 512;                       // k_{i-1}.k_i + 1, fp16 B fragments
constexpr int kOffEta = kOffKx + 512;
constexpr int kStageBytes = ((kOffEta + 64 + 1023) / 1024) * 1024;
constexpr int kFS = kD + 8;  // halves per row of a [16][d] fp16 buffer (rows padded by 16 bytes)
constexpr int kOffStages = 0;
constexpr int kGBytes = kB * kFS * 2;
constexpr int kYS = kD + 4;  // floats per row of the Yq hand-off
constexpr uint32_t kTmemCols = 128;  // two H warps per lane quarter x 64 columns
// named barriers: H <-> Y hand-offs (all H and Y threads), Y-internal rounds
constexpr int kBarX2k = 1, kBarG = 2, kBarX2q = 3 /* and 4, by step parity */, kBarYln = 5;
// Every mbarrier wait of this kernel polls without suspending the thread: the
// waits on the recurrence (the Y exchange, the H/Y hand-offs) then resume as
// soon as their phase completes, which measured faster than letting the
// hardware suspend the waiting warps.
constexpr bool kSpinWaits = true;

// Warps and shared memory of a CTA that owns kHid / NR hidden units: the whole
// chain (NR = 1) or one half of it in a two-CTA cluster (NR = 2).
template <int NR>
struct Lay {
    static constexpr int kHidL = kHid / NR;  // hidden units of this CTA
    static constexpr int kMH = NR == 1 ? 2 : 1;  // 16-unit row blocks per H warp
    static constexpr int kHW = 16 * kMH;         // hidden units per H warp
    static constexpr int kNH = kHidL / kHW;      // H warps
    static constexpr int kWarpY = kWarpH + kNH;
    static constexpr int kWarps = kWarpY + kNY;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kHY = (kNH + kNY) * 32;
    // fp16 activation / weight buffers, rows padded by 16 bytes (conflict-free ldmatrix)
    static constexpr int kHS = kHidL + 8;                    // halves per row of a [*][hidden] buffer
    static constexpr int kW2hBytes = kD * kHS * 2;           // one fp16 copy of W2, [d][kHS]
    static constexpr int kOffW2h = kStages * kStageBytes;    // 3 copies: W2_j in buffer j % 3
    static constexpr int kX2Bytes = kB * kHS * 2;            // one [16][kHS] fp16 activation tile
    static constexpr int kOffX2k = kOffW2h + 3 * kW2hBytes;  // 3 x gelu(Z1) of the keys, step j in j % 3
    static constexpr int kOffX2q = kOffX2k + 3 * kX2Bytes;   // 2 x gelu(Z1q), step j in j & 1
    static constexpr int kOffGh = kOffX2q + 2 * kX2Bytes;    // 2 x [16][kFS] G, step j in j & 1
    static constexpr int kOffGt = kOffGh + 2 * kGBytes;      // 2 x [16][kFS] A~2 = -(eta/b) G
    static constexpr int kOffRed = kOffGt + 2 * kGBytes;     // 2 bufs x [2 Y warps][16] float4
    static constexpr int kOffYq = kOffRed + 2 * kNY * kB * 16;  // 2 slots x [16][kYS] fp32 Yq (Y -> P)
    static constexpr int kOffMq2 = kOffYq + 2 * kB * kYS * 4;   // 2 x causal x2q.x2k + 1 fragments (P -> Y)
    // cluster form: the other CTA's Y partial (2 slots x [Y warp][4][32 lanes] float4)
    static constexpr int kOffYp = kOffMq2 + 2 * 512;
    static constexpr int kYpBytes = NR == 2 ? 2 * kNY * 4 * 32 * 16 : 0;
    // cluster form, CTA 0: the other CTA's Yq partial (2 slots x [16][kYS] fp32)
    static constexpr int kOffYqp = kOffYp + kYpBytes;
    static constexpr int kYqpBytes = NR == 2 ? 2 * kB * kYS * 4 : 0;
    static constexpr int kOffTmem = kOffYqp + kYqpBytes;
    static constexpr int kOffBar = kOffTmem + 16;
    static constexpr int kNumBars = 3 * kStages + 8 + (NR == 2 ? 6 : 0);
    static constexpr int kSmem = kOffBar + kNumBars * 8 + 16;
    static constexpr int kSmemAlloc = kSmem + 1024;
    // Warp roles: L 0, P 1, H 2..9, Y 10, 11. A warp issues on scheduler
    // partition warp % 4, and tensor memory lets it reach the lanes of quarter
    // warp % 4 only: H warps w and w + 4 share a quarter, w + 4 taking the
    // columns after w's (16 * kMH x 2 per warp: its W2 columns, 64 features).
    __device__ static int h_index(int warp) { return warp >= kWarpH && warp < kWarpY ? warp - kWarpH : -1; }
    __device__ static int y_index(int warp) { return warp >= kWarpY && warp < kWarps ? warp - kWarpY : -1; }
    __device__ static uint32_t tmem_cols(int w) { return (uint32_t)(32 * kMH * (w / 4)); }
    static constexpr int kYpTx = kNY * 32 * 64;       // bytes of one Y partial
    static constexpr int kYqpTx = kNY * 32 * 16 * 4;  // bytes of one Yq partial
};
constexpr float kGeluA = 0.7978845608028654f;  // sqrt(2/pi)
constexpr float kGeluC = 0.044715f;

// mbarriers: full/prep/empty (stage ring); hq[2] (H -> P: X2q of step j is
// written; by step parity, because the H warps may arrive for step j + 1
// before P has waited for step j, never for step j + 2: that needs G_{j+2},
// which the Y warps hand over only after P's Gram of step j); mq2[2] (P -> Y:
// Gram fragments of step j in buffer j & 1); yqfull/yqempty[2] (Yq hand-off Y <-> P). Cluster form:
// ypeer[2] (the other CTA's Y partial of step j landed, slot j & 1), yqpfull[2]
// (CTA 0: the other CTA's Yq partial landed), yqpempty[2] (CTA 1: CTA 0's P
// has read the slot).
struct Ring {
    uint64_t *full, *prep, *empty, *hq, *mq2, *yqfull, *yqempty, *ypeer, *yqpfull, *yqpempty;
    volatile int *flags;  // [0] abort, [1] fp16 range violation seen
};

__device__ __forceinline__ uint8_t *stage_ptr(uint8_t *sm, int st) { return sm + kOffStages + st * kStageBytes; }

// gelu_tanh(u) and its derivative.
__device__ __forceinline__ void gelu2(float u, float &g, float &gp)
{
    const float th = tanh_fast(kGeluA * fmaf(kGeluC * u * u, u, u));
    g = 0.5f * u * (1.f + th);
    gp = 0.5f * (1.f + th) + 0.5f * u * (1.f - th * th) * kGeluA * fmaf(3.f * kGeluC, u * u, 1.f);
}

__device__ __forceinline__ float gelu1(float u)
{
    const float th = tanh_fast(kGeluA * fmaf(kGeluC * u * u, u, u));
    return 0.5f * u * (1.f + th);
}

// ------------------------------------------------------------------ P: prep and output
__device__ __forceinline__ uint32_t hb(uint32_t base, int row, int col, int stride);

// Step i's input side: fp16 copies of the K/Q tiles, causal Q K^T + 1
// fragments and (i > 0) K_{i-1} K_i^T + 1 fragments for the Z1 look-ahead.
__device__ __forceinline__ void prep_stage(uint8_t *stg, const uint8_t *stg_prev, int lane, uint32_t &mag,
                                           bool prefix, bool q_is_k)
{
    const int g = lane >> 2, c4 = lane & 3;
    const int ra = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int rb = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
    for (int tile = 0; tile < 2; ++tile) {
        if (tile == 1 && q_is_k) break;  // the key tile stands in for the query tile
        const uint4 *src = reinterpret_cast<const uint4 *>(stg + (tile == 0 ? kOffK : kOffQ));
        uint4 *dst = reinterpret_cast<uint4 *>(stg + (tile == 0 ? kOffKh : kOffQh));
#pragma unroll
        for (int ch = lane; ch < 2 * kD; ch += 32) {
            const uint4 x = src[ch];
            mag = __vmaxu2(mag, __vmaxu2(__vmaxu2(x.x & 0x7fff7fffu, x.y & 0x7fff7fffu),
                                         __vmaxu2(x.z & 0x7fff7fffu, x.w & 0x7fff7fffu)));
            dst[ch] = make_uint4(bf2_to_h2(x.x), bf2_to_h2(x.y), bf2_to_h2(x.z), bf2_to_h2(x.w));
        }
    }
    __syncwarp();
    // dq[j][r] = q_t . k_s with t = g + 8(r>>1), s = 8j + 2c4 + (r&1)
    const uint32_t sK = smem_u32(stg + kOffKh), sQ = smem_u32(stg + (q_is_k ? kOffKh : kOffQh));
    float dq[2][4] = {}, dx[2][4] = {};  // dx[j][r] = k_t . k'_s, t in step i, s in step i-1
#pragma unroll
    for (int ks = 0; ks < kD / 16; ++ks) {
        uint32_t aq[4], bk[4];
        ldsm_x4(aq, sQ + swz(ra, 2 * ks + (lane >> 4)));
        ldsm_x4(bk, sK + swz(rb, 2 * ks + ((lane >> 3) & 1)));
        mma16816(dq[0], aq, bk[0], bk[1]);
        mma16816(dq[1], aq, bk[2], bk[3]);
        if (stg_prev) {
            uint32_t ak[4], bp[4];
            ldsm_x4(ak, sK + swz(ra, 2 * ks + (lane >> 4)));
            ldsm_x4(bp, smem_u32(stg_prev + kOffKh) + swz(rb, 2 * ks + ((lane >> 3) & 1)));
            mma16816(dx[0], ak, bp[0], bp[1]);
            mma16816(dx[1], ak, bp[2], bp[3]);
        }
    }
    if (stg_prev)  // B fragments (k = s of step i-1, n = t of step i)
        reinterpret_cast<uint4 *>(stg + kOffKx)[lane] =
            make_uint4(pack_h2(dx[0][0] + 1.f, dx[0][1] + 1.f), pack_h2(dx[1][0] + 1.f, dx[1][1] + 1.f),
                       pack_h2(dx[0][2] + 1.f, dx[0][3] + 1.f), pack_h2(dx[1][2] + 1.f, dx[1][3] + 1.f));
    auto mq = [&](int j, int r) {  // under the anchor rule no update of the batch is seen
        const int t = g + 8 * (r >> 1), s = 8 * j + 2 * c4 + (r & 1);
        return prefix && s <= t ? dq[j][r] + 1.f : 0.f;
    };
    reinterpret_cast<uint4 *>(stg + kOffMq)[lane] =
        make_uint4(pack_h2(mq(0, 0), mq(0, 1)), pack_h2(mq(1, 0), mq(1, 1)), pack_h2(mq(0, 2), mq(0, 3)),
                   pack_h2(mq(1, 2), mq(1, 3)));
}

// P runs the input side ahead of the output side: iteration i preps stage i,
// builds the X2q X2k^T Gram of step i - 2 for the Y warps, then writes the
// outputs (Z = Q + LN(Yq), L_t) of step i - kOutLag once the Y warps have
// handed Yq over. In the cluster form kOutLag is 3, not 2, which keeps P's own
// waits off the recurrence there (its outputs also wait for the other CTA's
// Yq): the H warps' look-ahead at step i needs stage i + 2 prepared, and the
// Y warps' output product of step i needs the Gram of step i, neither of which
// then waits for an output of a step less than two back. (The Gram of step j lands in buffer j & 1: the Y
// warps may still read step j - 1's when P builds step j's.) In the cluster
// form the Gram covers this CTA's hidden units (its "+ 1" only in CTA 0), and
// only CTA 0 writes outputs, from its own Yq plus the one CTA 1 sends. After
// a failed wait P keeps going in step like the other warps (the cluster's
// exchanges need every step's arrivals).
constexpr int kGramLag = 2;
template <int NR>
__device__ void role_prep(const MlpParams &p, uint8_t *sm, const Ring &R, int hi, size_t tok0, int lane, int nsteps,
                          int rank)
{
    using L = Lay<NR>;
    constexpr int kOutLag = NR == 1 ? 2 : 3;
    const int g = lane >> 2, c4 = lane & 3;
    uint32_t mag = 0;  // per-halfword max of |bf16 bits|: >= 0x4780 means |x| >= 2^16 (or inf/nan)
    const int tl = lane >> 1, half = lane & 1;  // output side: token and half of the features
    float gam[32], bet[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        gam[k] = p.ln_g[hi * kD + 32 * half + k];
        bet[k] = p.ln_b[hi * kD + 32 * half + k];
    }
    const uint32_t sX2k = smem_u32(sm + L::kOffX2k), sX2q = smem_u32(sm + L::kOffX2q);
    const int offQ = p.q_is_k ? kOffK : kOffQ;  // the key tile stands in for the queries
    const float invD = 1.f / (float)kD, eps = p.eps;
    const float gram_one = rank == 0 ? 1.f : 0.f;  // the "+ 1" of Mq2 enters once
    const bool writes_out = NR == 1 || rank == 0;
    for (int i = 0; i < nsteps + kOutLag; ++i) {
        if (i < nsteps) {
            const int st = i % kStages;
            if (!wait_bar<kSpinWaits>(&R.full[st], parity_of(i / kStages), R.flags)) abort_chain(R.flags, p.status);
            if (p.eta_gate && lane < kB) {  // eta = eta_base * sigmoid(logit); 0 past T
                float *se = reinterpret_cast<float *>(stage_ptr(sm, st) + kOffEta);
                const int t = i * kB + lane;
                se[lane] = t < p.T ? __fdividef(p.eta_base, 1.f + __expf(-se[lane])) : 0.f;
            }
            prep_stage(stage_ptr(sm, st), i > 0 ? stage_ptr(sm, (i + kStages - 1) % kStages) : nullptr, lane, mag,
                       p.prefix != 0, p.q_is_k != 0);
            warp_arrive(&R.prep[st], lane);
        }
        const int jg = i - kGramLag;
        // Gram of step jg: Mq2[s][t] = (s <= t)(x2q_t . x2k_s + 1) as B fragments (k = s, n = t).
        if (jg >= 0 && jg < nsteps) {
            if (!wait_bar<kSpinWaits>(&R.hq[jg & 1], parity_of(jg >> 1), R.flags)) abort_chain(R.flags, p.status);
            uint4 *mq2 = reinterpret_cast<uint4 *>(sm + L::kOffMq2 + (jg & 1) * 512);
            if (!p.prefix) {  // anchor rule: Yq sees no update of the batch
                mq2[lane] = make_uint4(0u, 0u, 0u, 0u);
            } else {
                const int j = jg;
                const int ra = (lane & 7) + ((lane >> 3) & 1) * 8, ca = 8 * (lane >> 4);
                const int rb = (lane & 7) + (lane >> 4) * 8, cb = 8 * ((lane >> 3) & 1);
                // four k-slices of independent accumulators (the mma latency, not its rate, bounds this)
                float dq4[4][2][4] = {};
                const uint32_t sQj = sX2q + (uint32_t)((j & 1) * L::kX2Bytes);
                const uint32_t sKj = sX2k + (uint32_t)((j % 3) * L::kX2Bytes);
    #pragma unroll
                for (int ks = 0; ks < L::kHidL / 16; ++ks) {
                    uint32_t aq[4], bk[4];
                    ldsm_x4(aq, hb(sQj, ra, 16 * ks + ca, L::kHS));
                    ldsm_x4(bk, hb(sKj, rb, 16 * ks + cb, L::kHS));
                    mma16816(dq4[ks & 3][0], aq, bk[0], bk[1]);
                    mma16816(dq4[ks & 3][1], aq, bk[2], bk[3]);
                }
                float dq[2][4];
    #pragma unroll
                for (int jj = 0; jj < 2; ++jj)
    #pragma unroll
                    for (int r = 0; r < 4; ++r) dq[jj][r] = (dq4[0][jj][r] + dq4[1][jj][r]) + (dq4[2][jj][r] + dq4[3][jj][r]);
                auto mq = [&](int jj, int r) {
                    const int t = g + 8 * (r >> 1), s = 8 * jj + 2 * c4 + (r & 1);
                    return s <= t ? dq[jj][r] + gram_one : 0.f;
                };
                mq2[lane] = make_uint4(pack_h2(mq(0, 0), mq(0, 1)), pack_h2(mq(1, 0), mq(1, 1)),
                                       pack_h2(mq(0, 2), mq(0, 3)), pack_h2(mq(1, 2), mq(1, 3)));
            }
            warp_arrive(&R.mq2[jg & 1], lane);
        }
        if (i < kOutLag) continue;
        const int j = i - kOutLag, stj = j % kStages, slot = j & 1;
        uint8_t *stg = stage_ptr(sm, stj);
        if (!writes_out) {
            warp_arrive(&R.empty[stj], lane);
            continue;
        }
        // Output of step j: z = q + LN(yq), L_t = ||z_t - v_t||^2; lane pair per token.
        if (!wait_bar<kSpinWaits>(&R.yqfull[slot], parity_of(j >> 1), R.flags)) abort_chain(R.flags, p.status);
        if constexpr (NR == 2) {  // the other CTA's Yq partial (every step, aborted or not)
            if (lane == 0) mbar_arrive_expect_tx(&R.yqpfull[slot], L::kYqpTx);
            if (!wait_peer<kSpinWaits>(&R.yqpfull[slot], parity_of(j >> 1))) abort_chain(R.flags, p.status);
        }
        const float *ys = reinterpret_cast<const float *>(sm + L::kOffYq) + slot * kB * kYS + tl * kYS + 32 * half;
        float yv[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float4 v = *reinterpret_cast<const float4 *>(ys + 4 * k);
            if constexpr (NR == 2) {
                const float4 u = *reinterpret_cast<const float4 *>(ys + (L::kOffYqp - L::kOffYq) / 4 + 4 * k);
                v = make_float4(v.x + u.x, v.y + u.y, v.z + u.z, v.w + u.w);
            }
            yv[4 * k] = v.x;
            yv[4 * k + 1] = v.y;
            yv[4 * k + 2] = v.z;
            yv[4 * k + 3] = v.w;
        }
        warp_arrive(&R.yqempty[slot], lane);
        if constexpr (NR == 2) {  // the slot may be rewritten by CTA 1
            if (lane == 0) mbar_arrive_remote(map_shared(smem_u32(&R.yqpempty[slot]), 1));
        }
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) s += yv[k];
        s += __shfl_xor_sync(kFull, s, 1);
        const float mu = s * invD;
        float v2 = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) v2 = fmaf(yv[k] - mu, yv[k] - mu, v2);
        v2 += __shfl_xor_sync(kFull, v2, 1);
        const float rs = rsqrtf(v2 * invD + eps);
        float l = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int chunk = 4 * half + c;  // 8 features per 16-byte chunk
            const uint4 qb = *reinterpret_cast<const uint4 *>(stg + offQ + swz(tl, chunk));
            const uint4 vb = *reinterpret_cast<const uint4 *>(stg + kOffV + swz(tl, chunk));
            const uint32_t qw[4] = {qb.x, qb.y, qb.z, qb.w}, vw[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int k = 8 * c + q;
                const float qf = bf16_bits_to_f32(q & 1 ? qw[q >> 1] >> 16 : qw[q >> 1] & 0xffffu);
                const float vf = bf16_bits_to_f32(q & 1 ? vw[q >> 1] >> 16 : vw[q >> 1] & 0xffffu);
                const float z = qf + fmaf(gam[k], (yv[k] - mu) * rs, bet[k]);
                yv[k] = z;
                l = fmaf(z - vf, z - vf, l);
            }
        }
        l += __shfl_xor_sync(kFull, l, 1);
        const size_t row = tok0 + (size_t)j * kB + tl;
        const bool valid = j * kB + tl < p.T;  // rows past T (zero-filled tail) are not stored
        if (!valid) {
        } else if (p.z_f32) {
            float4 *Zr = reinterpret_cast<float4 *>(static_cast<float *>(p.Z) + row * kD + 32 * half);
#pragma unroll
            for (int k = 0; k < 8; ++k) Zr[k] = make_float4(yv[4 * k], yv[4 * k + 1], yv[4 * k + 2], yv[4 * k + 3]);
        } else {
            uint4 *Zr = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.Z) + row * kD + 32 * half);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                Zr[k] = make_uint4(pack_bf2(yv[8 * k], yv[8 * k + 1]), pack_bf2(yv[8 * k + 2], yv[8 * k + 3]),
                                   pack_bf2(yv[8 * k + 4], yv[8 * k + 5]), pack_bf2(yv[8 * k + 6], yv[8 * k + 7]));
        }
        if (p.loss && half == 0 && valid) p.loss[row] = l;
        warp_arrive(&R.empty[stj], lane);
    }
    const bool range_bad = (mag & 0xffffu) >= 0x4780u || (mag >> 16) >= 0x4780u;
    if (__any_sync(kFull, range_bad) && lane == 0) {
        R.flags[1] = 1;
        record(p.status, TTT_ERR_RANGE);
    }
}

// Shared-memory byte address of element (row, col) of a padded fp16 buffer.
__device__ __forceinline__ uint32_t hb(uint32_t base, int row, int col, int stride)
{
    return base + (uint32_t)((row * stride + col) * 2);
}

// H warps, before the main loop: W2 columns h0 + 8nt + 2c4 (+1) of rows
// 16mf + g (+8) into this warp's tensor-memory columns (fp32 master) and into
// fp16 buffers 1 and 2 (the copies steps 0 and 1 read as W2_{-2}, W2_{-1}).
// h0 and the buffers count this CTA's hidden units; hbase is its first one.
template <int NR>
__device__ void hidden_init_w2(const MlpParams &p, uint8_t *sm, int w, int warp, int bi, int hi, uint32_t tmem,
                               int lane, int hbase)
{
    using L = Lay<NR>;
    constexpr int MH = L::kMH, NT = 2 * MH;  // 16-unit row blocks, 8-unit column tiles
    const int g = lane >> 2, c4 = lane & 3;
    const int h0 = L::kHW * w;
    const float *W20 = p.W2 + bi * p.w_bstride + (long long)hi * kD * kHid;
    const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + L::tmem_cols(w);
    uint32_t v[MH][32];
#pragma unroll
    for (int mf = 0; mf < 4; ++mf)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int f0 = 16 * mf + g, hc = h0 + 8 * nt + 2 * c4;
            const float2 a = *reinterpret_cast<const float2 *>(W20 + f0 * kHid + hbase + hc);
            const float2 b = *reinterpret_cast<const float2 *>(W20 + (f0 + 8) * kHid + hbase + hc);
            const int idx = (mf * NT + nt) * 4;
            v[idx >> 5][(idx & 31) + 0] = __float_as_uint(a.x);
            v[idx >> 5][(idx & 31) + 1] = __float_as_uint(a.y);
            v[idx >> 5][(idx & 31) + 2] = __float_as_uint(b.x);
            v[idx >> 5][(idx & 31) + 3] = __float_as_uint(b.y);
#pragma unroll
            for (int buf = 1; buf <= 2; ++buf) {  // W2_{-2} = W2_{-1} = W2_0 (buffers 1 and 2)
                uint8_t *w2 = sm + L::kOffW2h + buf * L::kW2hBytes;
                *reinterpret_cast<uint32_t *>(w2 + (f0 * L::kHS + hc) * 2) = pack_h2(a.x, a.y);
                *reinterpret_cast<uint32_t *>(w2 + ((f0 + 8) * L::kHS + hc) * 2) = pack_h2(b.x, b.y);
            }
        }
#pragma unroll
    for (int c = 0; c < MH; ++c) tmem_st32(taddr + 32 * c, v[c]);
    tmem_wait_st();
}

// ------------------------------------------------------------------ H: hidden-unit warps
template <int NR>
__device__ void role_hidden(const MlpParams &p, uint8_t *sm, const Ring &R, int w, int warp, int chain, int bi,
                            int hi, uint32_t tmem, int lane, int nsteps, int hbase)
{
    using L = Lay<NR>;
    constexpr int kHS = L::kHS, kHY = L::kHY, kX2Bytes = L::kX2Bytes, kW2hBytes = L::kW2hBytes;
    constexpr int MH = L::kMH, NT = 2 * MH;  // 16-unit row blocks, 8-unit column tiles
    const int g = lane >> 2, c4 = lane & 3;
    const int h0 = L::kHW * w;  // first hidden unit of this warp among the CTA's (hbase + h0 of the chain's)
    const int offQh = p.q_is_k ? kOffKh : kOffQh;  // the key tile stands in for the queries
    const float *W10 = p.W1 + bi * p.w_bstride + (long long)hi * kHid * kD;
    const float *c10 = p.c1 + bi * p.c1_bstride + (long long)hi * kHid;
    // W1 rows hbase + h0 + 16m + g (+8), columns 8nt + 2c4 (+1)
    float W1a[MH][8][4];
    float c1v[MH][2];
#pragma unroll
    for (int m = 0; m < MH; ++m) {
        const int r0 = hbase + h0 + 16 * m + g;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float2 a = *reinterpret_cast<const float2 *>(W10 + r0 * kD + 8 * nt + 2 * c4);
            const float2 b = *reinterpret_cast<const float2 *>(W10 + (r0 + 8) * kD + 8 * nt + 2 * c4);
            W1a[m][nt][0] = a.x;
            W1a[m][nt][1] = a.y;
            W1a[m][nt][2] = b.x;
            W1a[m][nt][3] = b.y;
        }
        c1v[m][0] = c10[r0];
        c1v[m][1] = c10[r0 + 8];
    }
    // This warp's 64 tensor-memory columns: lanes of its quarter, columns 0 or 64.
    const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + L::tmem_cols(w);
    const uint32_t sW2h = smem_u32(sm + L::kOffW2h), sX2k = smem_u32(sm + L::kOffX2k);
    const uint32_t sX2q = smem_u32(sm + L::kOffX2q);
    const uint32_t sGh = smem_u32(sm + L::kOffGh), sGt = smem_u32(sm + L::kOffGt);
    const int rb = (lane & 7) + (lane >> 4) * 8, cb16 = (lane >> 3) & 1;  // non-transposed B fragment rows
    const int rt = (lane & 7) + ((lane >> 3) & 1) * 8, ct = lane >> 4;   // transposed B fragment rows
    const int srow = (lane & 7) + 8 * (lane >> 4), scol = 8 * ((lane >> 3) & 1);  // stmatrix / trans-A rows
    auto wait_stage = [&](int k) {
        if (!wait_bar<kSpinWaits>(&R.full[k % kStages], parity_of(k / kStages), R.flags) ||
            !wait_bar<kSpinWaits>(&R.prep[k % kStages], parity_of(k / kStages), R.flags))
            abort_chain(R.flags, p.status);  // keep going in step with the other warps
    };
    // acc = c1 + W1 tile^T for this warp's 32 hidden units, for one or two tiles at
    // once (W1 packed to fp16 on the fly, once for both).
    auto w1_gemm2 = [&](uint32_t tile0, float (&acc0)[MH][2][4], uint32_t tile1, float (&acc1)[MH][2][4],
                        bool two) {
#pragma unroll
        for (int m = 0; m < MH; ++m)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc0[m][n][r] = acc1[m][n][r] = c1v[m][r >> 1];
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            uint32_t bk[4], bq[4];
            ldsm_x4(bk, tile0 + swz(rb, 2 * ks + cb16));
            if (two) ldsm_x4(bq, tile1 + swz(rb, 2 * ks + cb16));
#pragma unroll
            for (int m = 0; m < MH; ++m) {
                const uint32_t af[4] = {pack_h2(W1a[m][2 * ks][0], W1a[m][2 * ks][1]),
                                        pack_h2(W1a[m][2 * ks][2], W1a[m][2 * ks][3]),
                                        pack_h2(W1a[m][2 * ks + 1][0], W1a[m][2 * ks + 1][1]),
                                        pack_h2(W1a[m][2 * ks + 1][2], W1a[m][2 * ks + 1][3])};
                mma16816(acc0[m][0], af, bk[0], bk[1]);
                mma16816(acc0[m][1], af, bk[2], bk[3]);
                if (two) {
                    mma16816(acc1[m][0], af, bq[0], bq[1]);
                    mma16816(acc1[m][1], af, bq[2], bq[3]);
                }
            }
        }
    };
    // this warp's hidden columns of an activation tile [16 t][hidden] (fp16)
    auto write_x = [&](uint32_t base, const float (&x)[MH][2][4]) {
#pragma unroll
        for (int m = 0; m < MH; ++m)
            stsm_x4_t(hb(base, srow, h0 + 16 * m + scol, kHS), pack_h2(x[m][0][0], x[m][0][1]),
                      pack_h2(x[m][0][2], x[m][0][3]), pack_h2(x[m][1][0], x[m][1][1]),
                      pack_h2(x[m][1][2], x[m][1][3]));
    };
    // Prologue: Z1_0 = W1_0 K_0^T + c1_0, Rq1_0, and S1_1 = W1_0 K_1^T + c1_0.
    float z1[MH][2][4], s1[MH][2][4], rq[MH][2][4];
    __half2 gp[MH][2][2];  // gelu'(Z1) of the next step, fp16 pairs (it only scales an fp16-rounded value)
    auto gelu_x = [&](float (&x)[MH][2][4]) {  // x <- gelu(x), gp <- gelu'(x)
#pragma unroll
        for (int m = 0; m < MH; ++m)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float d0, d1;
                    gelu2(x[m][n][2 * u], x[m][n][2 * u], d0);
                    gelu2(x[m][n][2 * u + 1], x[m][n][2 * u + 1], d1);
                    gp[m][n][u] = __floats2half2_rn(d0, d1);
                }
    };
    if (nsteps > 0) {
        wait_stage(0);
        w1_gemm2(smem_u32(stage_ptr(sm, 0) + kOffKh), z1, smem_u32(stage_ptr(sm, 0) + offQh), rq, true);
        gelu_x(z1);
        write_x(sX2k, z1);
        named_bar_arrive(kBarX2k, kHY);
    }
    if (nsteps > 1) {
        wait_stage(1);
        w1_gemm2(smem_u32(stage_ptr(sm, 1) + kOffKh), s1, 0u, s1, false);
    }
    for (int i = 0; i < nsteps; ++i) {
        const int st = i % kStages;
        uint8_t *stg = stage_ptr(sm, st);
        const uint32_t sK = smem_u32(stg + kOffKh);
        const bool commit = (i + 1) * kB <= p.t_commit;  // false only for a partial last step
        if (w == 0) TTT_TRACE_AT(p, i, 0);
        named_bar_sync(kBarG, kHY);  // G_i and A~2_i (slot i & 1) are in shared memory
        if (w == 0) TTT_TRACE_AT(p, i, 3);
        // G1pre^T = W2_{i-1}^T G_i^T (W2 columns of buffer (i+2) % 3, transposed as the A operand).
        const uint32_t sW2p = sW2h + (uint32_t)(((i + 2) % 3) * kW2hBytes);
        const uint32_t sG = sGh + (uint32_t)((i & 1) * kGBytes);
        float gg[MH][2][4] = {}, gg2[MH][2][4] = {};  // even / odd k-steps: two independent chains each
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            uint32_t bg[4];
            ldsm_x4(bg, hb(sG, rb, 16 * ks + 8 * cb16, kFS));
#pragma unroll
            for (int m = 0; m < MH; ++m) {
                uint32_t aw[4];
                ldsm_x4_t(aw, hb(sW2p, 16 * ks + srow, h0 + 16 * m + scol, kHS));
                mma16816(ks & 1 ? gg2[m][0] : gg[m][0], aw, bg[0], bg[1]);
                mma16816(ks & 1 ? gg2[m][1] : gg[m][1], aw, bg[2], bg[3]);
            }
        }
#pragma unroll
        for (int m = 0; m < MH; ++m)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int r = 0; r < 4; ++r) gg[m][n][r] += gg2[m][n][r];
        if (w == 0) TTT_TRACE_AT(p, i, 2);
        // A~1 = -(eta/b) G1 with G1 = G1pre * gelu'(Z1), fp16 A fragments (rows h, columns t); c1 += A~1 1.
        const float *se = reinterpret_cast<const float *>(stg + kOffEta);
        float es[2][2];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const float2 e2 = *reinterpret_cast<const float2 *>(se + 8 * n + 2 * c4);
            es[n][0] = -e2.x * (1.f / (float)kB);
            es[n][1] = -e2.y * (1.f / (float)kB);
        }
        uint32_t af1[MH][4];
#pragma unroll
        for (int m = 0; m < MH; ++m) {
            float a[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const __half2 d = gp[m][n][r >> 1];
                    a[n][r] = round_h(es[n][r & 1] * gg[m][n][r] * __half2float(r & 1 ? __high2half(d) : __low2half(d)));
                }
            af1[m][0] = pack_h2(a[0][0], a[0][1]);
            af1[m][1] = pack_h2(a[0][2], a[0][3]);
            af1[m][2] = pack_h2(a[1][0], a[1][1]);
            af1[m][3] = pack_h2(a[1][2], a[1][3]);
            float sr0 = a[0][0] + a[0][1] + a[1][0] + a[1][1];
            float sr1 = a[0][2] + a[0][3] + a[1][2] + a[1][3];
            sr0 += __shfl_xor_sync(kFull, sr0, 1);
            sr0 += __shfl_xor_sync(kFull, sr0, 2);
            sr1 += __shfl_xor_sync(kFull, sr1, 1);
            sr1 += __shfl_xor_sync(kFull, sr1, 2);
            if (commit) {
                c1v[m][0] += sr0;
                c1v[m][1] += sr1;
            }
        }
        if (i + 1 < nsteps) {
            // The chain: Z1_{i+1}^T = S1_{i+1} + A~1_i (K_i K_{i+1}^T + 1), X2k_{i+1} -> Y warps.
            const uint4 kx = reinterpret_cast<const uint4 *>(stage_ptr(sm, (i + 1) % kStages) + kOffKx)[lane];
#pragma unroll
            for (int m = 0; m < MH; ++m) {
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int r = 0; r < 4; ++r) z1[m][n][r] = s1[m][n][r];
                mma16816(z1[m][0], af1[m], kx.x, kx.y);
                mma16816(z1[m][1], af1[m], kx.z, kx.w);
            }
            gelu_x(z1);
            write_x(sX2k + (uint32_t)(((i + 1) % 3) * kX2Bytes), z1);
            named_bar_arrive(kBarX2k, kHY);
        }
        if (w == 0) TTT_TRACE_AT(p, i, 1);
        // Output side: Z1q_i^T = Rq1_i^T + A~1_i Mq1_i, X2q = gelu(Z1q) -> shared memory.
        {
            const uint4 mq = reinterpret_cast<const uint4 *>(stg + kOffMq)[lane];
#pragma unroll
            for (int m = 0; m < MH; ++m) {
                mma16816(rq[m][0], af1[m], mq.x, mq.y);
                mma16816(rq[m][1], af1[m], mq.z, mq.w);
            }
        }
#pragma unroll
        for (int m = 0; m < MH; ++m)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int r = 0; r < 4; ++r) rq[m][n][r] = gelu1(rq[m][n][r]);
        write_x(sX2q + (uint32_t)((i & 1) * kX2Bytes), rq);
        named_bar_arrive(kBarX2q + (i & 1), kHY);  // also orders W2_{i-1} before the Y warps' Yq_i
        warp_arrive(&R.hq[i & 1], lane);
        if (w == 0) TTT_TRACE_AT(p, i, 4);
        // W1_i = W1_{i-1} + A~1_i K_i (both updates skipped for an uncommitted partial step).
        if (commit) {
#pragma unroll
            for (int j = 0; j < kD / 16; ++j) {
                uint32_t bt[4];
                ldsm_x4_t(bt, sK + swz(rt, 2 * j + ct));
#pragma unroll
                for (int m = 0; m < MH; ++m) {
                    mma16816(W1a[m][2 * j], af1[m], bt[0], bt[1]);
                    mma16816(W1a[m][2 * j + 1], af1[m], bt[2], bt[3]);
                }
            }
        }
        if (w == 0) TTT_TRACE_AT(p, i, 5);
        // W2_i = W2_{i-1} + A~2_i^T X2k_i (rows f, this warp's hidden columns): the fp32
        // master goes through tensor memory in chunks of 32 columns (MH of them: 4 / MH
        // feature blocks of 16 each), the fp16 copy to buffer i % 3.
        if (commit) {
            uint32_t bx[MH][4];  // B = X2k_i (k = t, n = h), pairs of n-tiles
            const uint32_t sXk = sX2k + (uint32_t)((i % 3) * kX2Bytes);
#pragma unroll
            for (int q = 0; q < MH; ++q) ldsm_x4_t(bx[q], hb(sXk, rt, h0 + 16 * q + 8 * ct, kHS));
            uint8_t *w2 = sm + L::kOffW2h + (i % 3) * kW2hBytes;
            const uint32_t sGa = sGt + (uint32_t)((i & 1) * kGBytes);
#pragma unroll
            for (int hf = 0; hf < MH; ++hf) {
                uint32_t v[32];
                tmem_ld32(taddr + 32 * hf, v);
                tmem_wait_ld();
#pragma unroll
                for (int mh = 0; mh < 4 / MH; ++mh) {
                    const int mf = (4 / MH) * hf + mh;
                    uint32_t ag[4];  // A = A~2 (rows f, columns t) from Gt[t][f], transposed
                    ldsm_x4_t(ag, hb(sGa, srow, 16 * mf + scol, kFS));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        uint32_t *vv = &v[(mh * NT + nt) * 4];
                        float acc[4] = {__uint_as_float(vv[0]), __uint_as_float(vv[1]), __uint_as_float(vv[2]),
                                        __uint_as_float(vv[3])};
                        mma16816(acc, ag, bx[nt >> 1][2 * (nt & 1)], bx[nt >> 1][2 * (nt & 1) + 1]);
#pragma unroll
                        for (int r = 0; r < 4; ++r) vv[r] = __float_as_uint(acc[r]);
                        const int f0 = 16 * mf + g, hc = h0 + 8 * nt + 2 * c4;
                        *reinterpret_cast<uint32_t *>(w2 + (f0 * kHS + hc) * 2) = pack_h2(acc[0], acc[1]);
                        *reinterpret_cast<uint32_t *>(w2 + ((f0 + 8) * kHS + hc) * 2) = pack_h2(acc[2], acc[3]);
                    }
                }
                tmem_st32(taddr + 32 * hf, v);
                tmem_wait_st();
            }
        }
        if (w == 0) TTT_TRACE_AT(p, i, 6);
        // Look-ahead products from W1_i: Rq1_{i+1} and S1_{i+2} (fp16 W1 packed once for both).
        if (i + 1 < nsteps) {
            const bool two = i + 2 < nsteps;
            if (two) wait_stage(i + 2);
            w1_gemm2(smem_u32(stage_ptr(sm, (i + 1) % kStages) + offQh), rq,
                     smem_u32(stage_ptr(sm, (i + 2) % kStages) + kOffKh), s1, two);
        }
        if (w == 0) TTT_TRACE_AT(p, i, 7);
        warp_arrive(&R.empty[st], lane);
    }
    // Final state.
    bool bad = false;
    const size_t ch = (size_t)chain;
#pragma unroll
    for (int m = 0; m < MH; ++m) {
        const int r0 = hbase + h0 + 16 * m + g;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) bad |= !isfinite(W1a[m][nt][r]);
        bad |= !isfinite(c1v[m][0]) || !isfinite(c1v[m][1]);
        if (p.W1_out) {
            float *Wo = p.W1_out + ch * kHid * kD;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                *reinterpret_cast<float2 *>(Wo + r0 * kD + 8 * nt + 2 * c4) = make_float2(W1a[m][nt][0], W1a[m][nt][1]);
                *reinterpret_cast<float2 *>(Wo + (r0 + 8) * kD + 8 * nt + 2 * c4) =
                    make_float2(W1a[m][nt][2], W1a[m][nt][3]);
            }
        }
        if (p.c1_out && c4 == 0) {
            p.c1_out[ch * kHid + r0] = c1v[m][0];
            p.c1_out[ch * kHid + r0 + 8] = c1v[m][1];
        }
    }
    {
        uint32_t v[MH][32];
#pragma unroll
        for (int c = 0; c < MH; ++c) tmem_ld32(taddr + 32 * c, v[c]);
        tmem_wait_ld();
#pragma unroll
        for (int mf = 0; mf < 4; ++mf)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int idx = (mf * NT + nt) * 4;
                const float a0 = __uint_as_float(v[idx >> 5][idx & 31]), a1v = __uint_as_float(v[idx >> 5][(idx & 31) + 1]);
                const float b0 = __uint_as_float(v[idx >> 5][(idx & 31) + 2]), b1 = __uint_as_float(v[idx >> 5][(idx & 31) + 3]);
                bad |= !isfinite(a0) || !isfinite(a1v) || !isfinite(b0) || !isfinite(b1);
                if (p.W2_out) {
                    float *Wo = p.W2_out + ch * kD * kHid;
                    const int f0 = 16 * mf + g, hc = hbase + h0 + 8 * nt + 2 * c4;
                    *reinterpret_cast<float2 *>(Wo + f0 * kHid + hc) = make_float2(a0, a1v);
                    *reinterpret_cast<float2 *>(Wo + (f0 + 8) * kHid + hc) = make_float2(b0, b1);
                }
            }
    }
    if (__any_sync(kFull, bad) && lane == 0) record(p.status, TTT_ERR_NONFINITE);
}

// ------------------------------------------------------------------ Y: output-feature warps
// LayerNorm statistics of the 16 token columns over the 64 features held by
// the two Y warps (32 rows each): local (mean, M2) per column, combined across
// the two warps by the parallel-variance formula. The local means are summed
// over the warp's eight lanes g of a column with three shuffle levels (every
// lane needs them); the M2s only by the lane that stores them, so the lanes
// split the four columns as they reduce (four shuffles instead of twelve).
// Returns mean and 1/std of the lane's four columns (8n + 2c4 + e).
__device__ __forceinline__ void y_ln_stats(const float (&x)[2][2][4], float4 *red, int &rnd, int y, int g, int c4,
                                           float eps, float (&mu)[2][2], float (&rs)[2][2])
{
    float ml[2][2], q[2][2];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float s = col_sum(x[0][n][e] + x[0][n][e + 2] + x[1][n][e] + x[1][n][e + 2]) * (1.f / 32.f);
            float qq = 0.f;
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float d = x[m][n][e + 2 * u] - s;
                    qq = fmaf(d, d, qq);
                }
            ml[n][e] = s;
            q[n][e] = qq;
        }
    // M2 of column (n, e) = (g bit 2, g bit 1) ends in the lanes with g bit 0 clear.
    const int bA = (g >> 2) & 1, bB = (g >> 1) & 1;
    float hA[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) hA[e] = (bA ? q[1][e] : q[0][e]) + __shfl_xor_sync(kFull, bA ? q[0][e] : q[1][e], 16);
    float m2 = (bB ? hA[1] : hA[0]) + __shfl_xor_sync(kFull, bB ? hA[0] : hA[1], 8);
    m2 += __shfl_xor_sync(kFull, m2, 4);
    float4 *rb = red + (rnd & 1) * kNY * kB;
    const float mlc = bA ? (bB ? ml[1][1] : ml[1][0]) : (bB ? ml[0][1] : ml[0][0]);
    if ((g & 1) == 0) rb[y * kB + 8 * bA + 2 * c4 + bB] = make_float4(mlc, m2, 0.f, 0.f);
    named_bar_sync(kBarYln, kNY * 32);
    ++rnd;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = 8 * n + 2 * c4 + e;
            const float4 a = rb[t], b = rb[kB + t];
            const float mean = 0.5f * (a.x + b.x);
            const float m2t = a.y + b.y + 32.f * ((a.x - mean) * (a.x - mean) + (b.x - mean) * (b.x - mean));
            mu[n][e] = mean;
            rs[n][e] = rsqrtf(m2t * (1.f / (float)kD) + eps);
        }
}

// Sums over the 64 features of three per-element quantities per column: each
// Y warp's twelve values (three quantities x the lane's four columns) are
// summed over its eight lanes g that share c4, the lanes splitting them as they
// go (g bit 2 picks n, bit 1 the column e, bit 0 quantity a or b, c): eleven
// shuffles where summing each value over all eight lanes takes thirty-six.
// The Y warps' totals then meet in shared memory as before.
__device__ __forceinline__ void y_sum3(float (&a)[2][2], float (&b)[2][2], float (&c)[2][2], float4 *red, int &rnd,
                                       int y, int g, int c4)
{
    const int bA = (g >> 2) & 1, bB = (g >> 1) & 1, bC = g & 1;
    float hA[3][2], hB[3];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        hA[0][e] = (bA ? a[1][e] : a[0][e]) + __shfl_xor_sync(kFull, bA ? a[0][e] : a[1][e], 16);
        hA[1][e] = (bA ? b[1][e] : b[0][e]) + __shfl_xor_sync(kFull, bA ? b[0][e] : b[1][e], 16);
        hA[2][e] = (bA ? c[1][e] : c[0][e]) + __shfl_xor_sync(kFull, bA ? c[0][e] : c[1][e], 16);
    }
#pragma unroll
    for (int k = 0; k < 3; ++k)
        hB[k] = (bB ? hA[k][1] : hA[k][0]) + __shfl_xor_sync(kFull, bB ? hA[k][0] : hA[k][1], 8);
    const float x0 = __shfl_xor_sync(kFull, bC ? hB[0] : hB[1], 4);
    const float x1 = __shfl_xor_sync(kFull, hB[2], 4);
    float4 *rb = red + (rnd & 1) * kNY * kB;
    {
        float *rx = reinterpret_cast<float *>(rb + y * kB + 8 * bA + 2 * c4 + bB);
        if (bC == 0) {  // quantity a
            rx[0] = hB[0] + x0;
        } else {        // quantities b and c
            rx[1] = hB[1] + x0;
            rx[2] = hB[2] + x1;
        }
    }
    named_bar_sync(kBarYln, kNY * 32);
    ++rnd;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = 8 * n + 2 * c4 + e;
            const float4 u = rb[t], v = rb[kB + t];
            a[n][e] = u.x + v.x;
            b[n][e] = u.y + v.y;
            c[n][e] = u.z + v.z;
        }
}

// Y^T (rows f0..f0+31, 16 token columns) += W2 (fp16 buffer) X^T over the CTA's
// hidden units; even and odd k-steps go to separate accumulators (8 independent chains).
template <int NR>
__device__ __forceinline__ void y_gemm(uint32_t sW2, uint32_t sX, int f0, int lane, float (&acc)[2][2][4])
{
    using L = Lay<NR>;
    constexpr int kHS = L::kHS;
    const int ra = (lane & 7) + ((lane >> 3) & 1) * 8, ca = 8 * (lane >> 4);   // A rows (non-transposed)
    const int rb = (lane & 7) + (lane >> 4) * 8, cb = 8 * ((lane >> 3) & 1);   // B rows (non-transposed)
    float acc2[2][2][4] = {};
#pragma unroll 4
    for (int ks = 0; ks < L::kHidL / 16; ks += 2) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            uint32_t bx[4];
            ldsm_x4(bx, hb(sX, rb, 16 * (ks + u) + cb, kHS));
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                uint32_t aw[4];
                ldsm_x4(aw, hb(sW2, f0 + 16 * m + ra, 16 * (ks + u) + ca, kHS));
                mma16816(u ? acc2[m][0] : acc[m][0], aw, bx[0], bx[1]);
                mma16816(u ? acc2[m][1] : acc[m][1], aw, bx[2], bx[3]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[m][n][r] += acc2[m][n][r];
}

// Y warps. Iteration i first runs step i's part of the recurrence (Y from the
// look-ahead, LayerNorm backward, G and A~2 to the H warps), then the output
// product of step i - 1 (Yq = X2q W2^T + c2 + A~2 Mq2, handed to P), which is
// off the recurrence and overlaps the H warps' work on step i. In the cluster
// form both products are this CTA's partials: the Y partial goes to the other
// CTA and comes back as the sum before the LayerNorm; CTA 1 sends its Yq
// partial to CTA 0 instead of handing it to its own P.
template <int NR>
__device__ void role_y(const MlpParams &p, uint8_t *sm, const Ring &R, int y, int chain, int bi, int hi, size_t tok0,
                       int lane, int nsteps, int rank)
{
    using L = Lay<NR>;
    constexpr int kHS = L::kHS, kHY = L::kHY, kX2Bytes = L::kX2Bytes, kW2hBytes = L::kW2hBytes;
    const bool lead = NR == 1 || rank == 0;  // adds c2 to Yq, writes inner_loss and c2_out
    const int g = lane >> 2, c4 = lane & 3;
    const int f0 = 32 * y;  // first output feature of this warp
    const float *c20 = p.c2 + bi * p.c2_bstride + (long long)hi * kD;
    float c2v[2][2], c2p[2][2], gam[2][2], bet[2][2];  // c2_{i-1} and c2_{i-2} at the top of iteration i
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int f = f0 + 16 * m + g + 8 * u;
            c2v[m][u] = c2p[m][u] = c20[f];
            gam[m][u] = p.ln_g[hi * kD + f];
            bet[m][u] = p.ln_b[hi * kD + f];
        }
    const uint32_t sW2h = smem_u32(sm + L::kOffW2h), sX2k = smem_u32(sm + L::kOffX2k);
    const uint32_t sX2q = smem_u32(sm + L::kOffX2q);
    const uint32_t sGh = smem_u32(sm + L::kOffGh), sGt = smem_u32(sm + L::kOffGt);
    float4 *red = reinterpret_cast<float4 *>(sm + L::kOffRed);
    int rnd = 0;
    const int rbt = (lane & 7) + (lane >> 4) * 8, cbt = (lane >> 3) & 1;        // ldmatrix.trans of a tile
    const int srow = (lane & 7) + 8 * (lane >> 4), scol = 8 * ((lane >> 3) & 1);  // stmatrix rows
    const int ra = (lane & 7) + ((lane >> 3) & 1) * 8, ca = 8 * (lane >> 4);     // A rows (non-transposed)
    const int rb = (lane & 7) + (lane >> 4) * 8, cb = 8 * ((lane >> 3) & 1);     // B rows (non-transposed)
    uint32_t a2f[2][4] = {};  // A~2_{i-1} as fp16 A fragments (rows f, columns t)
    const float eps = p.eps, invD = 1.f / (float)kD;
    const int T = p.T;
    for (int i = 0; i <= nsteps; ++i) {
        uint32_t a2n[2][4];
        float c2n[2][2];
        if (i < nsteps) {
            const int st = i % kStages;
            uint8_t *stg = stage_ptr(sm, st);
            if (!wait_bar<kSpinWaits>(&R.full[st], parity_of(i / kStages), R.flags) ||
                !wait_bar<kSpinWaits>(&R.prep[st], parity_of(i / kStages), R.flags))
                abort_chain(R.flags, p.status);
            // k - v + beta at this lane's (feature, token) positions: ldmatrix.trans of the bf16 tiles.
            float kv[2][2][4];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int chunk = 2 * (2 * y + m) + cbt;
                uint32_t kr[4], vr[4];
                ldsm_x4_t(kr, smem_u32(stg + kOffK) + swz(rbt, chunk));
                ldsm_x4_t(vr, smem_u32(stg + kOffV) + swz(rbt, chunk));
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t a = kr[2 * n + u], b = vr[2 * n + u];
                        kv[m][n][2 * u] = bf16_bits_to_f32(a & 0xffffu) - bf16_bits_to_f32(b & 0xffffu) + bet[m][u];
                        kv[m][n][2 * u + 1] = bf16_bits_to_f32(a >> 16) - bf16_bits_to_f32(b >> 16) + bet[m][u];
                    }
            }
            float es[2][2];
            {
                const float *se = reinterpret_cast<const float *>(stg + kOffEta);
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    const float2 e2 = *reinterpret_cast<const float2 *>(se + 8 * n + 2 * c4);
                    es[n][0] = -e2.x * (1.f / (float)kB);
                    es[n][1] = -e2.y * (1.f / (float)kB);
                }
            }
            if (y == 0) TTT_TRACE_AT(p, i, 8);
            named_bar_sync(kBarX2k, kHY);  // X2k_i written (and with it every W2 update up to step i-2)
            if (y == 0) TTT_TRACE_AT(p, i, 9);
            // Y^T = W2_{i-1} X2k^T + c2_{i-1}, read as W2_{i-2} X2k^T + c2_{i-1} + A~2_{i-1} (X2k_{i-1} X2k^T)
            // so that the W2 update of step i-1 is off this path.
            const uint32_t sXk = sX2k + (uint32_t)((i % 3) * kX2Bytes);
            float yk[2][2][4];  // NR = 2: this CTA's partial, c2 added after the exchange
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int r = 0; r < 4; ++r) yk[m][n][r] = NR == 1 ? c2v[m][r >> 1] : 0.f;
            y_gemm<NR>(sW2h + (uint32_t)(((i + 1) % 3) * kW2hBytes), sXk, f0, lane, yk);
            if (i > 0) {
                // dx[j][r] = x2_t . x2'_s, t in step i (rows), s in step i-1; four k-slices
                const uint32_t sXp = sX2k + (uint32_t)(((i + 2) % 3) * kX2Bytes);
                float dx4[4][2][4] = {};
#pragma unroll
                for (int ks = 0; ks < L::kHidL / 16; ++ks) {
                    uint32_t ax[4], bp[4];
                    ldsm_x4(ax, hb(sXk, ra, 16 * ks + ca, kHS));
                    ldsm_x4(bp, hb(sXp, rb, 16 * ks + cb, kHS));
                    mma16816(dx4[ks & 3][0], ax, bp[0], bp[1]);
                    mma16816(dx4[ks & 3][1], ax, bp[2], bp[3]);
                }
                float dx[2][4];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        dx[jj][r] = (dx4[0][jj][r] + dx4[1][jj][r]) + (dx4[2][jj][r] + dx4[3][jj][r]);
                const uint32_t bx[4] = {pack_h2(dx[0][0], dx[0][1]), pack_h2(dx[1][0], dx[1][1]),
                                        pack_h2(dx[0][2], dx[0][3]), pack_h2(dx[1][2], dx[1][3])};
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    mma16816(yk[m][0], a2f[m], bx[0], bx[1]);
                    mma16816(yk[m][1], a2f[m], bx[2], bx[3]);
                }
            }
            if constexpr (NR == 2) {
                // Exchange the partials: ours into the other CTA's slot i & 1 ([Y warp][4][lane]
                // float4), then theirs from our own slot; Y = (ours + theirs) + c2, the same
                // value in both CTAs.
                const int slot = i & 1;
                float4 *yp = reinterpret_cast<float4 *>(sm + L::kOffYp) + (slot * kNY + y) * 4 * 32 + lane;
                const uint32_t peer = (uint32_t)(rank ^ 1);
                const uint32_t rdst = map_shared(smem_u32(yp), peer);
                const uint32_t rbar = map_shared(smem_u32(&R.ypeer[slot]), peer);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float *v = yk[q >> 1][q & 1];
                    st_async_v4(rdst + (uint32_t)(q * 32 * 16),
                                make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                                           __float_as_uint(v[3])),
                                rbar);
                }
                if (y == 0 && lane == 0) mbar_arrive_expect_tx(&R.ypeer[slot], L::kYpTx);
                if (!wait_peer<kSpinWaits>(&R.ypeer[slot], parity_of(i >> 1))) abort_chain(R.flags, p.status);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 u = yp[q * 32];
                    float *v = yk[q >> 1][q & 1];
                    const int m = q >> 1;
                    v[0] = (v[0] + u.x) + c2v[m][0];
                    v[1] = (v[1] + u.y) + c2v[m][0];
                    v[2] = (v[2] + u.z) + c2v[m][1];
                    v[3] = (v[3] + u.w) + c2v[m][1];
                }
            }
            if (y == 0) TTT_TRACE_AT(p, i, 10);
            // LayerNorm forward + backward: G = dl/dY, inner loss.
            float mu[2][2], rs[2][2];
            y_ln_stats(yk, red, rnd, y, g, c4, eps, mu, rs);
            float s1[2][2] = {}, s2[2][2] = {}, sl[2][2] = {};
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int e = r & 1, u = r >> 1;
                        const float yh = (yk[m][n][r] - mu[n][e]) * rs[n][e];
                        const float E = fmaf(gam[m][u], yh, kv[m][n][r]);
                        const float dh = 2.f * gam[m][u] * E;
                        s1[n][e] += dh;
                        s2[n][e] = fmaf(dh, yh, s2[n][e]);
                        sl[n][e] = fmaf(E, E, sl[n][e]);
                    }
            y_sum3(s1, s2, sl, red, rnd, y, g, c4);
            float gh[2][2][4], a2[2][2][4];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int e = r & 1, u = r >> 1;
                        const float yh = (yk[m][n][r] - mu[n][e]) * rs[n][e];
                        const float E = fmaf(gam[m][u], yh, kv[m][n][r]);
                        const float G = rs[n][e] * (2.f * gam[m][u] * E - s1[n][e] * invD - yh * s2[n][e] * invD);
                        gh[m][n][r] = G;
                        a2[m][n][r] = round_h(es[n][e] * G);
                    }
            // G and A~2 to shared memory as [t][f] (the H warps' operands), slot i & 1.
            const uint32_t sG = sGh + (uint32_t)((i & 1) * kGBytes), sA = sGt + (uint32_t)((i & 1) * kGBytes);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                stsm_x4_t(hb(sG, srow, f0 + 16 * m + scol, kFS), pack_h2(gh[m][0][0], gh[m][0][1]),
                          pack_h2(gh[m][0][2], gh[m][0][3]), pack_h2(gh[m][1][0], gh[m][1][1]),
                          pack_h2(gh[m][1][2], gh[m][1][3]));
                stsm_x4_t(hb(sA, srow, f0 + 16 * m + scol, kFS), pack_h2(a2[m][0][0], a2[m][0][1]),
                          pack_h2(a2[m][0][2], a2[m][0][3]), pack_h2(a2[m][1][0], a2[m][1][1]),
                          pack_h2(a2[m][1][2], a2[m][1][3]));
            }
            named_bar_arrive(kBarG, kHY);
            if (y == 0) TTT_TRACE_AT(p, i, 11);
            if (p.inner_loss && lead && y == 0 && g == 0) {
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int t = i * kB + 8 * n + 2 * c4 + e;
                        if (t < T) p.inner_loss[tok0 + t] = sl[n][e];
                    }
            }
            // c2_i = c2_{i-1} + A~2_i 1, and A~2_i as A fragments for the next step.
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                float s0 = a2[m][0][0] + a2[m][0][1] + a2[m][1][0] + a2[m][1][1];
                float s1r = a2[m][0][2] + a2[m][0][3] + a2[m][1][2] + a2[m][1][3];
                s0 += __shfl_xor_sync(kFull, s0, 1);
                s0 += __shfl_xor_sync(kFull, s0, 2);
                s1r += __shfl_xor_sync(kFull, s1r, 1);
                s1r += __shfl_xor_sync(kFull, s1r, 2);
                const bool commit = (i + 1) * kB <= p.t_commit;  // false only for a partial last step
                c2n[m][0] = commit ? c2v[m][0] + s0 : c2v[m][0];
                c2n[m][1] = commit ? c2v[m][1] + s1r : c2v[m][1];
                a2n[m][0] = pack_h2(a2[m][0][0], a2[m][0][1]);
                a2n[m][1] = pack_h2(a2[m][0][2], a2[m][0][3]);
                a2n[m][2] = pack_h2(a2[m][1][0], a2[m][1][1]);
                a2n[m][3] = pack_h2(a2[m][1][2], a2[m][1][3]);
            }
            warp_arrive(&R.empty[st], lane);
        }
        if (i > 0) {
            // Output of step j = i - 1: Yq^T = W2_{j-1} X2q^T + c2_{j-1} + A~2_j Mq2, Mq2 (causal x2q.x2k + 1) from P.
            const int j = i - 1;
            named_bar_sync(kBarX2q + (j & 1), kHY);  // X2q_j written (and W2_{j-1} before it)
            if (y == 0) TTT_TRACE_AT(p, j, 12);
            float yq[2][2][4];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int r = 0; r < 4; ++r) yq[m][n][r] = lead ? c2p[m][r >> 1] : 0.f;
            y_gemm<NR>(sW2h + (uint32_t)(((j + 2) % 3) * kW2hBytes), sX2q + (uint32_t)((j & 1) * kX2Bytes), f0, lane,
                       yq);
            if (!wait_bar<kSpinWaits>(&R.mq2[j & 1], parity_of(j >> 1), R.flags)) abort_chain(R.flags, p.status);
            {
                const uint4 mq2 = reinterpret_cast<const uint4 *>(sm + L::kOffMq2 + (j & 1) * 512)[lane];
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    mma16816(yq[m][0], a2f[m], mq2.x, mq2.y);
                    mma16816(yq[m][1], a2f[m], mq2.z, mq2.w);
                }
            }
            if (y == 0) TTT_TRACE_AT(p, j, 13);
            const int slot = j & 1;
            if (lead) {
                if (!wait_bar<kSpinWaits>(&R.yqempty[slot], parity_of(j >> 1) ^ 1u, R.flags)) abort_chain(R.flags, p.status);
                float *ys = reinterpret_cast<float *>(sm + L::kOffYq) + slot * kB * kYS;
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            ys[(8 * n + 2 * c4 + (r & 1)) * kYS + f0 + 16 * m + g + 8 * (r >> 1)] = yq[m][n][r];
                warp_arrive(&R.yqfull[slot], lane);
            } else if constexpr (NR == 2) {
                // CTA 1: the partial goes to CTA 0's slot, same [token][feature] layout, once
                // CTA 0's P has read what was there (every step, aborted or not).
                if (!wait_peer<kSpinWaits>(&R.yqpempty[slot], parity_of(j >> 1) ^ 1u)) abort_chain(R.flags, p.status);
                const uint32_t rys = map_shared(smem_u32(sm + L::kOffYqp + slot * kB * kYS * 4), 0);
                const uint32_t rbar = map_shared(smem_u32(&R.yqpfull[slot]), 0);
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            st_async_b32(rys + (uint32_t)(((8 * n + 2 * c4 + (r & 1)) * kYS + f0 + 16 * m + g +
                                                           8 * (r >> 1)) * 4),
                                         __float_as_uint(yq[m][n][r]), rbar);
            }
            if (y == 0) TTT_TRACE_AT(p, j, 14);
        }
        if (i < nsteps) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    c2p[m][u] = c2v[m][u];
                    c2v[m][u] = c2n[m][u];
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) a2f[m][q] = a2n[m][q];
            }
        }
    }
    bool bad = false;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            bad |= !isfinite(c2v[m][u]);
            if (p.c2_out && lead && c4 == 0) p.c2_out[(size_t)chain * kD + f0 + 16 * m + g + 8 * u] = c2v[m][u];
        }
    if (__any_sync(kFull, bad) && lane == 0) record(p.status, TTT_ERR_NONFINITE);
}

// ------------------------------------------------------------------ kernel
template <int NR>
__device__ __forceinline__ void mlp_tc_body(const CUtensorMap *tmQ, const CUtensorMap *tmK, const CUtensorMap *tmV,
                                            const MlpParams &p)
{
    using L = Lay<NR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1024(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rank = NR == 2 ? (int)cluster_ctarank() : 0;
    const int chain = blockIdx.x / NR;
    const int bi = chain / p.H, hi = chain % p.H;
    const int nsteps = (p.T + kB - 1) / kB;  // a partial last step (T % 16 tokens) is not committed
    const size_t tok0 = (size_t)chain * p.T;
    const int hbase = rank * L::kHidL;  // first hidden unit of this CTA

    Ring R;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
    R.full = bar;
    R.prep = bar + kStages;
    R.empty = bar + 2 * kStages;
    R.hq = bar + 3 * kStages;
    R.mq2 = R.hq + 2;
    R.yqfull = R.hq + 4;
    R.yqempty = R.hq + 6;
    R.ypeer = R.hq + 8;  // cluster form only (the next six)
    R.yqpfull = R.hq + 10;
    R.yqpempty = R.hq + 12;
    R.flags = reinterpret_cast<volatile int *>(bar + L::kNumBars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kOffTmem);

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&R.full[s], 33);                 // expect_tx arrive + 32 cp.async arrivals
            mbar_init(&R.prep[s], 1);
            mbar_init(&R.empty[s], L::kNH + kNY + 1);  // H warps, Y warps, P
        }
        mbar_init(&R.hq[0], L::kNH);
        mbar_init(&R.hq[1], L::kNH);
        for (int j = 0; j < 2; ++j) {
            mbar_init(&R.mq2[j], 1);
            mbar_init(&R.yqfull[j], kNY);
            mbar_init(&R.yqempty[j], 1);
            if (NR == 2) {
                mbar_init(&R.ypeer[j], 1);     // Y warp 0's expect_tx arrival + the peer's bytes
                mbar_init(&R.yqpfull[j], 1);   // P's expect_tx arrival + the peer's bytes
                mbar_init(&R.yqpempty[j], 1);  // CTA 0's P, remotely
            }
        }
        R.flags[0] = 0;
        R.flags[1] = 0;
        fence_mbar_init();
    }
    tmem_fence_before_sync();
    __syncthreads();  // (0) barriers and the tensor-memory address
    tmem_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int hw = L::h_index(warp), yw = L::y_index(warp);
    if (hw >= 0) hidden_init_w2<NR>(p, sm, hw, warp, bi, hi, tmem, lane, hbase);
    tmem_fence_before_sync();
    __syncthreads();  // (1) initial W2 copies visible; tensor-memory stores complete
    tmem_fence_after_sync();
    if constexpr (NR == 2) cluster_sync();  // both CTAs' barriers are initialised before any remote use

    if (warp == kWarpL) {
        const StageGeom geom{kStages, kStageBytes, kOffK, p.q_is_k ? -1 : kOffQ, kOffV, kOffEta};
        role_loader<kD, kSpinWaits>(tmQ, tmK, tmV, p.eta + tok0, p.T, p.status, sm + kOffStages, geom, R.full, R.empty, R.flags,
                        chain, lane, nsteps,
#ifdef TTT_FAULT_HOOKS
                        p.drop_step
#else
                        -1
#endif
        );
    } else if (warp == kWarpP) {
        role_prep<NR>(p, sm, R, hi, tok0, lane, nsteps, rank);
    } else if (hw >= 0) {
        role_hidden<NR>(p, sm, R, hw, warp, chain, bi, hi, tmem, lane, nsteps, hbase);
    } else if (yw >= 0) {
        role_y<NR>(p, sm, R, yw, chain, bi, hi, tok0, lane, nsteps, rank);
    }
    tmem_fence_before_sync();
    __syncthreads();  // (2) every tensor-memory access is complete
    // Cluster form: every store and arrival one CTA makes in the other's shared memory
    // was waited for by the other (the exchanges run every step), so neither leaves
    // while the other may still write to it.
    if constexpr (NR == 2) cluster_sync();
    if (warp == 0) {
        tmem_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// kStd: the prefix rule with separate queries, no in-kernel gate and bf16 Z, fixed
// at compile time, so the branches on those fields drop out of the hot code (the
// cluster form measured 1.53 -> 1.46 ms on the 4 x 12-chain T = 8192 workload).
__device__ __forceinline__ MlpParams std_params(const MlpParams &p, bool std_case)
{
    MlpParams q = p;
    if (std_case) {
        q.prefix = 1;
        q.q_is_k = 0;
        q.eta_gate = 0;
        q.z_f32 = 0;
    }
    return q;
}

template <bool kStd>
__global__ void __launch_bounds__(Lay<1>::kThreads, 1)
mlp_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const MlpParams p)
{
    const MlpParams q = std_params(p, kStd);
    mlp_tc_body<1>(&tmQ, &tmK, &tmV, q);
}

// One chain per cluster of two CTAs (blocks 2c and 2c + 1), hidden units split.
template <bool kStd>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Lay<2>::kThreads, 1)
mlp_tc_cluster_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const MlpParams p)
{
    const MlpParams q = std_params(p, kStd);
    mlp_tc_body<2>(&tmQ, &tmK, &tmV, q);
}

std::atomic<int> g_mlp_cluster_mode{1};

// The cluster form runs when every chain gets its pair of SMs in one wave
// (mode 1, the default), always (2) or never (0).
bool mlp_use_cluster_form(int chains)
{
    const int mode = g_mlp_cluster_mode.load(std::memory_order_relaxed);
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

}  // namespace

bool mlp_tc_supported(int io, int d, int hidden, int mb)
{
    return io == TTT_BF16 && d == kD && hidden == kHid && mb == kB;
}

int mlp_cluster_mode(int mode)
{
    if (mode >= 0 && mode <= 2) g_mlp_cluster_mode.store(mode, std::memory_order_relaxed);
    return g_mlp_cluster_mode.load(std::memory_order_relaxed);
}

cudaError_t launch_mlp_tc(const MlpParams &p, int chains, cudaStream_t s)
{
    CUtensorMap mQ, mK, mV;
    if (!make_map(&mQ, p.Q, kD, p.T, chains, 16) || !make_map(&mK, p.K, kD, p.T, chains, 16) ||
        !make_map(&mV, p.V, kD, p.T, chains, 16))
        return cudaErrorInvalidValue;
    const bool std_case = p.prefix != 0 && !p.q_is_k && !p.eta_gate && !p.z_f32;
    if (mlp_use_cluster_form(chains)) {
        if (std_case) {
            cudaError_t e = ensure_smem<mlp_tc_cluster_kernel<true>>(Lay<2>::kSmemAlloc);
            if (e != cudaSuccess) return e;
            mlp_tc_cluster_kernel<true><<<2 * chains, Lay<2>::kThreads, Lay<2>::kSmemAlloc, s>>>(mQ, mK, mV, p);
        } else {
            cudaError_t e = ensure_smem<mlp_tc_cluster_kernel<false>>(Lay<2>::kSmemAlloc);
            if (e != cudaSuccess) return e;
            mlp_tc_cluster_kernel<false><<<2 * chains, Lay<2>::kThreads, Lay<2>::kSmemAlloc, s>>>(mQ, mK, mV, p);
        }
        return cudaGetLastError();
    }
    if (std_case) {
        cudaError_t e = ensure_smem<mlp_tc_kernel<true>>(Lay<1>::kSmemAlloc);
        if (e != cudaSuccess) return e;
        mlp_tc_kernel<true><<<chains, Lay<1>::kThreads, Lay<1>::kSmemAlloc, s>>>(mQ, mK, mV, p);
    } else {
        cudaError_t e = ensure_smem<mlp_tc_kernel<false>>(Lay<1>::kSmemAlloc);
        if (e != cudaSuccess) return e;
        mlp_tc_kernel<false><<<chains, Lay<1>::kThreads, Lay<1>::kSmemAlloc, s>>>(mQ, mK, mV, p);
    }
    return cudaGetLastError();
}

}  // namespace ttt
