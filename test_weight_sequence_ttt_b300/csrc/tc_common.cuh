// tc_common.cuh -- pieces shared by the tensor-core TTT kernels (sm_103a):
// the 16-token super-step, the 128B-swizzled tile addressing, bounded waits,
// the TMA tile loader role and the host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace tc {

constexpr int kSS = 16;  // tokens per super-step
constexpr unsigned kFull = 0xffffffffu;

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

// Waits come in two kinds. By default a waiting thread lets the hardware
// suspend it between polls, so a waiting warp takes no issue slots from the
// warps that share its scheduler. With kSpin it polls without suspending and
// resumes the moment the phase completes, at the cost of issue slots.
// Measured on B300: the TTT-MLP kernel runs faster with spinning waits
// (1.57 -> 1.52 ms on the 4 x 12-chain T = 8192 workload), the TTT-Linear
// kernel slower (7.15 -> 7.28 ms on 32 chains of T = 128K).

// Bounded wait that also gives up as soon as another warp has aborted
// (flags[0] != 0).
template <bool kSpin = false>
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *flags)
{
    if (kSpin ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (kSpin ? mbar_test_wait(bar, parity) : mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if (flags[0]) return false;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

// wait_bar for phases completed from another CTA of the cluster.
__device__ __forceinline__ bool wait_bar_cluster(uint64_t *bar, uint32_t parity, volatile int *flags)
{
    if (mbar_try_wait_cluster(bar, parity, 0)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity, kSleepHintNs)) return true;
        if (flags[0]) return false;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Wait for data or a release that the other CTA of the cluster sends every
// step, aborted or not: it does not give up when this CTA has aborted, so the
// two CTAs' exchanges stay in step (a barrier is never re-armed before its
// phase completed, and no CTA leaves with the peer's stores still landing).
// Bounded all the same.
template <bool kSpin = false>
__device__ __forceinline__ bool wait_peer(uint64_t *bar, uint32_t parity)
{
    if (kSpin ? mbar_test_wait_cluster(bar, parity) : mbar_try_wait_cluster(bar, parity, 0)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (kSpin ? mbar_test_wait_cluster(bar, parity) : mbar_try_wait_cluster(bar, parity, kSleepHintNs))
            return true;
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

// Tokens of a super-step that are committed: the partial last mini-batch (from
// token t_commit on) is emitted but its update is not applied.
__device__ __forceinline__ int committed_in_step(int t_commit, int step)
{
    const int n = t_commit - step * kSS;
    return n < 0 ? 0 : (n > kSS ? kSS : n);
}

// Zero the token columns t >= tc of an m16n8k16 A fragment whose k axis is the
// 16 tokens of a super-step (a0/a1: tokens 2c4, 2c4+1; a2/a3: 8 + 2c4, 9 + 2c4).
__device__ __forceinline__ void mask_tokens(uint32_t (&a)[4], int tc, int lane)
{
    if (tc >= kSS) return;
    const int t = 2 * (lane & 3);
    const uint32_t lo = (t < tc ? 0x0000ffffu : 0u) | (t + 1 < tc ? 0xffff0000u : 0u);
    const uint32_t hi = (t + 8 < tc ? 0x0000ffffu : 0u) | (t + 9 < tc ? 0xffff0000u : 0u);
    a[0] &= lo;
    a[1] &= lo;
    a[2] &= hi;
    a[3] &= hi;
}

// Two bf16 values (one 32-bit word) -> fp16x2, round to nearest even.
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w)
{
    return pack_h2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Geometry of one input stage: bf16 K/Q/V tiles [16 x D] at the given byte
// offsets (1024-aligned; off_q < 0: no query tile is loaded) and 16 fp32
// learning rates.
struct StageGeom {
    int stages, stage_bytes, off_k, off_q, off_v, off_eta;
};

// L role: TMA loads of the K/Q/V tiles of super-step i (boxes of 64 columns
// x 16 rows, 128B swizzle) and cp.async of its eta into stage i % stages,
// after every consumer has released the stage (empty[s]). Zero fill past T.
template <int D, bool kSpin = false>
__device__ void role_loader(const CUtensorMap *tmQ, const CUtensorMap *tmK, const CUtensorMap *tmV,
                            const float *eta_chain, int T, int *status, uint8_t *stages, const StageGeom g,
                            uint64_t *full, uint64_t *empty, volatile int *flags, int chain, int lane, int nsteps,
                            int drop_step = -1)
{
    if (lane == 0) {
        prefetch_tmap(tmQ);
        prefetch_tmap(tmK);
        prefetch_tmap(tmV);
    }
    int issued = 0;
    for (int i = 0; i < nsteps; ++i) {
        const int st = i % g.stages;
        if (!wait_bar<kSpin>(&empty[st], parity_of(i / g.stages) ^ 1u, flags)) {
            abort_chain(flags, status);
            break;
        }
        if (i == drop_step) {  // failure-detection tests only (-1 otherwise): this stage never lands
            issued = i + 1;
            continue;
        }
        uint8_t *stg = stages + st * g.stage_bytes;
        const int t0 = i * kSS;
        float *se = reinterpret_cast<float *>(stg + g.off_eta);
        if (lane < kSS) {
            const int t = t0 + lane;
            cp_async_4(se + lane, eta_chain + (t < T ? t : 0), t < T ? 4u : 0u);  // zero-fill past T
        }
        cp_async_mbar_arrive_noinc(&full[st]);
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[st], (g.off_q < 0 ? 2 : 3) * 32 * D);
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                tma_load_3d(stg + g.off_k + h * 2048, tmK, &full[st], h * 64, t0, chain);
                if (g.off_q >= 0) tma_load_3d(stg + g.off_q + h * 2048, tmQ, &full[st], h * 64, t0, chain);
                tma_load_3d(stg + g.off_v + h * 2048, tmV, &full[st], h * 64, t0, chain);
            }
        }
        issued = i + 1;
    }
    // Never leave while a copy issued here may still be landing in shared memory.
    for (int i = issued > g.stages ? issued - g.stages : 0; i < issued; ++i)
        (void)mbar_wait(&full[i % g.stages], parity_of(i / g.stages));
}

// ------------------------------------------------------------------ host side
inline PFN_cuTensorMapEncodeTiled_v12000 get_encode()
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
inline bool make_map(CUtensorMap *m, const void *base, int D, int T, int chains, int rows)
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

}  // namespace tc
}  // namespace ttt
