/*
 * ttt.h -- C ABI of the test-time-training (TTT) inner-loop library for one
 * NVIDIA B300 (sm_103a).
 *
 * What the calls compute
 * ----------------------
 * For every chain (sequence beta, head h) independently, a fast weight is
 * trained on the chain's own tokens by mini-batch gradient descent and read
 * out after every token:
 *
 *   loss   (Eq. 4, "TTT layer" section of the survey page "Test-Time
 *           Training(TTT)과 LLM 메모리"):   l_t(W) = || f(k_t; W) - v_t ||^2
 *   update (Eq. 2 of the same section, mini-batched as in Eq. 5 of the
 *           "End-to-End Test-Time Training for Long Context" review, 2.3):
 *           W_i = W_{i-1} - (1/b) sum_{t in batch i} eta_t grad l_t(W_{i-1})
 *   output (Eq. 5 of the survey section):   z_t = f(q_t; W_t), where W_t is
 *           W_{i-1} minus the (1/b) eta_s grad l_s(W_{i-1}) terms of the
 *           tokens s <= t of batch i (the in-batch prefix). Two other output
 *           rules the pages discuss are selectable (`out_rule`, below); the
 *           weight trajectory, W_out, c_out and inner_loss do not depend on it.
 *   f(x; W) = x + LN(f_res(x; W))  (residual form, survey section
 *           "재현성과 공개 구현"), LN with frozen gamma/beta, biased variance,
 *           eps inside the square root.
 *   TTT-Linear: f_res(x) = W x + c,                      W [d][d], c [d]
 *   TTT-MLP:    f_res(x) = W2 gelu_tanh(W1 x + c1) + c2,  W1 [h][d], W2 [d][h]
 *   Per-token reconstruction loss L_t = || z_t - v_t ||^2 ("SR-TTT:
 *           Surprisal-Aware Residual Test-Time Training", section 2).
 * The biases c (c1, c2) are fast weights updated like W.
 *
 * Conventions
 * -----------
 * Memory:    every pointer is device memory owned by the caller; the library
 *            allocates nothing and keeps no state between calls.
 * Layout:    all tensors contiguous, row-major, chain-major:
 *              Q, K, V               [B][H][T][d]  (element type `io`)
 *              Z                     [B][H][T][d]  (element type `z_io`)
 *              eta, loss, inner_loss [B][H][T]     fp32
 *              ln_g, ln_b            [H][d]        fp32
 *            initial weights [B or 1][H][...] fp32 with a batch stride in
 *            elements (0 = one set shared by every sequence, a learned W_0).
 *            Final weights [B][H][...] fp32.
 * Alignment: every pointer 16-byte aligned.
 * Aliasing:  outputs must not overlap inputs or each other.
 * Execution: asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *            Host-side validation runs first and returns before any launch.
 * Errors:    a non-TTT_OK return means nothing was launched (validation) or
 *            the launch failed (TTT_ERR_CUDA). Problems found on the device
 *            (a bounded wait that gave up, a non-finite final state, an input
 *            outside the fp16 operand range) are written to *status_dev (if
 *            given; must hold 0 on entry) and are read by the caller after
 *            synchronising.
 * Threads:   calls on distinct streams with distinct buffers may run
 *            concurrently.
 * Z dtype:   bf16 Z rounds every output to 8 significant bits (relative error
 *            up to 2^-8 |z|); fp32 Z returns the kernel's result unrounded.
 */
#ifndef TTT_B300_H
#define TTT_B300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TTT_ABI_VERSION 10

typedef enum {
    TTT_OK = 0,
    TTT_ERR_NULL = 1,            /* a required pointer is NULL                       */
    TTT_ERR_SHAPE = 2,           /* B,H,T,d,mb,hidden out of range, or T % mb != 0   */
                                 /* without partial_tail                            */
    TTT_ERR_UNSUPPORTED = 3,     /* no kernel for (io, d, mb, hidden), or bad rule   */
    TTT_ERR_ALIGN = 4,           /* a pointer is not 16-byte aligned                 */
    TTT_ERR_NOT_DEVICE_PTR = 5,  /* a pointer is neither device memory of the        */
                                 /* current device nor managed memory               */
    TTT_ERR_CUDA = 6,            /* a CUDA runtime call or launch failed             */
    TTT_ERR_TIMEOUT = 7,         /* device: a bounded wait gave up, chain abandoned  */
    TTT_ERR_NONFINITE = 8,       /* device: non-finite value in the final state      */
    TTT_ERR_ALIAS = 9,           /* an output overlaps an input or another output    */
    TTT_ERR_RANGE = 10,          /* device: an input exceeds the fp16 operand range  */
    TTT_ERR_SCRATCH = 11         /* the call needs more than the library's static    */
                                 /* scratch (ttt_linear_backward_noalloc)           */
} ttt_status;

typedef enum { TTT_F32 = 0, TTT_BF16 = 1 } ttt_dtype;

/* Output rule: which weights and which input produce z_t for token t of
 * mini-batch i (the weight trajectory is the same under every rule).
 *  TTT_OUT_PREFIX  z_t = f(q_t; W_t), W_t = W_{i-1} plus the updates of the
 *                  tokens s <= t of batch i: Eq. 5 of the "TTT layer" section
 *                  of the survey page, Eq. 8 of the review's section 2.4.1.
 *  TTT_OUT_ANCHOR  z_t = f(q_t; W_{i-1}) for every token of the batch: the
 *                  mini-batch TTT of the "End-to-End Test-Time Training for
 *                  Long Context" review, section 2.3 (every prediction of a
 *                  batch is made with the weights before it).
 *  TTT_OUT_KEY     z_t = f(k_t; W_{i-1}): the simplified output rule, Eq. 9
 *                  of the review's section 2.4.2 (the inner loss's own
 *                  prediction reused as the output; Q is not read and may be
 *                  NULL). Then z_t - v_t is the inner residual, so
 *                  loss == inner_loss. With mb = 1 the anchor W_{i-1} is
 *                  W_{t-1}, exactly as Eq. 9 writes it. */
typedef enum { TTT_OUT_PREFIX = 0, TTT_OUT_ANCHOR = 1, TTT_OUT_KEY = 2 } ttt_out_rule;

/* Learning-rate gate. The learnable per-token learning rate of the survey's
 * "TTT layer" section is eta_t = eta_base * sigmoid(theta_lr . x_t). With
 * eta_gate = 0, `eta` holds eta_t. With eta_gate = 1 it holds the gate logits
 * theta_lr . x_t (the gate's projection, computed with the Q/K/V projections
 * outside the library, like them) and the kernels apply eta_base * sigmoid()
 * themselves; tokens past T of a partial tail keep eta = 0. */

/* Partial last mini-batch (decode / chunked prefill). With partial_tail = 0, T
 * must be a multiple of mb. With partial_tail = 1 it need not be: the last
 * r = T % mb tokens form a mini-batch that is emitted but not committed, as in
 * section 2.3.2 of the "End-to-End Test-Time Training for Long Context" review
 * (a gradient step is taken only once the decoded tokens fill a mini-batch).
 * Their Z, loss and inner_loss follow out_rule with the same 1/mb and the same
 * in-batch masks, so they equal the first r rows the completed batch will give
 * (bit for bit on the tensor-core kernels); W_out/c_out hold the state after
 * the last full mini-batch. Committing later is a resume: call again from
 * W_out/c_out with the completed mini-batch. */

/* ---------------------------------------------------------------------- */
/* TTT-Linear                                                              */
/* ---------------------------------------------------------------------- */
typedef struct {
    int32_t B, H, T, d;      /* sequences, heads, tokens per chain, head dim   */
    int32_t mb;              /* mini-batch size b (see partial_tail)           */
    int32_t io;              /* ttt_dtype of Q, K and V                        */
    int32_t z_io;            /* ttt_dtype of Z (TTT_F32 or TTT_BF16)           */
    float ln_eps;            /* LayerNorm epsilon (1e-6 on the pages' configs) */
    const void *Q, *K, *V;   /* [B][H][T][d] io: test / training / label views */
    const float *eta;        /* [B][H][T] learning rate (or gate logit)        */
    const float *W0;         /* [B|1][H][d][d] initial W (f_res = W x + c)     */
    const float *c0;         /* [B|1][H][d] initial bias                       */
    int64_t w0_bstride;      /* elements between sequences in W0 (0 = shared)  */
    int64_t c0_bstride;      /* elements between sequences in c0 (0 = shared)  */
    const float *ln_g;       /* [H][d] LayerNorm gamma                         */
    const float *ln_b;       /* [H][d] LayerNorm beta                          */
    void *Z;                 /* [B][H][T][d] z_io out (see out_rule)           */
    float *W_out;            /* [B][H][d][d] final W, or NULL                  */
    float *c_out;            /* [B][H][d] final c, or NULL                     */
    float *loss;             /* [B][H][T] L_t = ||z_t - v_t||^2, or NULL       */
    float *inner_loss;       /* [B][H][T] l_t(W_{i-1}) at the anchor, or NULL  */
    int32_t *status_dev;     /* device int32 (0 on entry), or NULL             */
    int32_t out_rule;        /* ttt_out_rule; 0 = TTT_OUT_PREFIX               */
    int32_t partial_tail;    /* 1: T % mb tokens at the end, not committed     */
    int32_t eta_gate;        /* 1: eta holds gate logits (see above)           */
    float eta_base;          /* gate scale (eta_gate = 1 only), finite, >= 0   */
} ttt_linear_args;

/* Supported: io = TTT_F32 or TTT_BF16 with 1 <= d <= 128, 1 <= mb <= 64 and
 *            d(d+1) + d + 4 mb d + mb^2 + mb floats <= 227 KB
 *            (fp32 FFMA kernel; kind 1);
 *            io = TTT_BF16 with d in {64, 128}, mb a power of two in [1, 1024]
 *            (tensor-core kernel, kind 2: fp16 MMA operands, fp32
 *            accumulation, fp32 weight state); kind 2 wins where both apply.
 *            ttt_linear_kernel_kind() reports the choice. */
ttt_status ttt_linear_forward(const ttt_linear_args *args, void *stream);

/* ---------------------------------------------------------------------- */
/* TTT-MLP                                                                 */
/* ---------------------------------------------------------------------- */
typedef struct {
    int32_t B, H, T, d, hidden; /* hidden = MLP width h (4d on the pages)       */
    int32_t mb;
    int32_t io, z_io;        /* dtypes of Q/K/V and of Z, as for TTT-Linear   */
    float ln_eps;
    const void *Q, *K, *V;
    const float *eta;
    const float *W1_0;       /* [B|1][H][hidden][d] */
    const float *c1_0;       /* [B|1][H][hidden]    */
    const float *W2_0;       /* [B|1][H][d][hidden] */
    const float *c2_0;       /* [B|1][H][d]         */
    int64_t w_bstride;       /* elements between sequences in W1_0 and W2_0 (0 = shared) */
    int64_t c1_bstride, c2_bstride;
    const float *ln_g, *ln_b;
    void *Z;
    float *W1_out, *c1_out, *W2_out, *c2_out; /* [B][H][...] or NULL */
    float *loss, *inner_loss;
    int32_t *status_dev;
    int32_t out_rule;        /* ttt_out_rule, as for TTT-Linear               */
    int32_t partial_tail;    /* as for TTT-Linear                             */
    int32_t eta_gate;        /* as for TTT-Linear                             */
    float eta_base;
} ttt_mlp_args;

/* Supported: io = TTT_F32 or TTT_BF16 with d <= 256, hidden <= 1024,
 *            mb <= 64 and the per-chain state in 227 KB of shared memory
 *            (fp32 FFMA kernel; kind 1);
 *            io = TTT_BF16 with d = 64, hidden = 256, mb = 16 (tensor-core
 *            kernel, kind 2: fp16 MMA operands, fp32 accumulation, fp32 W1 in
 *            registers and fp32 W2 in tensor memory, tanh-approximation GELU);
 *            kind 2 wins where both apply. ttt_mlp_kernel_kind() reports the
 *            choice. */
ttt_status ttt_mlp_forward(const ttt_mlp_args *args, void *stream);

/* ---------------------------------------------------------------------- */
/* TTT-Linear backward (outer-loop training)                               */
/* ---------------------------------------------------------------------- */
/* Gradients of the TTT-Linear inner loop with respect to its inputs, for
 * training the outer parameters by backpropagation through the inner loop
 * (section 2.2 of the "End-to-End Test-Time Training for Long Context" review:
 * the update itself contains a gradient, so this differentiates a gradient).
 * For the prefix output rule (TTT_OUT_PREFIX) and T a multiple of mb, with
 * upstream gradients dZ and optional seeds dW_n, dc_n on the final state, the
 * call returns the gradients of
 *     J = sum(dZ * Z) + sum(dW_n * W_n) + sum(dc_n * c_n)
 * with respect to Q, K, V, eta (the gate logits when eta_gate = 1), W0, c0,
 * ln_g and ln_b, where Z, W_n and c_n are what ttt_linear_forward returns for
 * the same inputs. Gradients of W0, c0, ln_g and ln_b come back per chain
 * ([B][H][...]); a W0 shared by the sequences (w0_bstride = 0) or the [H][d]
 * LayerNorm parameters take the sum over B.
 * Workspace: the call recomputes the forward and keeps every mini-batch's
 * starting state (W_{i-1}, c_{i-1}) and key-side activations in `workspace`,
 * caller-allocated device memory of at least
 * ttt_linear_backward_workspace_bytes() bytes (B H ((T/mb)(d^2 + d) +
 * T (3d + 2)) floats), 16-byte aligned; its contents on entry are ignored and
 * on return are unspecified. Device problems (non-finite
 * gradients of the initial state or LayerNorm) go to *status_dev. */
typedef struct {
    int32_t B, H, T, d, mb;
    int32_t io;              /* ttt_dtype of Q, K, V and dZ                    */
    float ln_eps;
    const void *Q, *K, *V;   /* [B][H][T][d] io, as for the forward            */
    const float *eta;        /* [B][H][T] learning rate (or gate logit)        */
    const float *W0, *c0;    /* [B|1][H][d][d], [B|1][H][d]                    */
    int64_t w0_bstride, c0_bstride;
    const float *ln_g, *ln_b;/* [H][d]                                         */
    const void *dZ;          /* [B][H][T][d] io: dJ/dZ                         */
    const float *dW_n;       /* [B][H][d][d] dJ/dW_n, or NULL (zero)           */
    const float *dc_n;       /* [B][H][d] dJ/dc_n, or NULL (zero)              */
    float *dQ, *dK, *dV;     /* [B][H][T][d] fp32 out                          */
    float *deta;             /* [B][H][T] fp32 out                             */
    float *dW0;              /* [B][H][d][d] fp32 out, per chain               */
    float *dc0;              /* [B][H][d] fp32 out, per chain                  */
    float *dln_g, *dln_b;    /* [B][H][d] fp32 out, per chain                  */
    void *workspace;         /* device scratch (see above)                     */
    uint64_t workspace_bytes;/* its size in bytes                              */
    int32_t *status_dev;     /* device int32 (0 on entry), or NULL             */
    int32_t eta_gate;        /* as for the forward                             */
    float eta_base;
    int32_t math;            /* TTT_BWD_FP32 (default) or TTT_BWD_TF32          */
} ttt_linear_bwd_args;

/* Arithmetic of the backward's contractions (ttt_linear_bwd_args.math).
 *  TTT_BWD_FP32  fp32-grade products: max|err| <= 1e-4 RMS per gradient tensor
 *                against an fp64 reference on the tested sizes. For d = 64,
 *                mb = 16 they run on the tensor cores in split precision (each
 *                operand as a sum of two tf32 values, three tf32 products with
 *                fp32 accumulation); other sizes use fp32 FFMA.
 *  TTT_BWD_TF32  for d = 64, mb = 16: one tf32 product each (operands rounded
 *                to 10 mantissa bits, fp32 accumulation) in the reverse sweep;
 *                the forward recompute of the weight trajectory keeps split
 *                precision. Faster; gradients within 2e-2 RMS per tensor
 *                (measured up to 1.5e-2 at T = 2048). Other sizes run as
 *                TTT_BWD_FP32. LayerNorm rows and the other elementwise work
 *                are fp32 in every mode. */
typedef enum { TTT_BWD_FP32 = 0, TTT_BWD_TF32 = 1 } ttt_bwd_math;

/* Supported: io = TTT_F32 or TTT_BF16 with 1 <= d <= 128, 1 <= mb <= 64 and
 *            2d(d+1) + 6d + 11 mb d + 2 mb^2 + 4 mb floats <= 227 KB (fp32
 *            FFMA kernel, one CTA per chain). TTT_ERR_SHAPE if T % mb != 0 or
 *            workspace_bytes is too small; every output is required. */
ttt_status ttt_linear_backward(const ttt_linear_bwd_args *args, void *stream);
/* Workspace size for ttt_linear_backward (0 if the sizes are invalid). */
uint64_t ttt_linear_backward_workspace_bytes(int32_t B, int32_t H, int32_t T, int32_t d, int32_t mb);

/* TTT-Linear backward without a caller workspace. The paper has no
 * counterpart of this call; it exists for callers that cannot allocate device
 * memory at the time of the call (code with no device allocator of its own, or
 * a host program that must keep a fixed, planned footprint and cannot risk an
 * allocation failing or synchronising in the middle of its work). It computes
 * exactly what ttt_linear_backward computes, with the same arguments, but keeps
 * the per-mini-batch checkpoints in a static array inside the library
 * (TTT_NOALLOC_SCRATCH_BYTES on every GPU that loads the library, held until
 * the process exits) instead of `workspace`; args->workspace and
 * args->workspace_bytes are ignored. It allocates nothing. Calls whose
 * ttt_linear_backward_workspace_bytes() exceeds TTT_NOALLOC_SCRATCH_BYTES
 * return TTT_ERR_SCRATCH before any launch. Every call on a GPU shares the one
 * array, and it keeps the previous call's contents (the kernel overwrites
 * everything it reads), so calls that overlap on the GPU -- on different
 * streams, or from different host threads -- race: issue them in order on one
 * stream. The array belongs to the library's module in the runtime's context
 * of the current device; every call looks its device address up there
 * (cudaGetSymbolAddress), so no address outlives a cudaDeviceReset. The first
 * call on a device, and the first after a cudaDeviceReset, loads the module
 * into that context: make it before any stream capture. */
#define TTT_NOALLOC_SCRATCH_BYTES (32u << 20)
ttt_status ttt_linear_backward_noalloc(const ttt_linear_bwd_args *args, void *stream);

/* ---------------------------------------------------------------------- */
/* TTT-MLP backward (outer-loop training)                                  */
/* ---------------------------------------------------------------------- */
/* The TTT-MLP counterpart of ttt_linear_backward: for the prefix rule and T a
 * multiple of mb, the gradients of
 *     J = sum(dZ * Z) + sum(dW1_n * W1_n) + sum(dc1_n * c1_n)
 *                     + sum(dW2_n * W2_n) + sum(dc2_n * c2_n)
 * with respect to Q, K, V, eta (the gate logits when eta_gate = 1), W1_0, c1_0,
 * W2_0, c2_0, ln_g and ln_b; weight and LayerNorm gradients per chain, as for
 * TTT-Linear. Workspace: at least ttt_mlp_backward_workspace_bytes() bytes
 * (per chain (T/mb)(2 hidden d + hidden + d) + 2 hidden d + T (2 hidden + 3 d + 2)
 * floats: every mini-batch's starting state, the weight-gradient accumulators
 * and every mini-batch's key-side activations), 16-byte aligned, contents
 * ignored on entry and unspecified on return. */
typedef struct {
    int32_t B, H, T, d, hidden, mb;
    int32_t io;              /* ttt_dtype of Q, K, V and dZ                    */
    float ln_eps;
    const void *Q, *K, *V;   /* [B][H][T][d] io                                */
    const float *eta;        /* [B][H][T]                                      */
    const float *W1_0, *c1_0, *W2_0, *c2_0; /* as for ttt_mlp_forward          */
    int64_t w_bstride, c1_bstride, c2_bstride;
    const float *ln_g, *ln_b;/* [H][d]                                         */
    const void *dZ;          /* [B][H][T][d] io                                */
    const float *dW1_n, *dc1_n, *dW2_n, *dc2_n; /* [B][H][...] seeds, or NULL  */
    float *dQ, *dK, *dV;     /* [B][H][T][d] fp32 out                          */
    float *deta;             /* [B][H][T] fp32 out                             */
    float *dW1, *dc1, *dW2, *dc2; /* [B][H][hidden][d], [B][H][hidden], [B][H][d][hidden], [B][H][d] */
    float *dln_g, *dln_b;    /* [B][H][d] fp32 out, per chain                  */
    void *workspace;
    uint64_t workspace_bytes;
    int32_t *status_dev;
    int32_t eta_gate;
    float eta_base;
} ttt_mlp_bwd_args;

/* Supported: io = TTT_F32 or TTT_BF16, 4 <= d <= 128 and 4 <= hidden with both
 *            multiples of 4, mb in {1, 2, 4, 8, 16}, and
 *            2 hidden + 6 d + 13 mb d + 9 mb hidden + 4 mb^2 + 4 mb floats
 *            <= 227 KB (fp32 FFMA kernel, one CTA of 512 threads per chain).
 *            With mb = 16 and hidden a multiple of 8 (and the half-width
 *            state fitting 227 KB) each chain runs on a cluster of two CTAs
 *            instead, each holding half of the hidden units' weights. */
ttt_status ttt_mlp_backward(const ttt_mlp_bwd_args *args, void *stream);
uint64_t ttt_mlp_backward_workspace_bytes(int32_t B, int32_t H, int32_t T, int32_t d, int32_t hidden,
                                          int32_t mb);

/* ---------------------------------------------------------------------- */
/* Introspection                                                           */
/* ---------------------------------------------------------------------- */
const char *ttt_status_string(ttt_status s);   /* static string, never NULL */
int ttt_abi_version(void);                     /* == TTT_ABI_VERSION        */
/* Which kernel a call with these sizes would launch: 0 = none (unsupported),
 * 1 = fp32 FFMA kernel, 2 = tensor-core kernel. No CUDA call is made. */
int ttt_linear_kernel_kind(int32_t io, int32_t d, int32_t mb);
int ttt_mlp_kernel_kind(int32_t io, int32_t d, int32_t hidden, int32_t mb);

/* Form of the tensor-core TTT-Linear kernel for d = 64, mb = 16 (kind 2).
 * A chain's mini-batch steps are serial ("End-to-End Test-Time Training for
 * Long Context" review, section 2.3, Eq. 5: each step starts from the weights
 * the previous one left), so with few (sequence, head) chains most SMs would
 * idle. The cluster form runs each chain on a cluster of two CTAs (two SMs)
 * that split the work by role: one SM runs the serial chain and the weight
 * update W_i = W_{i-1} - (1/b) G_i^T diag(eta) K_i, the other keeps a copy of
 * the fast weights in step (each step's update matrix -(eta/b) G_i^T crosses
 * over in distributed shared memory) and computes the outputs z_t. Results
 * agree with the one-CTA form's to rounding (the chain adds its LayerNorm sums
 * in another order). On a B300 the one-CTA form measured faster at every chain
 * count, so it is the default.
 *   mode 0: never (default); 1: when 2 * B * H <= the device's SM count;
 *   2: always. Process-wide, for later calls; any other value only returns the
 *   current mode. */
int32_t ttt_linear_cluster_mode(int32_t mode);

/* Form of the tensor-core TTT-MLP kernel (kind 2 of ttt_mlp_kernel_kind). The
 * chain is serial as above, and with few chains most SMs would idle. The
 * cluster form runs each chain on a cluster of two CTAs that split the hidden
 * units of f_res(x) = W2 gelu(W1 x + c1) + c2 ("TTT layer" section of the
 * "Test-Time Training(TTT)과 LLM 메모리" survey page): each owns 128 rows of W1
 * and c1 and 128 columns of W2, and every sum over the hidden units (the key
 * forward Y, the output forward Yq) adds the two CTAs' partial sums, which
 * cross over in distributed shared memory. Results agree with the one-CTA
 * form's to rounding (each sum over the hidden units is taken in two halves).
 *   mode 0: never; 1: when 2 * B * H <= the device's SM count (default);
 *   2: always. Process-wide, for later calls; any other value only returns the
 *   current mode. */
int32_t ttt_mlp_cluster_mode(int32_t mode);

/* Failure-detection testing hook. In the library built with fault hooks
 * (libttt_b300_faults.so; never the product library) it makes the loader of
 * the tensor-core kernels skip the tile loads of super-step `step` (and their
 * barrier arrivals) in every chain of the following calls, so that the
 * consumers' bounded waits run out: the call then ends with TTT_ERR_TIMEOUT in
 * status_dev and the CUDA context stays usable. step = -1 turns it off.
 * Returns 0 in that library; the product library has no hook and returns -1. */
int ttt_debug_drop_load(int32_t step);

#ifdef __cplusplus
}
#endif
#endif /* TTT_B300_H */
