// api.cu -- the C ABI declared in include/ttt.h: host-side validation,
// dispatch to a kernel, launch. No allocation, no state between calls.
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ttt_internal.h"

namespace {

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

Range span(const void *p, size_t bytes)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Range{a, a + bytes};
}

bool overlap(const Range &a, const Range &b) { return a.lo < b.hi && b.lo < a.hi; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device memory of the current device (the one the kernels launch on), or
// managed memory. Memory of another GPU is refused: a kernel of this device
// would otherwise touch it through peer mappings, or fault where none exist.
bool is_device_ptr(const void *p)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();  // clear the sticky-free error of a failed query
        return false;
    }
    if (at.type == cudaMemoryTypeManaged) return true;
    if (at.type != cudaMemoryTypeDevice) return false;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return at.device == dev;
}

// Bytes spanned by an initial-weight array [B|1][H][per] with a batch stride.
size_t init_bytes(int B, int H, size_t per, int64_t bstride)
{
    return ((size_t)(B - 1) * (size_t)bstride + (size_t)H * per) * sizeof(float);
}

bool gate_ok(int eta_gate, float eta_base)
{
    if (eta_gate == 0) return true;
    return eta_gate == 1 && eta_base >= 0.f && eta_base <= 3.0e38f;  // finite, not NaN
}

bool dims_ok(int B, int H, int T, int d, int mb, int partial_tail)
{
    if (B < 1 || H < 1 || T < 1 || d < 1 || mb < 1) return false;
    if ((int64_t)B * H > INT32_MAX) return false;
    if (T > (1 << 30) || d > 4096) return false;
    if (partial_tail != 0 && partial_tail != 1) return false;
    return partial_tail || T % mb == 0;
}

#ifdef TTT_FAULT_HOOKS
int g_drop_step = -1;
#endif

#ifdef TTT_TRACE
unsigned long long *g_trace = nullptr;
#endif

}  // namespace

extern "C" {

#ifdef TTT_TRACE
// Diagnostic builds only: device buffer that receives phase timestamps.
void ttt_debug_set_trace(unsigned long long *buf) { g_trace = buf; }
#endif

const char *ttt_status_string(ttt_status s)
{
    switch (s) {
    case TTT_OK: return "ok";
    case TTT_ERR_NULL: return "a required pointer is NULL";
    case TTT_ERR_SHAPE: return "sizes out of range or T not a multiple of the mini-batch size";
    case TTT_ERR_UNSUPPORTED: return "no kernel for this (io dtype, d, mini-batch, hidden)";
    case TTT_ERR_ALIGN: return "a pointer or batch stride is not 16-byte aligned";
    case TTT_ERR_NOT_DEVICE_PTR: return "a pointer is not device memory";
    case TTT_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case TTT_ERR_TIMEOUT: return "a bounded device wait gave up; outputs are incomplete";
    case TTT_ERR_NONFINITE: return "the final fast-weight state is not finite";
    case TTT_ERR_ALIAS: return "an output overlaps an input or another output";
    case TTT_ERR_RANGE: return "an input is outside the fp16 operand range of the tensor-core kernel";
    case TTT_ERR_SCRATCH: return "the call needs more scratch than the library's static array holds";
    }
    return "unknown status";
}

int ttt_abi_version(void) { return TTT_ABI_VERSION; }

int ttt_debug_drop_load(int32_t step)
{
#ifdef TTT_FAULT_HOOKS
    g_drop_step = step < 0 ? -1 : step;
    return 0;
#else
    (void)step;
    return -1;
#endif
}

int32_t ttt_linear_cluster_mode(int32_t mode) { return ttt::linear_cluster_mode(mode); }

int32_t ttt_mlp_cluster_mode(int32_t mode) { return ttt::mlp_cluster_mode(mode); }

int ttt_linear_kernel_kind(int32_t io, int32_t d, int32_t mb)
{
    if (ttt::linear_tc_supported(io, d, mb)) return 2;
    if (ttt::linear_f32_supported(io, d, mb)) return 1;
    return 0;
}

int ttt_mlp_kernel_kind(int32_t io, int32_t d, int32_t hidden, int32_t mb)
{
    if (ttt::mlp_tc_supported(io, d, hidden, mb)) return 2;
    if (ttt::mlp_f32_supported(io, d, hidden, mb)) return 1;
    return 0;
}

ttt_status ttt_linear_forward(const ttt_linear_args *a, void *stream)
{
    if (!a) return TTT_ERR_NULL;
    if (a->out_rule < TTT_OUT_PREFIX || a->out_rule > TTT_OUT_KEY) return TTT_ERR_UNSUPPORTED;
    // Under the key rule the queries are the keys (Q is not read).
    const void *Qe = a->out_rule == TTT_OUT_KEY ? a->K : a->Q;
    if (!Qe || !a->K || !a->V || !a->eta || !a->W0 || !a->c0 || !a->ln_g || !a->ln_b || !a->Z)
        return TTT_ERR_NULL;
    if (!dims_ok(a->B, a->H, a->T, a->d, a->mb, a->partial_tail)) return TTT_ERR_SHAPE;
    if (a->io != TTT_F32 && a->io != TTT_BF16) return TTT_ERR_UNSUPPORTED;
    if (a->z_io != TTT_F32 && a->z_io != TTT_BF16) return TTT_ERR_UNSUPPORTED;
    if (!(a->ln_eps >= 0.f) || a->ln_eps > 1.f) return TTT_ERR_SHAPE;
    if (a->w0_bstride < 0 || a->c0_bstride < 0) return TTT_ERR_SHAPE;
    if (!gate_ok(a->eta_gate, a->eta_base)) return TTT_ERR_SHAPE;
    const int kind = ttt_linear_kernel_kind(a->io, a->d, a->mb);
    if (kind == 0) return TTT_ERR_UNSUPPORTED;

    const void *in[] = {Qe, a->K, a->V, a->eta, a->W0, a->c0, a->ln_g, a->ln_b};
    const void *out[] = {a->Z, a->W_out, a->c_out, a->loss, a->inner_loss, a->status_dev};
    for (const void *p : in)
        if (!aligned16(p)) return TTT_ERR_ALIGN;
    for (const void *p : out)
        if (p && !aligned16(p) && p != a->status_dev) return TTT_ERR_ALIGN;
    if ((a->w0_bstride & 3) || (a->c0_bstride & 3)) return TTT_ERR_ALIGN;

    const size_t B = a->B, H = a->H, T = a->T, d = a->d;
    const size_t es = a->io == TTT_BF16 ? 2 : 4;
    const size_t zs = a->z_io == TTT_BF16 ? 2 : 4;
    const size_t tok = B * H * T;
    const Range rin[] = {span(Qe, tok * d * es), span(a->K, tok * d * es), span(a->V, tok * d * es),
                         span(a->eta, tok * 4), span(a->W0, init_bytes(a->B, a->H, d * d, a->w0_bstride)),
                         span(a->c0, init_bytes(a->B, a->H, d, a->c0_bstride)), span(a->ln_g, H * d * 4),
                         span(a->ln_b, H * d * 4)};
    const Range rout[] = {span(a->Z, tok * d * zs), span(a->W_out, a->W_out ? B * H * d * d * 4 : 0),
                          span(a->c_out, a->c_out ? B * H * d * 4 : 0), span(a->loss, a->loss ? tok * 4 : 0),
                          span(a->inner_loss, a->inner_loss ? tok * 4 : 0),
                          span(a->status_dev, a->status_dev ? 4 : 0)};
    for (size_t i = 0; i < sizeof(rout) / sizeof(rout[0]); ++i) {
        if (rout[i].hi == rout[i].lo) continue;
        for (const Range &r : rin)
            if (overlap(rout[i], r)) return TTT_ERR_ALIAS;
        for (size_t j = i + 1; j < sizeof(rout) / sizeof(rout[0]); ++j)
            if (rout[j].hi != rout[j].lo && overlap(rout[i], rout[j])) return TTT_ERR_ALIAS;
    }
    for (const void *p : in)
        if (!is_device_ptr(p)) return TTT_ERR_NOT_DEVICE_PTR;
    for (const void *p : out)
        if (p && !is_device_ptr(p)) return TTT_ERR_NOT_DEVICE_PTR;

    ttt::LinearParams p;
    p.H = a->H;
    p.T = a->T;
    p.d = a->d;
    p.mb = a->mb;
    p.z_f32 = a->z_io == TTT_F32;
    p.eps = a->ln_eps;
    p.prefix = a->out_rule == TTT_OUT_PREFIX;
    p.q_is_k = a->out_rule == TTT_OUT_KEY;
    p.t_commit = a->T - a->T % a->mb;  // tokens whose updates are committed
    p.eta_gate = a->eta_gate;
    p.eta_base = a->eta_base;
#ifdef TTT_FAULT_HOOKS
    p.drop_step = g_drop_step;
#else
    p.drop_step = -1;
#endif
    p.Q = Qe;
    p.K = a->K;
    p.V = a->V;
    p.eta = a->eta;
    p.W0 = a->W0;
    p.c0 = a->c0;
    p.w0_bstride = a->w0_bstride;
    p.c0_bstride = a->c0_bstride;
    p.ln_g = a->ln_g;
    p.ln_b = a->ln_b;
    p.Z = a->Z;
    p.W_out = a->W_out;
    p.c_out = a->c_out;
    p.loss = a->loss;
    p.inner_loss = a->inner_loss;
    p.status = a->status_dev;
#ifdef TTT_TRACE
    p.trace = g_trace;
#else
    p.trace = nullptr;
#endif
    const int chains = a->B * a->H;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = kind == 2 ? ttt::launch_linear_tc(p, chains, s) : ttt::launch_linear_f32(p, a->io, chains, s);
    return e == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

ttt_status ttt_mlp_forward(const ttt_mlp_args *a, void *stream)
{
    if (!a) return TTT_ERR_NULL;
    if (a->out_rule < TTT_OUT_PREFIX || a->out_rule > TTT_OUT_KEY) return TTT_ERR_UNSUPPORTED;
    const void *Qe = a->out_rule == TTT_OUT_KEY ? a->K : a->Q;
    if (!Qe || !a->K || !a->V || !a->eta || !a->W1_0 || !a->c1_0 || !a->W2_0 || !a->c2_0 || !a->ln_g ||
        !a->ln_b || !a->Z)
        return TTT_ERR_NULL;
    if (!dims_ok(a->B, a->H, a->T, a->d, a->mb, a->partial_tail) || a->hidden < 1 || a->hidden > 4096)
        return TTT_ERR_SHAPE;
    if (a->io != TTT_F32 && a->io != TTT_BF16) return TTT_ERR_UNSUPPORTED;
    if (a->z_io != TTT_F32 && a->z_io != TTT_BF16) return TTT_ERR_UNSUPPORTED;
    if (!(a->ln_eps >= 0.f) || a->ln_eps > 1.f) return TTT_ERR_SHAPE;
    if (a->w_bstride < 0 || a->c1_bstride < 0 || a->c2_bstride < 0) return TTT_ERR_SHAPE;
    if (!gate_ok(a->eta_gate, a->eta_base)) return TTT_ERR_SHAPE;
    const int kind = ttt_mlp_kernel_kind(a->io, a->d, a->hidden, a->mb);
    if (kind == 0) return TTT_ERR_UNSUPPORTED;

    const void *in[] = {Qe, a->K, a->V, a->eta, a->W1_0, a->c1_0, a->W2_0, a->c2_0, a->ln_g, a->ln_b};
    const void *out[] = {a->Z, a->W1_out, a->c1_out, a->W2_out, a->c2_out, a->loss, a->inner_loss, a->status_dev};
    for (const void *p : in)
        if (!aligned16(p)) return TTT_ERR_ALIGN;
    for (const void *p : out)
        if (p && !aligned16(p) && p != a->status_dev) return TTT_ERR_ALIGN;
    if ((a->w_bstride & 3) || (a->c1_bstride & 3) || (a->c2_bstride & 3)) return TTT_ERR_ALIGN;

    const size_t B = a->B, H = a->H, T = a->T, d = a->d, h = a->hidden;
    const size_t es = a->io == TTT_BF16 ? 2 : 4;
    const size_t zs = a->z_io == TTT_BF16 ? 2 : 4;
    const size_t tok = B * H * T;
    const Range rin[] = {span(Qe, tok * d * es), span(a->K, tok * d * es), span(a->V, tok * d * es),
                         span(a->eta, tok * 4), span(a->W1_0, init_bytes(a->B, a->H, h * d, a->w_bstride)),
                         span(a->c1_0, init_bytes(a->B, a->H, h, a->c1_bstride)),
                         span(a->W2_0, init_bytes(a->B, a->H, h * d, a->w_bstride)),
                         span(a->c2_0, init_bytes(a->B, a->H, d, a->c2_bstride)), span(a->ln_g, H * d * 4),
                         span(a->ln_b, H * d * 4)};
    const Range rout[] = {span(a->Z, tok * d * zs),
                          span(a->W1_out, a->W1_out ? B * H * h * d * 4 : 0),
                          span(a->c1_out, a->c1_out ? B * H * h * 4 : 0),
                          span(a->W2_out, a->W2_out ? B * H * h * d * 4 : 0),
                          span(a->c2_out, a->c2_out ? B * H * d * 4 : 0),
                          span(a->loss, a->loss ? tok * 4 : 0),
                          span(a->inner_loss, a->inner_loss ? tok * 4 : 0),
                          span(a->status_dev, a->status_dev ? 4 : 0)};
    for (size_t i = 0; i < sizeof(rout) / sizeof(rout[0]); ++i) {
        if (rout[i].hi == rout[i].lo) continue;
        for (const Range &r : rin)
            if (overlap(rout[i], r)) return TTT_ERR_ALIAS;
        for (size_t j = i + 1; j < sizeof(rout) / sizeof(rout[0]); ++j)
            if (rout[j].hi != rout[j].lo && overlap(rout[i], rout[j])) return TTT_ERR_ALIAS;
    }
    for (const void *p : in)
        if (!is_device_ptr(p)) return TTT_ERR_NOT_DEVICE_PTR;
    for (const void *p : out)
        if (p && !is_device_ptr(p)) return TTT_ERR_NOT_DEVICE_PTR;

    ttt::MlpParams p;
    p.H = a->H;
    p.T = a->T;
    p.d = a->d;
    p.hidden = a->hidden;
    p.mb = a->mb;
    p.z_f32 = a->z_io == TTT_F32;
    p.eps = a->ln_eps;
    p.prefix = a->out_rule == TTT_OUT_PREFIX;
    p.q_is_k = a->out_rule == TTT_OUT_KEY;
    p.t_commit = a->T - a->T % a->mb;  // tokens whose updates are committed
    p.eta_gate = a->eta_gate;
    p.eta_base = a->eta_base;
#ifdef TTT_FAULT_HOOKS
    p.drop_step = g_drop_step;
#else
    p.drop_step = -1;
#endif
    p.Q = Qe;
    p.K = a->K;
    p.V = a->V;
    p.eta = a->eta;
    p.W1 = a->W1_0;
    p.c1 = a->c1_0;
    p.W2 = a->W2_0;
    p.c2 = a->c2_0;
    p.w_bstride = a->w_bstride;
    p.c1_bstride = a->c1_bstride;
    p.c2_bstride = a->c2_bstride;
    p.ln_g = a->ln_g;
    p.ln_b = a->ln_b;
    p.Z = a->Z;
    p.W1_out = a->W1_out;
    p.c1_out = a->c1_out;
    p.W2_out = a->W2_out;
    p.c2_out = a->c2_out;
    p.loss = a->loss;
    p.inner_loss = a->inner_loss;
    p.status = a->status_dev;
#ifdef TTT_TRACE
    p.trace = g_trace;
#else
    p.trace = nullptr;
#endif
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e =
        kind == 2 ? ttt::launch_mlp_tc(p, a->B * a->H, s) : ttt::launch_mlp_f32(p, a->io, a->B * a->H, s);
    return e == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

uint64_t ttt_linear_backward_workspace_bytes(int32_t B, int32_t H, int32_t T, int32_t d, int32_t mb)
{
    if (!dims_ok(B, H, T, d, mb, 0)) return 0;
    return ttt::linear_bwd_workspace_bytes(B, H, T, d, mb);
}

ttt_status ttt_linear_backward(const ttt_linear_bwd_args *a, void *stream)
{
    if (!a) return TTT_ERR_NULL;
    if (!a->Q || !a->K || !a->V || !a->eta || !a->W0 || !a->c0 || !a->ln_g || !a->ln_b || !a->dZ || !a->dQ ||
        !a->dK || !a->dV || !a->deta || !a->dW0 || !a->dc0 || !a->dln_g || !a->dln_b || !a->workspace)
        return TTT_ERR_NULL;
    if (!dims_ok(a->B, a->H, a->T, a->d, a->mb, 0)) return TTT_ERR_SHAPE;
    if (a->io != TTT_F32 && a->io != TTT_BF16) return TTT_ERR_UNSUPPORTED;
    if (!(a->ln_eps >= 0.f) || a->ln_eps > 1.f) return TTT_ERR_SHAPE;
    if (a->w0_bstride < 0 || a->c0_bstride < 0) return TTT_ERR_SHAPE;
    if (!gate_ok(a->eta_gate, a->eta_base)) return TTT_ERR_SHAPE;
    if (a->math != TTT_BWD_FP32 && a->math != TTT_BWD_TF32) return TTT_ERR_UNSUPPORTED;
    if (!ttt::linear_bwd_supported(a->io, a->d, a->mb)) return TTT_ERR_UNSUPPORTED;
    const size_t wsb = ttt::linear_bwd_workspace_bytes(a->B, a->H, a->T, a->d, a->mb);
    if (a->workspace_bytes < wsb) return TTT_ERR_SHAPE;

    const void *in[] = {a->Q, a->K, a->V, a->eta, a->W0, a->c0, a->ln_g, a->ln_b, a->dZ};
    const void *opt_in[] = {a->dW_n, a->dc_n};
    const void *out[] = {a->dQ, a->dK, a->dV, a->deta, a->dW0, a->dc0, a->dln_g, a->dln_b, a->workspace};
    for (const void *p : in)
        if (!aligned16(p)) return TTT_ERR_ALIGN;
    for (const void *p : opt_in)
        if (p && !aligned16(p)) return TTT_ERR_ALIGN;
    for (const void *p : out)
        if (!aligned16(p)) return TTT_ERR_ALIGN;
    if ((a->w0_bstride & 3) || (a->c0_bstride & 3)) return TTT_ERR_ALIGN;

    const size_t B = a->B, H = a->H, T = a->T, d = a->d;
    const size_t es = a->io == TTT_BF16 ? 2 : 4;
    const size_t tok = B * H * T;
    const Range rin[] = {span(a->Q, tok * d * es), span(a->K, tok * d * es), span(a->V, tok * d * es),
                         span(a->eta, tok * 4), span(a->W0, init_bytes(a->B, a->H, d * d, a->w0_bstride)),
                         span(a->c0, init_bytes(a->B, a->H, d, a->c0_bstride)), span(a->ln_g, H * d * 4),
                         span(a->ln_b, H * d * 4), span(a->dZ, tok * d * es),
                         span(a->dW_n, a->dW_n ? B * H * d * d * 4 : 0), span(a->dc_n, a->dc_n ? B * H * d * 4 : 0)};
    const Range rout[] = {span(a->dQ, tok * d * 4),       span(a->dK, tok * d * 4),
                          span(a->dV, tok * d * 4),       span(a->deta, tok * 4),
                          span(a->dW0, B * H * d * d * 4), span(a->dc0, B * H * d * 4),
                          span(a->dln_g, B * H * d * 4),  span(a->dln_b, B * H * d * 4),
                          span(a->workspace, wsb),        span(a->status_dev, a->status_dev ? 4 : 0)};
    for (size_t i = 0; i < sizeof(rout) / sizeof(rout[0]); ++i) {
        if (rout[i].hi == rout[i].lo) continue;
        for (const Range &r : rin)
            if (r.hi != r.lo && overlap(rout[i], r)) return TTT_ERR_ALIAS;
        for (size_t j = i + 1; j < sizeof(rout) / sizeof(rout[0]); ++j)
            if (rout[j].hi != rout[j].lo && overlap(rout[i], rout[j])) return TTT_ERR_ALIAS;
    }
    for (const void *p : in)
        if (!is_device_ptr(p)) return TTT_ERR_NOT_DEVICE_PTR;
    for (const void *p : opt_in)
        if (p && !is_device_ptr(p)) return TTT_ERR_NOT_DEVICE_PTR;
    for (const void *p : out)
        if (!is_device_ptr(p)) return TTT_ERR_NOT_DEVICE_PTR;
    if (a->status_dev && !is_device_ptr(a->status_dev)) return TTT_ERR_NOT_DEVICE_PTR;

    ttt::LinearBwdParams p;
    p.H = a->H;
    p.T = a->T;
    p.d = a->d;
    p.mb = a->mb;
    p.tf32 = a->math == TTT_BWD_TF32;
    p.eta_gate = a->eta_gate;
    p.eta_base = a->eta_base;
    p.eps = a->ln_eps;
    p.Q = a->Q;
    p.K = a->K;
    p.V = a->V;
    p.dZ = a->dZ;
    p.eta = a->eta;
    p.W0 = a->W0;
    p.c0 = a->c0;
    p.w0_bstride = a->w0_bstride;
    p.c0_bstride = a->c0_bstride;
    p.ln_g = a->ln_g;
    p.ln_b = a->ln_b;
    p.dW_n = a->dW_n;
    p.dc_n = a->dc_n;
    p.dQ = a->dQ;
    p.dK = a->dK;
    p.dV = a->dV;
    p.deta = a->deta;
    p.dW0 = a->dW0;
    p.dc0 = a->dc0;
    p.dln_g = a->dln_g;
    p.dln_b = a->dln_b;
    p.ws = static_cast<float *>(a->workspace);
    p.status = a->status_dev;
    const cudaError_t e = ttt::launch_linear_bwd(p, a->io, a->B * a->H, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

ttt_status ttt_linear_backward_noalloc(const ttt_linear_bwd_args *a, void *stream)
{
    if (!a) return TTT_ERR_NULL;
    const uint64_t need = ttt_linear_backward_workspace_bytes(a->B, a->H, a->T, a->d, a->mb);
    if (need == 0) return TTT_ERR_SHAPE;
    if (need > TTT_NOALLOC_SCRATCH_BYTES) return TTT_ERR_SCRATCH;
    void *scratch = nullptr;
    if (ttt::linear_bwd_noalloc_scratch(&scratch) != cudaSuccess) return TTT_ERR_CUDA;
    ttt_linear_bwd_args b = *a;
    b.workspace = scratch;
    b.workspace_bytes = TTT_NOALLOC_SCRATCH_BYTES;
    return ttt_linear_backward(&b, stream);
}

uint64_t ttt_mlp_backward_workspace_bytes(int32_t B, int32_t H, int32_t T, int32_t d, int32_t hidden, int32_t mb)
{
    if (!dims_ok(B, H, T, d, mb, 0) || hidden < 1 || hidden > 4096) return 0;
    return ttt::mlp_bwd_workspace_bytes(B, H, T, d, hidden, mb);
}

ttt_status ttt_mlp_backward(const ttt_mlp_bwd_args *a, void *stream)
{
    if (!a) return TTT_ERR_NULL;
    if (!a->Q || !a->K || !a->V || !a->eta || !a->W1_0 || !a->c1_0 || !a->W2_0 || !a->c2_0 || !a->ln_g ||
        !a->ln_b || !a->dZ || !a->dQ || !a->dK || !a->dV || !a->deta || !a->dW1 || !a->dc1 || !a->dW2 ||
        !a->dc2 || !a->dln_g || !a->dln_b || !a->workspace)
        return TTT_ERR_NULL;
    if (!dims_ok(a->B, a->H, a->T, a->d, a->mb, 0) || a->hidden < 1 || a->hidden > 4096) return TTT_ERR_SHAPE;
    if (a->io != TTT_F32 && a->io != TTT_BF16) return TTT_ERR_UNSUPPORTED;
    if (!(a->ln_eps >= 0.f) || a->ln_eps > 1.f) return TTT_ERR_SHAPE;
    if (a->w_bstride < 0 || a->c1_bstride < 0 || a->c2_bstride < 0) return TTT_ERR_SHAPE;
    if (!gate_ok(a->eta_gate, a->eta_base)) return TTT_ERR_SHAPE;
    if (!ttt::mlp_bwd_supported(a->io, a->d, a->hidden, a->mb)) return TTT_ERR_UNSUPPORTED;
    const size_t wsb = ttt::mlp_bwd_workspace_bytes(a->B, a->H, a->T, a->d, a->hidden, a->mb);
    if (a->workspace_bytes < wsb) return TTT_ERR_SHAPE;

    const void *in[] = {a->Q, a->K, a->V, a->eta, a->W1_0, a->c1_0, a->W2_0, a->c2_0, a->ln_g, a->ln_b, a->dZ};
    const void *opt_in[] = {a->dW1_n, a->dc1_n, a->dW2_n, a->dc2_n};
    const void *out[] = {a->dQ, a->dK, a->dV, a->deta, a->dW1, a->dc1, a->dW2, a->dc2, a->dln_g, a->dln_b,
                         a->workspace};
    for (const void *p : in)
        if (!aligned16(p)) return TTT_ERR_ALIGN;
    for (const void *p : opt_in)
        if (p && !aligned16(p)) return TTT_ERR_ALIGN;
    for (const void *p : out)
        if (!aligned16(p)) return TTT_ERR_ALIGN;
    if ((a->w_bstride & 3) || (a->c1_bstride & 3) || (a->c2_bstride & 3)) return TTT_ERR_ALIGN;

    const size_t B = a->B, H = a->H, T = a->T, d = a->d, h = a->hidden;
    const size_t es = a->io == TTT_BF16 ? 2 : 4;
    const size_t tok = B * H * T;
    const Range rin[] = {span(a->Q, tok * d * es), span(a->K, tok * d * es), span(a->V, tok * d * es),
                         span(a->eta, tok * 4), span(a->W1_0, init_bytes(a->B, a->H, h * d, a->w_bstride)),
                         span(a->c1_0, init_bytes(a->B, a->H, h, a->c1_bstride)),
                         span(a->W2_0, init_bytes(a->B, a->H, h * d, a->w_bstride)),
                         span(a->c2_0, init_bytes(a->B, a->H, d, a->c2_bstride)), span(a->ln_g, H * d * 4),
                         span(a->ln_b, H * d * 4), span(a->dZ, tok * d * es),
                         span(a->dW1_n, a->dW1_n ? B * H * h * d * 4 : 0), span(a->dc1_n, a->dc1_n ? B * H * h * 4 : 0),
                         span(a->dW2_n, a->dW2_n ? B * H * h * d * 4 : 0), span(a->dc2_n, a->dc2_n ? B * H * d * 4 : 0)};
    const Range rout[] = {span(a->dQ, tok * d * 4),        span(a->dK, tok * d * 4),
                          span(a->dV, tok * d * 4),        span(a->deta, tok * 4),
                          span(a->dW1, B * H * h * d * 4), span(a->dc1, B * H * h * 4),
                          span(a->dW2, B * H * h * d * 4), span(a->dc2, B * H * d * 4),
                          span(a->dln_g, B * H * d * 4),   span(a->dln_b, B * H * d * 4),
                          span(a->workspace, wsb),         span(a->status_dev, a->status_dev ? 4 : 0)};
    for (size_t i = 0; i < sizeof(rout) / sizeof(rout[0]); ++i) {
        if (rout[i].hi == rout[i].lo) continue;
        for (const Range &r : rin)
            if (r.hi != r.lo && overlap(rout[i], r)) return TTT_ERR_ALIAS;
        for (size_t j = i + 1; j < sizeof(rout) / sizeof(rout[0]); ++j)
            if (rout[j].hi != rout[j].lo && overlap(rout[i], rout[j])) return TTT_ERR_ALIAS;
    }
    for (const void *p : in)
        if (!is_device_ptr(p)) return TTT_ERR_NOT_DEVICE_PTR;
    for (const void *p : opt_in)
        if (p && !is_device_ptr(p)) return TTT_ERR_NOT_DEVICE_PTR;
    for (const void *p : out)
        if (!is_device_ptr(p)) return TTT_ERR_NOT_DEVICE_PTR;
    if (a->status_dev && !is_device_ptr(a->status_dev)) return TTT_ERR_NOT_DEVICE_PTR;

    ttt::MlpBwdParams p;
    p.H = a->H;
    p.T = a->T;
    p.d = a->d;
    p.hidden = a->hidden;
    p.mb = a->mb;
    p.eta_gate = a->eta_gate;
    p.eta_base = a->eta_base;
    p.eps = a->ln_eps;
    p.Q = a->Q;
    p.K = a->K;
    p.V = a->V;
    p.dZ = a->dZ;
    p.eta = a->eta;
    p.W1 = a->W1_0;
    p.c1 = a->c1_0;
    p.W2 = a->W2_0;
    p.c2 = a->c2_0;
    p.w_bstride = a->w_bstride;
    p.c1_bstride = a->c1_bstride;
    p.c2_bstride = a->c2_bstride;
    p.ln_g = a->ln_g;
    p.ln_b = a->ln_b;
    p.dW1_n = a->dW1_n;
    p.dc1_n = a->dc1_n;
    p.dW2_n = a->dW2_n;
    p.dc2_n = a->dc2_n;
    p.dQ = a->dQ;
    p.dK = a->dK;
    p.dV = a->dV;
    p.deta = a->deta;
    p.dW1 = a->dW1;
    p.dc1 = a->dc1;
    p.dW2 = a->dW2;
    p.dc2 = a->dc2;
    p.dln_g = a->dln_g;
    p.dln_b = a->dln_b;
    p.ws = static_cast<float *>(a->workspace);
    p.status = a->status_dev;
    const cudaError_t e = ttt::launch_mlp_bwd(p, a->io, a->B * a->H, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

}  // extern "C"
