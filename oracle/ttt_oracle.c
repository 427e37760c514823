/*
 * ttt_oracle.c -- fp64 CPU oracle of the test-time-training (TTT) inner loop.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load this file's library. The CUDA library never calls it,
 * and the two share no code, header, table or constant.
 *
 * Pages followed (cited by title and section/equation):
 *   [TTT-survey] "Test-Time Training(TTT)과 LLM 메모리: fast weights, continual
 *       learning, 손실 압축으로 읽는 개념 정리" (juhoplayground.github.io),
 *       section "TTT layer": Eq. 2 (update), Eq. 4 (loss), Eq. 5 (output);
 *       TTT-Linear and TTT-MLP; mini-batch TTT with b = 16; learnable W_0;
 *       per-token learning rate eta(x) = eta_base * sigmoid(theta_lr . x).
 *       Section "재현성과 공개 구현" (reproducibility): residual form
 *       f(x) = x + LN(f_res(x)).
 *   [E2E-review] "End-to-End Test-Time Training for Long Context" paper review
 *       (aiflower.tistory.com), section 2.3, Eq. 5: one gradient step per
 *       mini-batch of b tokens, every gradient taken at W_{i-1} and averaged
 *       with weight 1/b; b = 1 recovers Eq. 2.
 *   [SR-TTT] "SR-TTT: Surprisal-Aware Residual Test-Time Training"
 *       (gist.science), section 2 (methodology): per-token reconstruction loss
 *       L_t = ||z_t - v_t||^2.
 *
 * Readings taken where the pages leave a step open (each one is listed with its
 * reason in the design notes of this repository):
 *   - Output inside a mini-batch uses the in-batch prefix
 *       W_t = W_{i-1} - (1/b) sum_{s <= t in batch i} eta_s grad l_s(W_{i-1})
 *     (Eq. 5 of [TTT-survey] evaluates z_t with W_t; the "dual form" of the same
 *     section and its Theorem 1 equivalence need the prefix).
 *   - eta_s scales token s's gradient; the 1/b is the constant of Eq. 5 of
 *     [E2E-review].
 *   - The bias c of f_res is a fast weight updated like W; LN gamma/beta are
 *     frozen inputs.
 *   - LN uses the biased variance with eps inside the square root.
 *   - The loss is the squared L2 sum (no 1/d).
 *   - GELU is the tanh form.
 *
 * Partial last mini-batch (argument `tail`): with tail = 1, T need not be a
 * multiple of b. The last T % b tokens form a mini-batch that is emitted but not
 * committed ([E2E-review] section 2.3.2: a gradient step is taken only once the
 * decoded tokens fill a whole mini-batch): their inner losses and outputs follow
 * the same rules (same 1/b, in-batch prefix for the prefix rule), and the final
 * state is the one after the last full mini-batch.
 *
 * Output rules (argument `rule`; the weight trajectory does not depend on it):
 *   0  prefix: z_t = f(q_t; W_t), the in-batch prefix above ([TTT-survey] Eq. 5).
 *   1  anchor: z_t = f(q_t; W_{i-1}) for every token of batch i: [E2E-review]
 *      section 2.3, where every prediction of a mini-batch is made with the
 *      weights before it.
 *   2  key: z_t = f(k_t; W_{i-1}): the simplified output rule of [E2E-review]
 *      section 2.4.2, Eq. 9 (the inner loss's own prediction is the output; its
 *      W_{t-1} is the anchor under mini-batch updates, and exactly W_{t-1} at b = 1).
 *
 * Everything is double precision, plain loops, one (sequence, head) chain at a
 * time; chains are independent and run on OpenMP threads.
 *
 * Layouts (all row-major, contiguous):
 *   Q, K, V, Z      [B][H][T][d]
 *   eta, loss, inner_loss [B][H][T]
 *   TTT-Linear: W [.][H][d][d] (f_res(x) = W x + c), c [.][H][d]
 *   TTT-MLP:    W1 [.][H][h][d], c1 [.][H][h], W2 [.][H][d][h], c2 [.][H][d]
 *   ln_g, ln_b      [H][d]
 * Initial-weight arrays take a batch stride in elements (0 = one W_0 shared by
 * every sequence, as a learned W_0 is).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* LayerNorm forward and backward on one vector of length n.           */
/* LN(y) = gamma * (y - mean) / sqrt(var + eps) + beta, biased var.    */
/* ------------------------------------------------------------------ */
static void ln_forward(int n, const double *y, const double *g, const double *bt,
                       double eps, double *yhat, double *out, double *rstd_out)
{
    double mu = 0.0, var = 0.0;
    for (int j = 0; j < n; ++j) mu += y[j];
    mu /= n;
    for (int j = 0; j < n; ++j) var += (y[j] - mu) * (y[j] - mu);
    var /= n;
    double rstd = 1.0 / sqrt(var + eps);
    for (int j = 0; j < n; ++j) {
        yhat[j] = (y[j] - mu) * rstd;
        out[j] = g[j] * yhat[j] + bt[j];
    }
    *rstd_out = rstd;
}

/* Given dout = d loss / d out, return dy = d loss / d y (standard calculus). */
static void ln_backward(int n, const double *yhat, double rstd, const double *g,
                        const double *dout, double *dy)
{
    double m1 = 0.0, m2 = 0.0;
    for (int j = 0; j < n; ++j) {
        double dh = dout[j] * g[j];
        m1 += dh;
        m2 += dh * yhat[j];
    }
    m1 /= n;
    m2 /= n;
    for (int j = 0; j < n; ++j) {
        double dh = dout[j] * g[j];
        dy[j] = rstd * (dh - m1 - yhat[j] * m2);
    }
}

/* f(x) = x + LN(y) when ln_res != 0, else f(x) = y, where y = f_res(x).
 * Writes e = f(x) - v and returns ||e||^2; also returns g = d||e||^2 / d y. */
static double recon_loss_and_grad(int d, int ln_res, const double *x, const double *y,
                                  const double *v, const double *lg, const double *lb,
                                  double eps, double *g, double *work /* 3d */)
{
    double *yhat = work, *out = work + d, *e = work + 2 * d;
    double l = 0.0;
    if (ln_res) {
        double rstd;
        ln_forward(d, y, lg, lb, eps, yhat, out, &rstd);
        for (int j = 0; j < d; ++j) {
            e[j] = x[j] + out[j] - v[j];
            l += e[j] * e[j];
        }
        for (int j = 0; j < d; ++j) out[j] = 2.0 * e[j]; /* d loss / d out */
        ln_backward(d, yhat, rstd, lg, out, g);
    } else {
        for (int j = 0; j < d; ++j) {
            e[j] = y[j] - v[j];
            l += e[j] * e[j];
            g[j] = 2.0 * e[j];
        }
    }
    return l;
}

/* z = f(x) given y = f_res(x). */
static void output_rule(int d, int ln_res, const double *x, const double *y,
                        const double *lg, const double *lb, double eps, double *z,
                        double *work /* 2d */)
{
    if (ln_res) {
        double rstd;
        ln_forward(d, y, lg, lb, eps, work, work + d, &rstd);
        for (int j = 0; j < d; ++j) z[j] = x[j] + work[d + j];
    } else {
        for (int j = 0; j < d; ++j) z[j] = y[j];
    }
}

/* y = W x + c, W [m][n] row-major. */
static void affine(int m, int n, const double *W, const double *c, const double *x, double *y)
{
    for (int r = 0; r < m; ++r) {
        double acc = c[r];
        const double *w = W + (size_t)r * n;
        for (int j = 0; j < n; ++j) acc += w[j] * x[j];
        y[r] = acc;
    }
}

/* tanh-form GELU and its derivative. */
static const double GELU_A = 0.7978845608028654; /* sqrt(2/pi) */
static const double GELU_C = 0.044715;
static double gelu(double u)
{
    return 0.5 * u * (1.0 + tanh(GELU_A * (u + GELU_C * u * u * u)));
}
static double gelu_prime(double u)
{
    double w = GELU_A * (u + GELU_C * u * u * u);
    double th = tanh(w);
    return 0.5 * (1.0 + th) + 0.5 * u * (1.0 - th * th) * GELU_A * (1.0 + 3.0 * GELU_C * u * u);
}

/* ------------------------------------------------------------------ */
/* Single-token gradient of Eq. 4 ([TTT-survey]) for TTT-Linear.        */
/* l(W, c) = || f(k; W, c) - v ||^2 with f_res(x) = W x + c.            */
/* dW = g k^T, dc = g.  Exposed for the gradient pins.                  */
/* ------------------------------------------------------------------ */
double oracle_linear_token_grad(int d, int ln_res, const double *W, const double *c,
                                const double *k, const double *v, const double *lg,
                                const double *lb, double eps, double *dW, double *dc)
{
    double *y = malloc(sizeof(double) * 5 * d);
    double *work = y + d, *g = y + 4 * d;
    affine(d, d, W, c, k, y);
    double l = recon_loss_and_grad(d, ln_res, k, y, v, lg, lb, eps, g, work);
    for (int r = 0; r < d; ++r) {
        dc[r] = g[r];
        for (int j = 0; j < d; ++j) dW[(size_t)r * d + j] = g[r] * k[j];
    }
    free(y);
    return l;
}

/* Single-token gradient for TTT-MLP: f_res(x) = W2 gelu(W1 x + c1) + c2. */
double oracle_mlp_token_grad(int d, int h, int ln_res, const double *W1, const double *c1,
                             const double *W2, const double *c2, const double *k,
                             const double *v, const double *lg, const double *lb, double eps,
                             double *dW1, double *dc1, double *dW2, double *dc2)
{
    double *buf = malloc(sizeof(double) * (3 * h + 5 * d));
    double *z1 = buf, *x2 = buf + h, *dz1 = buf + 2 * h;
    double *y = buf + 3 * h, *g = y + d, *work = g + d;
    affine(h, d, W1, c1, k, z1);
    for (int j = 0; j < h; ++j) x2[j] = gelu(z1[j]);
    affine(d, h, W2, c2, x2, y);
    double l = recon_loss_and_grad(d, ln_res, k, y, v, lg, lb, eps, g, work);
    for (int r = 0; r < d; ++r) {
        dc2[r] = g[r];
        for (int j = 0; j < h; ++j) dW2[(size_t)r * h + j] = g[r] * x2[j];
    }
    for (int j = 0; j < h; ++j) {
        double s = 0.0;
        for (int r = 0; r < d; ++r) s += W2[(size_t)r * h + j] * g[r];
        dz1[j] = s * gelu_prime(z1[j]);
    }
    for (int j = 0; j < h; ++j) {
        dc1[j] = dz1[j];
        for (int i = 0; i < d; ++i) dW1[(size_t)j * d + i] = dz1[j] * k[i];
    }
    free(buf);
    return l;
}

/* ------------------------------------------------------------------ */
/* TTT-Linear inner loop, primal token form.                            */
/* ------------------------------------------------------------------ */
static void linear_chain(int T, int d, int b, int ln_res, int rule, int tail, const double *Q, const double *K,
                         const double *V, const double *eta, const double *W0,
                         const double *c0, const double *lg, const double *lb, double eps,
                         double *Z, double *W_out, double *c_out, double *loss,
                         double *inner_loss)
{
    size_t dd = (size_t)d * d;
    double *W = malloc(sizeof(double) * (2 * dd + 2 * d + (size_t)b * d + 6 * d));
    double *Wa = W + dd, *c = Wa + dd, *ca = c + d, *G = ca + d;
    double *y = G + (size_t)b * d, *work = y + d, *z = work + 3 * d, *e = z + d;
    memcpy(W, W0, sizeof(double) * dd);
    memcpy(c, c0, sizeof(double) * d);
    const int n = tail ? (T + b - 1) / b : T / b;
    for (int i = 0; i < n; ++i) {
        const int t0 = i * b;
        const int nb = T - t0 < b ? T - t0 : b; /* tokens in this mini-batch (< b: the uncommitted tail) */
        /* Anchor W_{i-1}: every gradient of mini-batch i is taken here (Eq. 5 of [E2E-review]). */
        memcpy(Wa, W, sizeof(double) * dd);
        memcpy(ca, c, sizeof(double) * d);
        for (int s = 0; s < nb; ++s) {
            const double *k = K + (size_t)(t0 + s) * d, *v = V + (size_t)(t0 + s) * d;
            affine(d, d, Wa, ca, k, y);                                    /* f_res(k; W_{i-1}) */
            double l = recon_loss_and_grad(d, ln_res, k, y, v, lg, lb, eps, G + (size_t)s * d, work);
            if (inner_loss) inner_loss[t0 + s] = l;                        /* Eq. 4 at W_{i-1} */
        }
        for (int t = 0; t < nb; ++t) {
            const double *k = K + (size_t)(t0 + t) * d, *q = Q + (size_t)(t0 + t) * d;
            const double *v = V + (size_t)(t0 + t) * d, *g = G + (size_t)t * d;
            const double s = eta[t0 + t] / b;
            /* Eq. 2 step for token t with its gradient from W_{i-1}: W becomes W_t. */
            for (int r = 0; r < d; ++r) {
                for (int j = 0; j < d; ++j) W[(size_t)r * d + j] -= s * g[r] * k[j];
                c[r] -= s * g[r];
            }
            /* Output: Eq. 5 z_t = f(q_t; W_t), or f(q_t; W_{i-1}) / f(k_t; W_{i-1}). */
            const double *x = rule == 2 ? k : q;
            if (rule == 0)
                affine(d, d, W, c, x, y);
            else
                affine(d, d, Wa, ca, x, y);
            output_rule(d, ln_res, x, y, lg, lb, eps, z, work);
            double L = 0.0;
            for (int j = 0; j < d; ++j) {
                Z[(size_t)(t0 + t) * d + j] = z[j];
                e[j] = z[j] - v[j];
                L += e[j] * e[j];
            }
            if (loss) loss[t0 + t] = L; /* L_t of [SR-TTT] */
        }
        if (nb < b) { /* the partial mini-batch is not committed */
            memcpy(W, Wa, sizeof(double) * dd);
            memcpy(c, ca, sizeof(double) * d);
        }
    }
    if (W_out) memcpy(W_out, W, sizeof(double) * dd);
    if (c_out) memcpy(c_out, c, sizeof(double) * d);
    free(W);
}

void oracle_ttt_linear(int B, int H, int T, int d, int b, int ln_res, int rule, int tail, const double *Q,
                       const double *K, const double *V, const double *eta, const double *W0,
                       const double *c0, long w0_bstride, long c0_bstride, const double *ln_g,
                       const double *ln_b, double eps, double *Z, double *W_out, double *c_out,
                       double *loss, double *inner_loss, int nthreads)
{
    const long chains = (long)B * H;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long ch = 0; ch < chains; ++ch) {
        const long bi = ch / H, hi = ch % H;
        const size_t tok = (size_t)ch * T;
        linear_chain(T, d, b, ln_res, rule, tail, Q + tok * d, K + tok * d, V + tok * d, eta + tok,
                     W0 + bi * w0_bstride + hi * (size_t)d * d, c0 + bi * c0_bstride + hi * (size_t)d,
                     ln_g + hi * (size_t)d, ln_b + hi * (size_t)d, eps, Z + tok * d,
                     W_out ? W_out + (size_t)ch * d * d : NULL, c_out ? c_out + (size_t)ch * d : NULL,
                     loss ? loss + tok : NULL, inner_loss ? inner_loss + tok : NULL);
    }
}

/* ------------------------------------------------------------------ */
/* TTT-MLP inner loop, primal token form.                               */
/* f_res(x) = W2 gelu(W1 x + c1) + c2, W1 [h][d], W2 [d][h].            */
/* ------------------------------------------------------------------ */
static void mlp_chain(int T, int d, int h, int b, int ln_res, int rule, int tail, const double *Q, const double *K,
                      const double *V, const double *eta, const double *W10, const double *c10,
                      const double *W20, const double *c20, const double *lg, const double *lb,
                      double eps, double *Z, double *W1o, double *c1o, double *W2o, double *c2o,
                      double *loss, double *inner_loss)
{
    const size_t hd = (size_t)h * d;
    double *W1 = malloc(sizeof(double) * (4 * hd + 2 * h + 2 * d + (size_t)b * (d + 2 * h) + 3 * h + 8 * d));
    double *W2 = W1 + hd, *W1a = W2 + hd, *W2a = W1a + hd;
    double *c1 = W2a + hd, *c1a = c1 + h, *c2 = c1a + h, *c2a = c2 + d;
    double *G = c2a + d, *X2 = G + (size_t)b * d, *DZ1 = X2 + (size_t)b * h;
    double *z1 = DZ1 + (size_t)b * h, *x2 = z1 + h, *dx2 = x2 + h;
    double *y = dx2 + h, *work = y + d, *z = work + 3 * d, *e = z + d, *gtmp = e + d;
    (void)gtmp;
    memcpy(W1, W10, sizeof(double) * hd);
    memcpy(W2, W20, sizeof(double) * hd);
    memcpy(c1, c10, sizeof(double) * h);
    memcpy(c2, c20, sizeof(double) * d);
    const int n = tail ? (T + b - 1) / b : T / b;
    for (int i = 0; i < n; ++i) {
        const int t0 = i * b;
        const int nb = T - t0 < b ? T - t0 : b; /* < b: the uncommitted tail */
        memcpy(W1a, W1, sizeof(double) * hd);
        memcpy(W2a, W2, sizeof(double) * hd);
        memcpy(c1a, c1, sizeof(double) * h);
        memcpy(c2a, c2, sizeof(double) * d);
        for (int s = 0; s < nb; ++s) {
            const double *k = K + (size_t)(t0 + s) * d, *v = V + (size_t)(t0 + s) * d;
            double *g = G + (size_t)s * d, *xs = X2 + (size_t)s * h, *dz = DZ1 + (size_t)s * h;
            affine(h, d, W1a, c1a, k, z1);
            for (int j = 0; j < h; ++j) xs[j] = gelu(z1[j]);
            affine(d, h, W2a, c2a, xs, y);
            double l = recon_loss_and_grad(d, ln_res, k, y, v, lg, lb, eps, g, work);
            if (inner_loss) inner_loss[t0 + s] = l;
            /* back-propagate to the first layer at the anchor weights */
            for (int j = 0; j < h; ++j) {
                double acc = 0.0;
                for (int r = 0; r < d; ++r) acc += W2a[(size_t)r * h + j] * g[r];
                dz[j] = acc * gelu_prime(z1[j]);
            }
        }
        for (int t = 0; t < nb; ++t) {
            const double *k = K + (size_t)(t0 + t) * d, *q = Q + (size_t)(t0 + t) * d;
            const double *v = V + (size_t)(t0 + t) * d;
            const double *g = G + (size_t)t * d, *xs = X2 + (size_t)t * h, *dz = DZ1 + (size_t)t * h;
            const double s = eta[t0 + t] / b;
            for (int r = 0; r < d; ++r) {
                for (int j = 0; j < h; ++j) W2[(size_t)r * h + j] -= s * g[r] * xs[j];
                c2[r] -= s * g[r];
            }
            for (int j = 0; j < h; ++j) {
                for (int r = 0; r < d; ++r) W1[(size_t)j * d + r] -= s * dz[j] * k[r];
                c1[j] -= s * dz[j];
            }
            /* Output at W_t (prefix rule) or at the anchor (anchor and key rules). */
            const double *x = rule == 2 ? k : q;
            affine(h, d, rule == 0 ? W1 : W1a, rule == 0 ? c1 : c1a, x, z1);
            for (int j = 0; j < h; ++j) x2[j] = gelu(z1[j]);
            affine(d, h, rule == 0 ? W2 : W2a, rule == 0 ? c2 : c2a, x2, y);
            output_rule(d, ln_res, x, y, lg, lb, eps, z, work);
            double L = 0.0;
            for (int j = 0; j < d; ++j) {
                Z[(size_t)(t0 + t) * d + j] = z[j];
                e[j] = z[j] - v[j];
                L += e[j] * e[j];
            }
            if (loss) loss[t0 + t] = L;
        }
        if (nb < b) { /* the partial mini-batch is not committed */
            memcpy(W1, W1a, sizeof(double) * hd);
            memcpy(W2, W2a, sizeof(double) * hd);
            memcpy(c1, c1a, sizeof(double) * h);
            memcpy(c2, c2a, sizeof(double) * d);
        }
    }
    if (W1o) memcpy(W1o, W1, sizeof(double) * hd);
    if (c1o) memcpy(c1o, c1, sizeof(double) * h);
    if (W2o) memcpy(W2o, W2, sizeof(double) * hd);
    if (c2o) memcpy(c2o, c2, sizeof(double) * d);
    free(W1);
}

void oracle_ttt_mlp(int B, int H, int T, int d, int h, int b, int ln_res, int rule, int tail, const double *Q,
                    const double *K, const double *V, const double *eta, const double *W10,
                    const double *c10, const double *W20, const double *c20, long w_bstride,
                    long c1_bstride, long c2_bstride, const double *ln_g, const double *ln_b,
                    double eps, double *Z, double *W1o, double *c1o, double *W2o, double *c2o,
                    double *loss, double *inner_loss, int nthreads)
{
    const long chains = (long)B * H;
    const size_t hd = (size_t)h * d;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long ch = 0; ch < chains; ++ch) {
        const long bi = ch / H, hi = ch % H;
        const size_t tok = (size_t)ch * T;
        mlp_chain(T, d, h, b, ln_res, rule, tail, Q + tok * d, K + tok * d, V + tok * d, eta + tok,
                  W10 + bi * w_bstride + hi * hd, c10 + bi * c1_bstride + hi * (size_t)h,
                  W20 + bi * w_bstride + hi * hd, c20 + bi * c2_bstride + hi * (size_t)d,
                  ln_g + hi * (size_t)d, ln_b + hi * (size_t)d, eps, Z + tok * d,
                  W1o ? W1o + (size_t)ch * hd : NULL, c1o ? c1o + (size_t)ch * h : NULL,
                  W2o ? W2o + (size_t)ch * hd : NULL, c2o ? c2o + (size_t)ch * d : NULL,
                  loss ? loss + tok : NULL, inner_loss ? inner_loss + tok : NULL);
    }
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
