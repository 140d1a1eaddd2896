/*
 * ttt_oracle.c -- plain, slow, single-threaded CPU oracle for the TTT layer's
 * inner loop (TTT-Linear and TTT-MLP, optional residual LayerNorm), forward only.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA path.
 *
 * Everything is IEEE double.  The sources are the pages collected for this
 * method (test_sequence_layers_08):
 *   [R]  damodev.csdn.net TTT article, section 3.1, the update/apply equation:
 *        W_t = W_{t-1} - eta * grad_W l(W_{t-1}; x_t),  o_t = f(x_t; W_t)
 *        (the output uses the weights AFTER the token's own update).
 *   [MB] same article, section 4.1: mini-batch TTT -- every gradient inside a
 *        mini-batch is taken at the mini-batch's starting weights.
 *   [D]  same article, section 4.2 (compute_mini_batch excerpt): target
 *        XV - XK, Z1 = XK @ W1 + b1, LayerNorm-fused L2 backward, dual form with
 *        tril(XQ XK^T), W1_last = W1_init - (eta*XK)^T G, b1_last = b1_init - sum(eta*G).
 *   [I]  same article, section 4.3: W1 is [heads, d, d] row-major, b1 [heads, 1, d].
 *   [F]  lryc.cn "测试时学习（TTT）" article, section 2.1: TTT-MLP is d -> 4d
 *        GELU -> d; residual form f(x) = x + LN(f_res(x)).
 *   [G]  same lryc.cn article, section 2.2: the learnable per-token learning
 *        rate eta(x) = eta_base * sigmoid(theta_lr . x).
 *   [M]  ai-feeds "Modular TTT" page, method overview: the loss (MSE or inner
 *        product) and weight decay are design dimensions of the inner learner.
 *
 * Readings where the pages are silent (all of them are also listed in the
 * design notes):
 *   - loss is 1/2 ||f(k) - v||^2 summed over the d features (no 1/d; a 1/d
 *     lives in eta when the caller wants it);
 *   - gradients inside a mini-batch are summed with per-token eta (no 1/b);
 *   - the token-s term of the dual form is scaled by eta_s (source token);
 *   - with the residual form the loss is 1/2 ||LN(z) - (v - k)||^2, because
 *     f(k) - v = k + LN(z) - v;
 *   - LayerNorm uses the biased variance and eps passed by the caller; the same
 *     gamma/beta serve the loss and the output;
 *   - GELU is the tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 *   - [M] gives no formulas; the readings taken: the inner-product loss is
 *     l = -<f(k), v>; weight decay lambda adds 1/2 lambda ||W||^2 to each
 *     token's loss for the weight matrices (W; W1, W2), not the biases, so a
 *     token's step is W -= eta_t (grad_W l_t + lambda W) with both terms taken
 *     at the mini-batch's starting weights like every other gradient [MB].
 *
 * Parity pins (what ties this file to something other than itself) live in
 * the CPU tests: autograd brute force of the definition, b = 1 online GD, eta = 0,
 * the single-mini-batch closed form, causal linear attention with zero initial
 * weights, primal == dual, finite differences of every hand-derived gradient,
 * the state carry, and a hand-worked d = 1 example.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEM 2

/* ------------------------------------------------------------------------ */
/* Per-token learning rate [G]                                               */
/* ------------------------------------------------------------------------ */

/* eta[b, h, t] = eta_base * sigmoid(theta[h] . x[b, t]) for x [B, L, Dx] (the
 * layer's input tokens) and theta [H, Dx] (one gate vector per head); eta is
 * [B, H, L].  sigmoid(u) = 1 / (1 + exp(-u)). */
int oracle_eta_gate(int B, int H, int L, int Dx, double eta_base, const double *x,
                    const double *theta, double *eta)
{
    if (B <= 0 || H <= 0 || L <= 0 || Dx <= 0 || !x || !theta || !eta) return ORACLE_BAD_ARG;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int t = 0; t < L; ++t) {
                const double *xt = x + ((size_t)b * L + t) * Dx;
                const double *th = theta + (size_t)h * Dx;
                double u = 0.0;
                for (int k = 0; k < Dx; ++k) u += th[k] * xt[k];
                eta[((size_t)b * H + h) * L + t] = eta_base / (1.0 + exp(-u));
            }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Elementwise pieces                                                        */
/* ------------------------------------------------------------------------ */

/* GELU, tanh form ([F] section 2.1 names GELU; the tanh form is the reading). */
double oracle_gelu(double x)
{
    const double s = sqrt(2.0 / M_PI);
    double u = s * (x + 0.044715 * x * x * x);
    return 0.5 * x * (1.0 + tanh(u));
}

/* d/dx of oracle_gelu, differentiated by hand. */
double oracle_gelu_prime(double x)
{
    const double s = sqrt(2.0 / M_PI);
    double u = s * (x + 0.044715 * x * x * x);
    double th = tanh(u);
    double du = s * (1.0 + 3.0 * 0.044715 * x * x);
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * du;
}

/* LayerNorm over n features: out = gamma * (z - mean) / sqrt(var + eps) + beta,
 * biased variance.  gamma/beta may be NULL (meaning 1 and 0). */
void oracle_ln_fwd(const double *z, int n, const double *gamma, const double *beta,
                   double eps, double *out)
{
    double mu = 0.0, var = 0.0;
    for (int i = 0; i < n; ++i) mu += z[i];
    mu /= n;
    for (int i = 0; i < n; ++i) var += (z[i] - mu) * (z[i] - mu);
    var /= n;
    double r = 1.0 / sqrt(var + eps);
    for (int i = 0; i < n; ++i) {
        double g = gamma ? gamma[i] : 1.0;
        double b = beta ? beta[i] : 0.0;
        out[i] = g * (z[i] - mu) * r + b;
    }
}

/* Gradient w.r.t. z of 1/2 || LN(z) - y ||^2, derived by hand ([D] section 4.2
 * calls this the LayerNorm-fused L2 backward):
 *   xh = (z - mu) r,  e = gamma xh + beta - y,  gx = gamma e,
 *   g  = r (gx - mean(gx) - xh mean(gx xh)). */
void oracle_ln_l2_bwd(const double *z, const double *y, int n, const double *gamma,
                      const double *beta, double eps, double *g)
{
    double mu = 0.0, var = 0.0;
    for (int i = 0; i < n; ++i) mu += z[i];
    mu /= n;
    for (int i = 0; i < n; ++i) var += (z[i] - mu) * (z[i] - mu);
    var /= n;
    double r = 1.0 / sqrt(var + eps);
    double *xh = (double *)malloc(sizeof(double) * (size_t)n);
    double *gx = (double *)malloc(sizeof(double) * (size_t)n);
    double m1 = 0.0, m2 = 0.0;
    for (int i = 0; i < n; ++i) {
        double gm = gamma ? gamma[i] : 1.0;
        double bt = beta ? beta[i] : 0.0;
        xh[i] = (z[i] - mu) * r;
        double e = gm * xh[i] + bt - y[i];
        gx[i] = gm * e;
        m1 += gx[i];
        m2 += gx[i] * xh[i];
    }
    m1 /= n;
    m2 /= n;
    for (int i = 0; i < n; ++i) g[i] = r * (gx[i] - m1 - xh[i] * m2);
    free(xh);
    free(gx);
}

/* Gradient w.r.t. z of a loss whose gradient w.r.t. LN(z) is u, by hand:
 *   xh = (z - mu) r,  gx = gamma u,  g = r (gx - mean(gx) - xh mean(gx xh)). */
static void ln_bwd_upstream(const double *z, const double *u, int n, const double *gamma,
                            double eps, double *g)
{
    double mu = 0.0, var = 0.0;
    for (int i = 0; i < n; ++i) mu += z[i];
    mu /= n;
    for (int i = 0; i < n; ++i) var += (z[i] - mu) * (z[i] - mu);
    var /= n;
    double r = 1.0 / sqrt(var + eps);
    double m1 = 0.0, m2 = 0.0;
    for (int i = 0; i < n; ++i) {
        double gx = (gamma ? gamma[i] : 1.0) * u[i];
        m1 += gx;
        m2 += gx * (z[i] - mu) * r;
    }
    m1 /= n;
    m2 /= n;
    for (int i = 0; i < n; ++i) {
        double gx = (gamma ? gamma[i] : 1.0) * u[i];
        g[i] = r * (gx - m1 - (z[i] - mu) * r * m2);
    }
}

/* dl/dz of one token for the loss `loss` (0: 1/2 ||f(k) - v||^2, 1: -<f(k), v>) with
 * f(k) = z (ln = 0) or k + LN(z) (ln = 1); y is scratch of n values. */
static void token_dz(const double *z, const double *k, const double *v, int n, int ln, int loss,
                     const double *gamma, const double *beta, double eps, double *y, double *g)
{
    if (loss == 1) {
        for (int j = 0; j < n; ++j) y[j] = -v[j];
        if (ln)
            ln_bwd_upstream(z, y, n, gamma, eps, g);
        else
            memcpy(g, y, sizeof(double) * (size_t)n);
    } else if (ln) {
        for (int j = 0; j < n; ++j) y[j] = v[j] - k[j];
        oracle_ln_l2_bwd(z, y, n, gamma, beta, eps, g);
    } else {
        for (int j = 0; j < n; ++j) g[j] = z[j] - v[j];
    }
}

/* The token loss from the output o = f(k): 1/2 ||o - v||^2 or -<o, v>. */
static double token_loss_value(const double *o, const double *v, int n, int loss)
{
    double l = 0.0;
    for (int j = 0; j < n; ++j) l += loss == 1 ? -o[j] * v[j] : 0.5 * (o[j] - v[j]) * (o[j] - v[j]);
    return l;
}

/* ------------------------------------------------------------------------ */
/* TTT-Linear: f(k) = k W + c  (row-vector convention of [D]/[I]),            */
/* residual form f(k) = k + LN(k W + c).                                      */
/* ------------------------------------------------------------------------ */

/* z = x W + c for one row; W is n_in x n_out row-major. */
static void row_times(const double *x, const double *W, const double *c, int n_in,
                      int n_out, double *z)
{
    for (int j = 0; j < n_out; ++j) z[j] = c ? c[j] : 0.0;
    for (int i = 0; i < n_in; ++i) {
        double xi = x[i];
        const double *Wi = W + (size_t)i * n_out;
        for (int j = 0; j < n_out; ++j) z[j] += xi * Wi[j];
    }
}

/* Per-token loss (1/2 ||f(k) - v||^2 or -<f(k), v>) at weights (W, c). */
double oracle_linear_token_loss_v(const double *k, const double *v, const double *W,
                                  const double *c, int d, int ln, int loss, const double *gamma,
                                  const double *beta, double eps)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)d);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    row_times(k, W, c, d, d, z);
    if (ln) {
        oracle_ln_fwd(z, d, gamma, beta, eps, o);
        for (int j = 0; j < d; ++j) o[j] += k[j];
    } else {
        memcpy(o, z, sizeof(double) * (size_t)d);
    }
    double l = token_loss_value(o, v, d, loss);
    free(z);
    free(o);
    return l;
}

double oracle_linear_token_loss(const double *k, const double *v, const double *W,
                                const double *c, int d, int ln, const double *gamma,
                                const double *beta, double eps)
{
    return oracle_linear_token_loss_v(k, v, W, c, d, ln, 0, gamma, beta, eps);
}

/* Hand gradient of the token loss: g = dl/dz; dl/dW = k^T g; dl/dc = g. */
void oracle_linear_token_grad_v(const double *k, const double *v, const double *W,
                                const double *c, int d, int ln, int loss, const double *gamma,
                                const double *beta, double eps, double *gW, double *gc)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)d);
    double *g = (double *)malloc(sizeof(double) * (size_t)d);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    row_times(k, W, c, d, d, z);
    token_dz(z, k, v, d, ln, loss, gamma, beta, eps, y, g);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) gW[(size_t)i * d + j] = k[i] * g[j];
    for (int j = 0; j < d; ++j) gc[j] = g[j];
    free(z);
    free(g);
    free(y);
}

void oracle_linear_token_grad(const double *k, const double *v, const double *W,
                              const double *c, int d, int ln, const double *gamma,
                              const double *beta, double eps, double *gW, double *gc)
{
    oracle_linear_token_grad_v(k, v, W, c, d, ln, 0, gamma, beta, eps, gW, gc);
}

/* Offsets of the initial state for (batch bi, head hi). */
static size_t init_index(int bi, int hi, int H, int per_batch)
{
    return per_batch ? (size_t)bi * H + hi : (size_t)hi;
}

/*
 * TTT-Linear forward, per-token primal form ([R] + [MB]).
 *   Q,K,V,Z: [B,H,L,d]; eta: [B,H,L]; W0: [H,d,d] (or [B,H,d,d] when
 *   init_per_batch); b0: [H,d] (or [B,H,d]); gamma, beta: [H,d] (used iff ln).
 *   W_final: [B,H,d,d]; b_final: [B,H,d].
 * For each mini-batch: gradients g_s for every token at the starting (W, c);
 * then, token by token, W -= eta_t k_t^T g_t, c -= eta_t g_t, and the output is
 * f(q_t) at the updated weights.
 */
int oracle_ttt_linear_v(int B, int H, int L, int d, int mb, int ln, double eps,
                        int init_per_batch, int loss, double wd, const double *Q,
                        const double *K, const double *V, const double *eta, const double *W0,
                        const double *b0, const double *gamma, const double *beta,
                        double *Z, double *W_final, double *b_final)
{
    if (B <= 0 || H <= 0 || L <= 0 || d <= 0 || mb <= 0 || L % mb != 0) return ORACLE_BAD_ARG;
    size_t dd = (size_t)d * d;
    double *W = (double *)malloc(sizeof(double) * dd);
    double *Ws = (double *)malloc(sizeof(double) * dd);
    double *c = (double *)malloc(sizeof(double) * (size_t)d);
    double *cs = (double *)malloc(sizeof(double) * (size_t)d);
    double *G = (double *)malloc(sizeof(double) * (size_t)mb * d);
    double *gW = (double *)malloc(sizeof(double) * dd);
    double *z = (double *)malloc(sizeof(double) * (size_t)d);
    if (!W || !Ws || !c || !cs || !G || !gW || !z) return ORACLE_NO_MEM;

    for (int bi = 0; bi < B; ++bi) {
        for (int hi = 0; hi < H; ++hi) {
            size_t bh = (size_t)bi * H + hi;
            size_t ii = init_index(bi, hi, H, init_per_batch);
            memcpy(W, W0 + ii * dd, sizeof(double) * dd);
            memcpy(c, b0 + ii * d, sizeof(double) * (size_t)d);
            const double *gm = ln ? gamma + (size_t)hi * d : NULL;
            const double *bt = ln ? beta + (size_t)hi * d : NULL;
            for (int n0 = 0; n0 < L; n0 += mb) {
                memcpy(Ws, W, sizeof(double) * dd);
                memcpy(cs, c, sizeof(double) * (size_t)d);
                /* every gradient of the mini-batch at its starting weights [MB] */
                for (int s = 0; s < mb; ++s) {
                    size_t row = (bh * L + n0 + s) * d;
                    oracle_linear_token_grad_v(K + row, V + row, Ws, cs, d, ln, loss, gm, bt, eps,
                                               gW, G + (size_t)s * d);
                }
                /* token-by-token update, then apply with the updated weights [R] */
                for (int t = 0; t < mb; ++t) {
                    size_t row = (bh * L + n0 + t) * d;
                    double et = eta[bh * L + n0 + t];
                    const double *kt = K + row;
                    const double *gt = G + (size_t)t * d;
                    /* W -= eta_t (k_t^T g_t + lambda W_start) */
                    for (int i = 0; i < d; ++i)
                        for (int j = 0; j < d; ++j)
                            W[(size_t)i * d + j] -= et * (kt[i] * gt[j] + wd * Ws[(size_t)i * d + j]);
                    for (int j = 0; j < d; ++j) c[j] -= et * gt[j];
                    row_times(Q + row, W, c, d, d, z);
                    if (ln) {
                        oracle_ln_fwd(z, d, gm, bt, eps, Z + row);
                        for (int j = 0; j < d; ++j) Z[row + j] += Q[row + j];
                    } else {
                        memcpy(Z + row, z, sizeof(double) * (size_t)d);
                    }
                }
            }
            memcpy(W_final + bh * dd, W, sizeof(double) * dd);
            memcpy(b_final + bh * d, c, sizeof(double) * (size_t)d);
        }
    }
    free(W); free(Ws); free(c); free(cs); free(G); free(gW); free(z);
    return ORACLE_OK;
}

int oracle_ttt_linear(int B, int H, int L, int d, int mb, int ln, double eps,
                      int init_per_batch, const double *Q, const double *K,
                      const double *V, const double *eta, const double *W0,
                      const double *b0, const double *gamma, const double *beta,
                      double *Z, double *W_final, double *b_final)
{
    return oracle_ttt_linear_v(B, H, L, d, mb, ln, eps, init_per_batch, 0, 0.0, Q, K, V, eta,
                               W0, b0, gamma, beta, Z, W_final, b_final);
}

/*
 * TTT-Linear forward, dual form, written separately from the primal above and
 * used only to check primal == dual.  Per mini-batch ([D] section 4.2):
 *   Zk   = K W + 1 c,   G = dl/dZk (row by row),
 *   A    = tril(Q K^T + 1) with column s scaled by eta_s (diagonal included),
 *   Zbar = Q W + 1 c - A G,    W <- W - K^T diag(eta) G,   c <- c - eta^T G.
 * The "+1" carries the bias: c_t = c - sum_{s<=t} eta_s g_s.
 * With weight decay lambda the Q W term of token t is scaled by
 * 1 - lambda sum_{s<=t} eta_s, and the carry by 1 - lambda sum_s eta_s.
 */
int oracle_ttt_linear_dual_v(int B, int H, int L, int d, int mb, int ln, double eps,
                             int init_per_batch, int loss, double wd, const double *Q,
                             const double *K, const double *V, const double *eta,
                             const double *W0, const double *b0, const double *gamma,
                             const double *beta, double *Z, double *W_final, double *b_final)
{
    if (B <= 0 || H <= 0 || L <= 0 || d <= 0 || mb <= 0 || L % mb != 0) return ORACLE_BAD_ARG;
    size_t dd = (size_t)d * d;
    double *W = (double *)malloc(sizeof(double) * dd);
    double *c = (double *)malloc(sizeof(double) * (size_t)d);
    double *Zk = (double *)malloc(sizeof(double) * (size_t)mb * d);
    double *G = (double *)malloc(sizeof(double) * (size_t)mb * d);
    double *A = (double *)malloc(sizeof(double) * (size_t)mb * mb);
    double *zb = (double *)malloc(sizeof(double) * (size_t)d);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    if (!W || !c || !Zk || !G || !A || !zb || !y) return ORACLE_NO_MEM;

    for (int bi = 0; bi < B; ++bi) {
        for (int hi = 0; hi < H; ++hi) {
            size_t bh = (size_t)bi * H + hi;
            size_t ii = init_index(bi, hi, H, init_per_batch);
            memcpy(W, W0 + ii * dd, sizeof(double) * dd);
            memcpy(c, b0 + ii * d, sizeof(double) * (size_t)d);
            const double *gm = ln ? gamma + (size_t)hi * d : NULL;
            const double *bt = ln ? beta + (size_t)hi * d : NULL;
            for (int n0 = 0; n0 < L; n0 += mb) {
                const double *Kn = K + (bh * L + n0) * d;
                const double *Qn = Q + (bh * L + n0) * d;
                const double *Vn = V + (bh * L + n0) * d;
                const double *en = eta + bh * L + n0;
                /* Zk and G */
                for (int s = 0; s < mb; ++s) {
                    row_times(Kn + (size_t)s * d, W, c, d, d, Zk + (size_t)s * d);
                    token_dz(Zk + (size_t)s * d, Kn + (size_t)s * d, Vn + (size_t)s * d, d, ln, loss,
                             gm, bt, eps, y, G + (size_t)s * d);
                }
                /* A = tril(Q K^T + 1) diag(eta) */
                for (int t = 0; t < mb; ++t)
                    for (int s = 0; s < mb; ++s) {
                        double a = 0.0;
                        if (s <= t) {
                            for (int i = 0; i < d; ++i) a += Qn[(size_t)t * d + i] * Kn[(size_t)s * d + i];
                            a = (a + 1.0) * en[s];
                        }
                        A[(size_t)t * mb + s] = a;
                    }
                /* outputs with the mini-batch's starting W (decay-scaled) */
                double cum = 0.0;
                for (int t = 0; t < mb; ++t) {
                    cum += en[t];
                    row_times(Qn + (size_t)t * d, W, NULL, d, d, zb);
                    for (int j = 0; j < d; ++j) zb[j] = (1.0 - wd * cum) * zb[j] + c[j];
                    for (int s = 0; s <= t; ++s)
                        for (int j = 0; j < d; ++j) zb[j] -= A[(size_t)t * mb + s] * G[(size_t)s * d + j];
                    double *zo = Z + (bh * L + n0 + t) * d;
                    if (ln) {
                        oracle_ln_fwd(zb, d, gm, bt, eps, zo);
                        for (int j = 0; j < d; ++j) zo[j] += Qn[(size_t)t * d + j];
                    } else {
                        memcpy(zo, zb, sizeof(double) * (size_t)d);
                    }
                }
                /* carry: W <- (1 - lambda sum eta) W - K^T diag(eta) G, c -= eta^T G */
                for (size_t i = 0; i < dd; ++i) W[i] *= 1.0 - wd * cum;
                for (int s = 0; s < mb; ++s)
                    for (int i = 0; i < d; ++i) {
                        double ks = en[s] * Kn[(size_t)s * d + i];
                        for (int j = 0; j < d; ++j) W[(size_t)i * d + j] -= ks * G[(size_t)s * d + j];
                    }
                for (int s = 0; s < mb; ++s)
                    for (int j = 0; j < d; ++j) c[j] -= en[s] * G[(size_t)s * d + j];
            }
            memcpy(W_final + bh * dd, W, sizeof(double) * dd);
            memcpy(b_final + bh * d, c, sizeof(double) * (size_t)d);
        }
    }
    free(W); free(c); free(Zk); free(G); free(A); free(zb); free(y);
    return ORACLE_OK;
}

int oracle_ttt_linear_dual(int B, int H, int L, int d, int mb, int ln, double eps,
                           int init_per_batch, const double *Q, const double *K,
                           const double *V, const double *eta, const double *W0,
                           const double *b0, const double *gamma, const double *beta,
                           double *Z, double *W_final, double *b_final)
{
    return oracle_ttt_linear_dual_v(B, H, L, d, mb, ln, eps, init_per_batch, 0, 0.0, Q, K, V,
                                    eta, W0, b0, gamma, beta, Z, W_final, b_final);
}

/* ------------------------------------------------------------------------ */
/* TTT-MLP ([F] section 2.1): f_res(k) = GELU(k W1 + b1) W2 + b2, W1: d x dh,  */
/* W2: dh x d; residual form f(k) = k + LN(f_res(k)).                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    double *z1, *x2, *z2, *g2, *gx2, *g1, *y, *o;
} mlp_scratch;

static int mlp_scratch_alloc(mlp_scratch *s, int d, int dh)
{
    s->z1 = (double *)malloc(sizeof(double) * (size_t)dh);
    s->x2 = (double *)malloc(sizeof(double) * (size_t)dh);
    s->gx2 = (double *)malloc(sizeof(double) * (size_t)dh);
    s->g1 = (double *)malloc(sizeof(double) * (size_t)dh);
    s->z2 = (double *)malloc(sizeof(double) * (size_t)d);
    s->g2 = (double *)malloc(sizeof(double) * (size_t)d);
    s->y = (double *)malloc(sizeof(double) * (size_t)d);
    s->o = (double *)malloc(sizeof(double) * (size_t)d);
    return s->z1 && s->x2 && s->gx2 && s->g1 && s->z2 && s->g2 && s->y && s->o;
}

static void mlp_scratch_free(mlp_scratch *s)
{
    free(s->z1); free(s->x2); free(s->gx2); free(s->g1);
    free(s->z2); free(s->g2); free(s->y); free(s->o);
}

/* Forward of the fast-weight MLP for one row; fills z1, x2, z2 and o = f(x). */
static void mlp_row_forward(const double *x, const double *W1, const double *b1,
                            const double *W2, const double *b2, int d, int dh, int ln,
                            const double *gamma, const double *beta, double eps,
                            mlp_scratch *s)
{
    row_times(x, W1, b1, d, dh, s->z1);
    for (int m = 0; m < dh; ++m) s->x2[m] = oracle_gelu(s->z1[m]);
    row_times(s->x2, W2, b2, dh, d, s->z2);
    if (ln) {
        oracle_ln_fwd(s->z2, d, gamma, beta, eps, s->o);
        for (int j = 0; j < d; ++j) s->o[j] += x[j];
    } else {
        memcpy(s->o, s->z2, sizeof(double) * (size_t)d);
    }
}

double oracle_mlp_token_loss_v(const double *k, const double *v, const double *W1,
                               const double *b1, const double *W2, const double *b2, int d,
                               int dh, int ln, int loss, const double *gamma, const double *beta,
                               double eps)
{
    mlp_scratch s;
    if (!mlp_scratch_alloc(&s, d, dh)) return NAN;
    mlp_row_forward(k, W1, b1, W2, b2, d, dh, ln, gamma, beta, eps, &s);
    double l = token_loss_value(s.o, v, d, loss);
    mlp_scratch_free(&s);
    return l;
}

double oracle_mlp_token_loss(const double *k, const double *v, const double *W1,
                             const double *b1, const double *W2, const double *b2, int d,
                             int dh, int ln, const double *gamma, const double *beta,
                             double eps)
{
    return oracle_mlp_token_loss_v(k, v, W1, b1, W2, b2, d, dh, ln, 0, gamma, beta, eps);
}

/* Hand back-propagation through the fast-weight MLP for one token:
 *   g2 = dl/dz2 (LN-fused L2 backward against v - k, or z2 - v),
 *   g1 = (g2 W2^T) * GELU'(z1),
 *   dW1 = k^T g1, db1 = g1, dW2 = x2^T g2, db2 = g2.
 * Outputs g1 (dh), g2 (d) and x2 (dh); the weight gradients are the outer
 * products above (formed by the callers).  `loss` as for token_dz. */
static void mlp_token_backward(const double *k, const double *v, const double *W1,
                               const double *b1, const double *W2, const double *b2,
                               int d, int dh, int ln, int loss, const double *gamma,
                               const double *beta, double eps, mlp_scratch *s)
{
    mlp_row_forward(k, W1, b1, W2, b2, d, dh, ln, gamma, beta, eps, s);
    token_dz(s->z2, k, v, d, ln, loss, gamma, beta, eps, s->y, s->g2);
    for (int m = 0; m < dh; ++m) {
        double a = 0.0;
        const double *W2m = W2 + (size_t)m * d;
        for (int j = 0; j < d; ++j) a += s->g2[j] * W2m[j];
        s->gx2[m] = a;
        s->g1[m] = a * oracle_gelu_prime(s->z1[m]);
    }
}

void oracle_mlp_token_grad_v(const double *k, const double *v, const double *W1,
                             const double *b1, const double *W2, const double *b2, int d,
                             int dh, int ln, int loss, const double *gamma, const double *beta,
                             double eps, double *gW1, double *gb1, double *gW2, double *gb2)
{
    mlp_scratch s;
    if (!mlp_scratch_alloc(&s, d, dh)) return;
    mlp_token_backward(k, v, W1, b1, W2, b2, d, dh, ln, loss, gamma, beta, eps, &s);
    for (int i = 0; i < d; ++i)
        for (int m = 0; m < dh; ++m) gW1[(size_t)i * dh + m] = k[i] * s.g1[m];
    for (int m = 0; m < dh; ++m) gb1[m] = s.g1[m];
    for (int m = 0; m < dh; ++m)
        for (int j = 0; j < d; ++j) gW2[(size_t)m * d + j] = s.x2[m] * s.g2[j];
    for (int j = 0; j < d; ++j) gb2[j] = s.g2[j];
    mlp_scratch_free(&s);
}

void oracle_mlp_token_grad(const double *k, const double *v, const double *W1,
                           const double *b1, const double *W2, const double *b2, int d,
                           int dh, int ln, const double *gamma, const double *beta,
                           double eps, double *gW1, double *gb1, double *gW2, double *gb2)
{
    oracle_mlp_token_grad_v(k, v, W1, b1, W2, b2, d, dh, ln, 0, gamma, beta, eps, gW1, gb1, gW2,
                            gb2);
}

/*
 * TTT-MLP forward, per-token primal form ([R] + [MB] + [F]).
 *   W1_0: [H,d,dh] (or [B,H,d,dh]), b1_0: [H,dh], W2_0: [H,dh,d], b2_0: [H,d];
 *   finals are [B,H,...].  Other arrays as for oracle_ttt_linear.
 */
int oracle_ttt_mlp_v(int B, int H, int L, int d, int dh, int mb, int ln, double eps,
                     int init_per_batch, int loss, double wd, const double *Q, const double *K,
                     const double *V, const double *eta, const double *W1_0,
                     const double *b1_0, const double *W2_0, const double *b2_0,
                     const double *gamma, const double *beta, double *Z, double *W1_f,
                     double *b1_f, double *W2_f, double *b2_f)
{
    if (B <= 0 || H <= 0 || L <= 0 || d <= 0 || dh <= 0 || mb <= 0 || L % mb != 0)
        return ORACLE_BAD_ARG;
    size_t n1 = (size_t)d * dh;
    double *W1 = (double *)malloc(sizeof(double) * n1);
    double *W2 = (double *)malloc(sizeof(double) * n1);
    double *W1s = (double *)malloc(sizeof(double) * n1);
    double *W2s = (double *)malloc(sizeof(double) * n1);
    double *b1 = (double *)malloc(sizeof(double) * (size_t)dh);
    double *b2 = (double *)malloc(sizeof(double) * (size_t)d);
    double *b1s = (double *)malloc(sizeof(double) * (size_t)dh);
    double *b2s = (double *)malloc(sizeof(double) * (size_t)d);
    double *G1 = (double *)malloc(sizeof(double) * (size_t)mb * dh);
    double *G2 = (double *)malloc(sizeof(double) * (size_t)mb * d);
    double *X2 = (double *)malloc(sizeof(double) * (size_t)mb * dh);
    mlp_scratch s;
    if (!W1 || !W2 || !W1s || !W2s || !b1 || !b2 || !b1s || !b2s || !G1 || !G2 || !X2 ||
        !mlp_scratch_alloc(&s, d, dh))
        return ORACLE_NO_MEM;

    for (int bi = 0; bi < B; ++bi) {
        for (int hi = 0; hi < H; ++hi) {
            size_t bh = (size_t)bi * H + hi;
            size_t ii = init_index(bi, hi, H, init_per_batch);
            memcpy(W1, W1_0 + ii * n1, sizeof(double) * n1);
            memcpy(W2, W2_0 + ii * n1, sizeof(double) * n1);
            memcpy(b1, b1_0 + ii * dh, sizeof(double) * (size_t)dh);
            memcpy(b2, b2_0 + ii * d, sizeof(double) * (size_t)d);
            const double *gm = ln ? gamma + (size_t)hi * d : NULL;
            const double *bt = ln ? beta + (size_t)hi * d : NULL;
            for (int n0 = 0; n0 < L; n0 += mb) {
                memcpy(W1s, W1, sizeof(double) * n1);
                memcpy(W2s, W2, sizeof(double) * n1);
                memcpy(b1s, b1, sizeof(double) * (size_t)dh);
                memcpy(b2s, b2, sizeof(double) * (size_t)d);
                for (int t = 0; t < mb; ++t) {
                    size_t row = (bh * L + n0 + t) * d;
                    mlp_token_backward(K + row, V + row, W1s, b1s, W2s, b2s, d, dh, ln, loss,
                                       gm, bt, eps, &s);
                    memcpy(G1 + (size_t)t * dh, s.g1, sizeof(double) * (size_t)dh);
                    memcpy(G2 + (size_t)t * d, s.g2, sizeof(double) * (size_t)d);
                    memcpy(X2 + (size_t)t * dh, s.x2, sizeof(double) * (size_t)dh);
                }
                for (int t = 0; t < mb; ++t) {
                    size_t row = (bh * L + n0 + t) * d;
                    double et = eta[bh * L + n0 + t];
                    const double *kt = K + row;
                    const double *g1 = G1 + (size_t)t * dh;
                    const double *g2 = G2 + (size_t)t * d;
                    const double *x2 = X2 + (size_t)t * dh;
                    for (int i = 0; i < d; ++i)
                        for (int m = 0; m < dh; ++m)
                            W1[(size_t)i * dh + m] -= et * (kt[i] * g1[m] + wd * W1s[(size_t)i * dh + m]);
                    for (int m = 0; m < dh; ++m) b1[m] -= et * g1[m];
                    for (int m = 0; m < dh; ++m)
                        for (int j = 0; j < d; ++j)
                            W2[(size_t)m * d + j] -= et * (x2[m] * g2[j] + wd * W2s[(size_t)m * d + j]);
                    for (int j = 0; j < d; ++j) b2[j] -= et * g2[j];
                    mlp_row_forward(Q + row, W1, b1, W2, b2, d, dh, ln, gm, bt, eps, &s);
                    memcpy(Z + row, s.o, sizeof(double) * (size_t)d);
                }
            }
            memcpy(W1_f + bh * n1, W1, sizeof(double) * n1);
            memcpy(W2_f + bh * n1, W2, sizeof(double) * n1);
            memcpy(b1_f + bh * dh, b1, sizeof(double) * (size_t)dh);
            memcpy(b2_f + bh * d, b2, sizeof(double) * (size_t)d);
        }
    }
    free(W1); free(W2); free(W1s); free(W2s); free(b1); free(b2); free(b1s); free(b2s);
    free(G1); free(G2); free(X2);
    mlp_scratch_free(&s);
    return ORACLE_OK;
}

int oracle_ttt_mlp(int B, int H, int L, int d, int dh, int mb, int ln, double eps,
                   int init_per_batch, const double *Q, const double *K, const double *V,
                   const double *eta, const double *W1_0, const double *b1_0,
                   const double *W2_0, const double *b2_0, const double *gamma,
                   const double *beta, double *Z, double *W1_f, double *b1_f,
                   double *W2_f, double *b2_f)
{
    return oracle_ttt_mlp_v(B, H, L, d, dh, mb, ln, eps, init_per_batch, 0, 0.0, Q, K, V, eta,
                            W1_0, b1_0, W2_0, b2_0, gamma, beta, Z, W1_f, b1_f, W2_f, b2_f);
}

/*
 * TTT-MLP forward, dual form (separately written; only for primal == dual).
 * Per mini-batch, with the starting weights:
 *   Z1 = K W1 + 1 b1, X2 = GELU(Z1), Z2 = X2 W2 + 1 b2, G2, G1 as in the primal;
 *   Zb1 = Q W1 + 1 b1 - (tril(Q K^T + 1) diag(eta)) G1,   Xb2 = GELU(Zb1),
 *   Zb2 = Xb2 W2 + 1 b2 - (tril(Xb2 X2^T + 1) diag(eta)) G2,
 *   out = Q + LN(Zb2) (or Zb2);  then W1 -= K^T diag(eta) G1, b1 -= eta^T G1,
 *   W2 -= X2^T diag(eta) G2, b2 -= eta^T G2.
 * With weight decay lambda, token t's Q W1 and Xb2 W2 terms are scaled by
 * 1 - lambda sum_{s<=t} eta_s and the carried W1, W2 by 1 - lambda sum_s eta_s.
 */
int oracle_ttt_mlp_dual_v(int B, int H, int L, int d, int dh, int mb, int ln, double eps,
                          int init_per_batch, int loss, double wd, const double *Q,
                          const double *K, const double *V, const double *eta,
                          const double *W1_0, const double *b1_0, const double *W2_0,
                          const double *b2_0, const double *gamma, const double *beta,
                          double *Z, double *W1_f, double *b1_f, double *W2_f, double *b2_f)
{
    if (B <= 0 || H <= 0 || L <= 0 || d <= 0 || dh <= 0 || mb <= 0 || L % mb != 0)
        return ORACLE_BAD_ARG;
    size_t n1 = (size_t)d * dh;
    double *W1 = (double *)malloc(sizeof(double) * n1);
    double *W2 = (double *)malloc(sizeof(double) * n1);
    double *b1 = (double *)malloc(sizeof(double) * (size_t)dh);
    double *b2 = (double *)malloc(sizeof(double) * (size_t)d);
    double *Z1 = (double *)malloc(sizeof(double) * (size_t)mb * dh);
    double *X2 = (double *)malloc(sizeof(double) * (size_t)mb * dh);
    double *Z2 = (double *)malloc(sizeof(double) * (size_t)mb * d);
    double *G1 = (double *)malloc(sizeof(double) * (size_t)mb * dh);
    double *G2 = (double *)malloc(sizeof(double) * (size_t)mb * d);
    double *Zb1 = (double *)malloc(sizeof(double) * (size_t)mb * dh);
    double *Xb2 = (double *)malloc(sizeof(double) * (size_t)mb * dh);
    double *Zb2 = (double *)malloc(sizeof(double) * (size_t)mb * d);
    double *A = (double *)malloc(sizeof(double) * (size_t)mb * mb);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    if (!W1 || !W2 || !b1 || !b2 || !Z1 || !X2 || !Z2 || !G1 || !G2 || !Zb1 || !Xb2 ||
        !Zb2 || !A || !y)
        return ORACLE_NO_MEM;

    for (int bi = 0; bi < B; ++bi) {
        for (int hi = 0; hi < H; ++hi) {
            size_t bh = (size_t)bi * H + hi;
            size_t ii = init_index(bi, hi, H, init_per_batch);
            memcpy(W1, W1_0 + ii * n1, sizeof(double) * n1);
            memcpy(W2, W2_0 + ii * n1, sizeof(double) * n1);
            memcpy(b1, b1_0 + ii * dh, sizeof(double) * (size_t)dh);
            memcpy(b2, b2_0 + ii * d, sizeof(double) * (size_t)d);
            const double *gm = ln ? gamma + (size_t)hi * d : NULL;
            const double *bt = ln ? beta + (size_t)hi * d : NULL;
            for (int n0 = 0; n0 < L; n0 += mb) {
                const double *Kn = K + (bh * L + n0) * d;
                const double *Qn = Q + (bh * L + n0) * d;
                const double *Vn = V + (bh * L + n0) * d;
                const double *en = eta + bh * L + n0;
                for (int s = 0; s < mb; ++s) {
                    row_times(Kn + (size_t)s * d, W1, b1, d, dh, Z1 + (size_t)s * dh);
                    for (int m = 0; m < dh; ++m)
                        X2[(size_t)s * dh + m] = oracle_gelu(Z1[(size_t)s * dh + m]);
                    row_times(X2 + (size_t)s * dh, W2, b2, dh, d, Z2 + (size_t)s * d);
                    token_dz(Z2 + (size_t)s * d, Kn + (size_t)s * d, Vn + (size_t)s * d, d, ln, loss,
                             gm, bt, eps, y, G2 + (size_t)s * d);
                    for (int m = 0; m < dh; ++m) {
                        double a = 0.0;
                        for (int j = 0; j < d; ++j) a += G2[(size_t)s * d + j] * W2[(size_t)m * d + j];
                        G1[(size_t)s * dh + m] = a * oracle_gelu_prime(Z1[(size_t)s * dh + m]);
                    }
                }
                /* first layer, query side */
                for (int t = 0; t < mb; ++t)
                    for (int s = 0; s < mb; ++s) {
                        double a = 0.0;
                        if (s <= t) {
                            for (int i = 0; i < d; ++i) a += Qn[(size_t)t * d + i] * Kn[(size_t)s * d + i];
                            a = (a + 1.0) * en[s];
                        }
                        A[(size_t)t * mb + s] = a;
                    }
                double cum = 0.0;
                for (int t = 0; t < mb; ++t) {
                    cum += en[t];
                    row_times(Qn + (size_t)t * d, W1, NULL, d, dh, Zb1 + (size_t)t * dh);
                    for (int m = 0; m < dh; ++m)
                        Zb1[(size_t)t * dh + m] = (1.0 - wd * cum) * Zb1[(size_t)t * dh + m] + b1[m];
                    for (int s = 0; s <= t; ++s)
                        for (int m = 0; m < dh; ++m)
                            Zb1[(size_t)t * dh + m] -= A[(size_t)t * mb + s] * G1[(size_t)s * dh + m];
                    for (int m = 0; m < dh; ++m)
                        Xb2[(size_t)t * dh + m] = oracle_gelu(Zb1[(size_t)t * dh + m]);
                }
                /* second layer, query side */
                for (int t = 0; t < mb; ++t)
                    for (int s = 0; s < mb; ++s) {
                        double a = 0.0;
                        if (s <= t) {
                            for (int m = 0; m < dh; ++m) a += Xb2[(size_t)t * dh + m] * X2[(size_t)s * dh + m];
                            a = (a + 1.0) * en[s];
                        }
                        A[(size_t)t * mb + s] = a;
                    }
                cum = 0.0;
                for (int t = 0; t < mb; ++t) {
                    cum += en[t];
                    row_times(Xb2 + (size_t)t * dh, W2, NULL, dh, d, Zb2 + (size_t)t * d);
                    for (int j = 0; j < d; ++j)
                        Zb2[(size_t)t * d + j] = (1.0 - wd * cum) * Zb2[(size_t)t * d + j] + b2[j];
                    for (int s = 0; s <= t; ++s)
                        for (int j = 0; j < d; ++j)
                            Zb2[(size_t)t * d + j] -= A[(size_t)t * mb + s] * G2[(size_t)s * d + j];
                    double *zo = Z + (bh * L + n0 + t) * d;
                    if (ln) {
                        oracle_ln_fwd(Zb2 + (size_t)t * d, d, gm, bt, eps, zo);
                        for (int j = 0; j < d; ++j) zo[j] += Qn[(size_t)t * d + j];
                    } else {
                        memcpy(zo, Zb2 + (size_t)t * d, sizeof(double) * (size_t)d);
                    }
                }
                /* carry (cum is now the mini-batch's sum of eta) */
                for (size_t i = 0; i < n1; ++i) {
                    W1[i] *= 1.0 - wd * cum;
                    W2[i] *= 1.0 - wd * cum;
                }
                for (int s = 0; s < mb; ++s) {
                    for (int i = 0; i < d; ++i) {
                        double ks = en[s] * Kn[(size_t)s * d + i];
                        for (int m = 0; m < dh; ++m) W1[(size_t)i * dh + m] -= ks * G1[(size_t)s * dh + m];
                    }
                    for (int m = 0; m < dh; ++m) b1[m] -= en[s] * G1[(size_t)s * dh + m];
                    for (int m = 0; m < dh; ++m) {
                        double xs = en[s] * X2[(size_t)s * dh + m];
                        for (int j = 0; j < d; ++j) W2[(size_t)m * d + j] -= xs * G2[(size_t)s * d + j];
                    }
                    for (int j = 0; j < d; ++j) b2[j] -= en[s] * G2[(size_t)s * d + j];
                }
            }
            memcpy(W1_f + bh * n1, W1, sizeof(double) * n1);
            memcpy(W2_f + bh * n1, W2, sizeof(double) * n1);
            memcpy(b1_f + bh * dh, b1, sizeof(double) * (size_t)dh);
            memcpy(b2_f + bh * d, b2, sizeof(double) * (size_t)d);
        }
    }
    free(W1); free(W2); free(b1); free(b2); free(Z1); free(X2); free(Z2); free(G1);
    free(G2); free(Zb1); free(Xb2); free(Zb2); free(A); free(y);
    return ORACLE_OK;
}

int oracle_ttt_mlp_dual(int B, int H, int L, int d, int dh, int mb, int ln, double eps,
                        int init_per_batch, const double *Q, const double *K,
                        const double *V, const double *eta, const double *W1_0,
                        const double *b1_0, const double *W2_0, const double *b2_0,
                        const double *gamma, const double *beta, double *Z, double *W1_f,
                        double *b1_f, double *W2_f, double *b2_f)
{
    return oracle_ttt_mlp_dual_v(B, H, L, d, dh, mb, ln, eps, init_per_batch, 0, 0.0, Q, K, V,
                                 eta, W1_0, b1_0, W2_0, b2_0, gamma, beta, Z, W1_f, b1_f, W2_f,
                                 b2_f);
}
