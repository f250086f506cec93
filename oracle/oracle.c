/*
 * Reference oracle for the normalization-fused Conv1d blocks (TEST INFRASTRUCTURE).
 *
 * Plain, slow, fp64 CPU code that evaluates each block straight from its
 * definition.  It exists only to check the CUDA library: only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * Sources (the three PopcornBench transcript pages; citations give the page
 * title and the passage):
 *   [P1] "Kimi-K2.6 l2_p12" (pre-norm residual block) -- opening problem
 *        statement: residual = x; x = BatchNorm1d(x); x = ReLU(x);
 *        x = Conv1d(x, k=3, padding=dilation, dilation); out = x + residual.
 *        Eval-mode BN: (x - running_mean)/sqrt(running_var + eps)*gamma + beta.
 *        Conv taps read t - padding + k*dilation; zero padding is applied to
 *        the conv input, i.e. after BN and ReLU.
 *   [P2] "FW-GLM-5-1 l2_p35" (Conv1d + GroupNorm) -- problem analysis:
 *        conv sum over c_in and k of x[n, c_in, t*stride - padding + k*dilation]
 *        * weight[c_out, c_in, k]; GroupNorm per (n, group) over the group's
 *        channels and all time steps, biased variance, then gamma/beta.
 *   [P3] "Kimi-K2.6 l2_p97" (Linear + BatchNorm1d + bias + divide + Swish) --
 *        training-mode BN uses the batch mean and biased variance; running
 *        stats follow new = (1 - momentum)*old + momentum*batch with the
 *        unbiased variance; then (y + bias)/divide and x*sigmoid(x).
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 * OpenMP (when compiled with -fopenmp) parallelises over independent output
 * rows; the arithmetic of each output element is the same sequential sum in
 * either case.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * [P1] BatchNorm1d in eval mode followed by ReLU, for one element.
 * The expression is evaluated in the order the page writes it.
 * ------------------------------------------------------------------------ */
static double bn_eval_relu(double xv, double rm, double rv, double gamma,
                           double beta, double eps)
{
    double y = (xv - rm) / sqrt(rv + eps) * gamma + beta;
    return y > 0.0 ? y : 0.0;
}

/*
 * [P1] Pre-norm residual block, for a chosen set of output rows (n, o).
 *
 *   z[n,c,s]  = relu(bn(x[n,c,s]))         for 0 <= s < L, else 0
 *   y[n,o,t]  = bias[o] + sum_c sum_k w[o,c,k] * z[n,c, t - padding + k*dilation]
 *   out[n,o,t] = x[n,o,t] + y[n,o,t]
 *
 * The Conv1d output length is L + 2*padding - dilation*(K-1); the residual add
 * needs it to equal L, which is checked.  rows_n/rows_o give the rows to
 * compute; out_rows receives nrows x L values (row r is (rows_n[r], rows_o[r])).
 * bias may be NULL (no conv bias).
 */
static void block_row(const double *x, int C, int L, int K, int dilation,
                      int padding, const double *rm, const double *rv,
                      const double *gamma, const double *beta, double eps,
                      const double *w, const double *bias, int n, int o, double *row)
{
    const double *xn = x + (size_t)n * C * L;
    for (int t = 0; t < L; ++t) row[t] = bias ? bias[o] : 0.0;
    /* Each row[t] receives the terms in the order c = 0..C-1, k = 0..K-1. */
    for (int c = 0; c < C; ++c) {
        const double *xc = xn + (size_t)c * L;
        for (int k = 0; k < K; ++k) {
            const double wk = w[((size_t)o * C + c) * K + k];
            for (int t = 0; t < L; ++t) {
                const int s = t - padding + k * dilation;
                if (s < 0 || s >= L) continue;              /* zero-padded z */
                row[t] += wk * bn_eval_relu(xc[s], rm[c], rv[c], gamma[c], beta[c], eps);
            }
        }
    }
    const double *xo = xn + (size_t)o * L;
    for (int t = 0; t < L; ++t) row[t] += xo[t];           /* residual */
}

int oracle_prenorm_block_rows(const double *x, int N, int C, int L, int K,
                              int dilation, int padding,
                              const double *rm, const double *rv,
                              const double *gamma, const double *beta, double eps,
                              const double *w, const double *bias,
                              const int *rows_n, const int *rows_o, int nrows,
                              double *out_rows, int nthreads)
{
    if (N <= 0 || C <= 0 || L <= 0 || K <= 0 || dilation <= 0 || padding < 0)
        return -1;
    if (L + 2 * padding - dilation * (K - 1) != L) return -2;
    for (int r = 0; r < nrows; ++r)
        if (rows_n[r] < 0 || rows_n[r] >= N || rows_o[r] < 0 || rows_o[r] >= C)
            return -3;
    set_threads(nthreads);
    #pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < nrows; ++r)
        block_row(x, C, L, K, dilation, padding, rm, rv, gamma, beta, eps, w, bias,
                  rows_n[r], rows_o[r], out_rows + (size_t)r * L);
    return 0;
}

/* [P1] Whole pre-norm residual block: every row (n, o), out is (N, C, L). */
int oracle_prenorm_block(const double *x, double *out, int N, int C, int L, int K,
                         int dilation, int padding,
                         const double *rm, const double *rv, const double *gamma,
                         const double *beta, double eps,
                         const double *w, const double *bias, int nthreads)
{
    if (N <= 0 || C <= 0 || L <= 0 || K <= 0 || dilation <= 0 || padding < 0)
        return -1;
    if (L + 2 * padding - dilation * (K - 1) != L) return -2;
    set_threads(nthreads);
    #pragma omp parallel for schedule(dynamic)
    for (int nc = 0; nc < N * C; ++nc)
        block_row(x, C, L, K, dilation, padding, rm, rv, gamma, beta, eps, w, bias,
                  nc / C, nc % C, out + (size_t)nc * L);
    return 0;
}

/* ------------------------------------------------------------------------
 * [P1] The same block with BatchNorm1d in training mode.  The page's
 * correctness discussion sets batch statistics against running statistics:
 * in training mode channel c is normalized with the mean and the biased
 * variance of x[:, c, :] over all N*L values, and the running buffers move
 * toward the batch values ([P3] states the rule and the update, with the
 * unbiased variance, for the BatchNorm1d after its Linear).
 *
 *   mu[c]  = sum_{n,s} x[n,c,s] / (N*L)
 *   var[c] = sum_{n,s} (x[n,c,s] - mu[c])^2 / (N*L)            (second pass)
 *   running_mean[c] <- (1 - momentum)*running_mean[c] + momentum*mu[c]
 *   running_var[c]  <- (1 - momentum)*running_var[c]
 *                      + momentum*var[c]*(N*L)/(N*L - 1)
 *   out = the eval-mode block above with mu, var in place of the running
 *         statistics (the running buffers' old values are not used).
 *
 * batch_mean and batch_var (C each) receive mu and var.  running_mean and
 * running_var may be NULL (no update).  rows_n == NULL computes every row
 * (out_rows is then (N, C, L)); otherwise the nrows rows (rows_n[r], rows_o[r]).
 * ------------------------------------------------------------------------ */
int oracle_prenorm_block_train(const double *x, int N, int C, int L, int K,
                               int dilation, int padding,
                               double *running_mean, double *running_var,
                               const double *gamma, const double *beta, double eps,
                               double momentum, const double *w, const double *bias,
                               const int *rows_n, const int *rows_o, int nrows,
                               double *out_rows, double *batch_mean, double *batch_var,
                               int nthreads)
{
    if (N <= 0 || C <= 0 || L <= 0 || K <= 0 || dilation <= 0 || padding < 0)
        return -1;
    if (L + 2 * padding - dilation * (K - 1) != L) return -2;
    const double cnt = (double)N * (double)L;
    if (cnt < 2.0) return -4;                   /* the unbiased variance needs N*L-1 */
    if (!batch_mean || !batch_var) return -5;
    if (rows_n)
        for (int r = 0; r < nrows; ++r)
            if (rows_n[r] < 0 || rows_n[r] >= N || rows_o[r] < 0 || rows_o[r] >= C)
                return -3;
    set_threads(nthreads);

    #pragma omp parallel for schedule(static)
    for (int c = 0; c < C; ++c) {
        double s = 0.0;
        for (int n = 0; n < N; ++n) {
            const double *xc = x + ((size_t)n * C + c) * L;
            for (int t = 0; t < L; ++t) s += xc[t];
        }
        const double mu = s / cnt;
        double ss = 0.0;
        for (int n = 0; n < N; ++n) {
            const double *xc = x + ((size_t)n * C + c) * L;
            for (int t = 0; t < L; ++t) {
                const double d = xc[t] - mu;
                ss += d * d;
            }
        }
        const double var = ss / cnt;
        batch_mean[c] = mu;
        batch_var[c] = var;
        if (running_mean)
            running_mean[c] = (1.0 - momentum) * running_mean[c] + momentum * mu;
        if (running_var)
            running_var[c] = (1.0 - momentum) * running_var[c] +
                             momentum * var * cnt / (cnt - 1.0);
    }

    if (!rows_n) {
        #pragma omp parallel for schedule(dynamic)
        for (int nc = 0; nc < N * C; ++nc)
            block_row(x, C, L, K, dilation, padding, batch_mean, batch_var, gamma, beta, eps,
                      w, bias, nc / C, nc % C, out_rows + (size_t)nc * L);
    } else {
        #pragma omp parallel for schedule(dynamic)
        for (int r = 0; r < nrows; ++r)
            block_row(x, C, L, K, dilation, padding, batch_mean, batch_var, gamma, beta, eps,
                      w, bias, rows_n[r], rows_o[r], out_rows + (size_t)r * L);
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * [P2] Conv1d followed by GroupNorm.
 *
 *   T_out = floor((T + 2*padding - dilation*(K-1) - 1)/stride) + 1
 *   y[n,o,t] = bias[o] + sum_c sum_k w[o,c,k] * x[n,c, t*stride - padding + k*dilation]
 *              (x taken as 0 outside [0, T); bias may be NULL)
 *   group g of channel o is o / (C_out/G)
 *   mu[n,g]  = mean of y over the group's C_out/G channels and all T_out steps
 *   var[n,g] = mean of (y - mu)^2 over the same set (biased; two passes)
 *   out = (y - mu)/sqrt(var + eps) * gamma[o] + beta[o]   (gamma/beta NULL: affine off)
 *
 * groups_n/groups_g choose the (n, g) groups to compute; out_groups receives,
 * per chosen group, (C_out/G) x T_out values (channel-major), and mean_var
 * (if not NULL) receives (mu, var) per chosen group.
 * ------------------------------------------------------------------------ */
int oracle_conv1d_out_len(int T, int K, int stride, int padding, int dilation)
{
    return (T + 2 * padding - dilation * (K - 1) - 1) / stride + 1;
}

static void gn_group(const double *x, int Cin, int Cout, int T, int K, int stride,
                     int padding, int dilation, const double *w, const double *bias,
                     int G, const double *gamma, const double *beta, double eps,
                     int n, int g, double *yg, double *mean_var)
{
    const int To = oracle_conv1d_out_len(T, K, stride, padding, dilation);
    const int cpg = Cout / G;
    const double *xn = x + (size_t)n * Cin * T;
    /* convolution for the group's channels */
    for (int j = 0; j < cpg; ++j) {
        const int o = g * cpg + j;
        double *yrow = yg + (size_t)j * To;
        for (int t = 0; t < To; ++t) yrow[t] = bias ? bias[o] : 0.0;
        for (int c = 0; c < Cin; ++c) {
            const double *xc = xn + (size_t)c * T;
            for (int k = 0; k < K; ++k) {
                const double wk = w[((size_t)o * Cin + c) * K + k];
                for (int t = 0; t < To; ++t) {
                    const int s = t * stride - padding + k * dilation;
                    if (s < 0 || s >= T) continue;          /* zero padding */
                    yrow[t] += wk * xc[s];
                }
            }
        }
    }
    /* group statistics: mean, then the biased variance about it */
    const size_t cnt = (size_t)cpg * To;
    double sum = 0.0;
    for (size_t i = 0; i < cnt; ++i) sum += yg[i];
    const double mu = sum / (double)cnt;
    double ss = 0.0;
    for (size_t i = 0; i < cnt; ++i) ss += (yg[i] - mu) * (yg[i] - mu);
    const double var = ss / (double)cnt;
    if (mean_var) { mean_var[0] = mu; mean_var[1] = var; }
    const double inv = 1.0 / sqrt(var + eps);
    for (int j = 0; j < cpg; ++j) {
        const int o = g * cpg + j;
        double *yrow = yg + (size_t)j * To;
        for (int t = 0; t < To; ++t) {
            double v = (yrow[t] - mu) * inv;
            if (gamma) v = v * gamma[o];
            if (beta) v = v + beta[o];
            yrow[t] = v;
        }
    }
}

static int gn_check(int N, int Cin, int Cout, int T, int K, int stride, int padding,
                    int dilation, int G)
{
    if (N <= 0 || Cin <= 0 || Cout <= 0 || T <= 0 || K <= 0 || stride <= 0 ||
        padding < 0 || dilation <= 0 || G <= 0)
        return -1;
    if (Cout % G != 0) return -2;
    if (oracle_conv1d_out_len(T, K, stride, padding, dilation) <= 0) return -3;
    return 0;
}

int oracle_conv_groupnorm_groups(const double *x, int N, int Cin, int Cout, int T,
                                 int K, int stride, int padding, int dilation,
                                 const double *w, const double *bias, int G,
                                 const double *gamma, const double *beta, double eps,
                                 const int *groups_n, const int *groups_g, int ngroups,
                                 double *out_groups, double *mean_var, int nthreads)
{
    int rc = gn_check(N, Cin, Cout, T, K, stride, padding, dilation, G);
    if (rc) return rc;
    const int To = oracle_conv1d_out_len(T, K, stride, padding, dilation);
    const int cpg = Cout / G;
    for (int r = 0; r < ngroups; ++r)
        if (groups_n[r] < 0 || groups_n[r] >= N || groups_g[r] < 0 || groups_g[r] >= G)
            return -4;
    set_threads(nthreads);
    #pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < ngroups; ++r)
        gn_group(x, Cin, Cout, T, K, stride, padding, dilation, w, bias, G, gamma,
                 beta, eps, groups_n[r], groups_g[r],
                 out_groups + (size_t)r * cpg * To, mean_var ? mean_var + 2 * r : NULL);
    return 0;
}

/* [P2] Whole Conv1d + GroupNorm: out is (N, C_out, T_out).  The channels of
 * group (n, g) are a contiguous block, at out + (n*G + g) * (C_out/G) * T_out. */
int oracle_conv_groupnorm(const double *x, double *out, int N, int Cin, int Cout, int T,
                          int K, int stride, int padding, int dilation,
                          const double *w, const double *bias, int G,
                          const double *gamma, const double *beta, double eps,
                          int nthreads)
{
    int rc = gn_check(N, Cin, Cout, T, K, stride, padding, dilation, G);
    if (rc) return rc;
    const int To = oracle_conv1d_out_len(T, K, stride, padding, dilation);
    const int cpg = Cout / G;
    set_threads(nthreads);
    #pragma omp parallel for schedule(dynamic)
    for (int ng = 0; ng < N * G; ++ng)
        gn_group(x, Cin, Cout, T, K, stride, padding, dilation, w, bias, G, gamma,
                 beta, eps, ng / G, ng % G, out + (size_t)ng * cpg * To, NULL);
    return 0;
}

/* ------------------------------------------------------------------------
 * [P3] Linear + BatchNorm1d + scalar bias + divide + Swish, for chosen
 * output columns j (BatchNorm1d statistics are per column, over the batch).
 *
 *   y[b,j]  = sum_i x[b,i] * W[j,i] + b_lin[j]           (b_lin may be NULL)
 *   training: mu_j = mean_b y[b,j];  var_j = mean_b (y[b,j] - mu_j)^2   (biased)
 *             running_mean[j] = (1-m)*running_mean[j] + m*mu_j
 *             running_var[j]  = (1-m)*running_var[j]  + m*var_j*B/(B-1)
 *   eval:     mu_j = running_mean[j]; var_j = running_var[j]; no update
 *   yhat = (y - mu_j)/sqrt(var_j + eps)*gamma[j] + beta[j]  (gamma/beta NULL: 1/0)
 *   u    = (yhat + add_bias)/divide_value
 *   out  = u * sigmoid(u),  sigmoid(u) = 1/(1+exp(-u)), evaluated as
 *          exp(u)/(1+exp(u)) for u < 0 so that exp never overflows.
 *
 * cols/ncols choose the columns; out_cols receives B x ncols values (row-major,
 * column r of the block is column cols[r]).  running_mean/running_var are
 * indexed by the true column j and updated in place when training.
 * ------------------------------------------------------------------------ */
static double sigmoid(double u)
{
    if (u >= 0.0) return 1.0 / (1.0 + exp(-u));
    const double e = exp(u);
    return e / (1.0 + e);
}

int oracle_linear_bn_swish_cols(const double *x, int B, int IN, int OUT,
                                const double *W, const double *b_lin,
                                const double *gamma, const double *beta,
                                double *running_mean, double *running_var,
                                double eps, double momentum, int training,
                                double add_bias, double divide_value,
                                const int *cols, int ncols, double *out_cols,
                                double *batch_mean_var, int nthreads)
{
    if (B <= 0 || IN <= 0 || OUT <= 0) return -1;
    if (training && B < 2) return -2;           /* unbiased variance needs B-1 */
    for (int r = 0; r < ncols; ++r)
        if (cols[r] < 0 || cols[r] >= OUT) return -3;
    set_threads(nthreads);

    #pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < ncols; ++r) {
        const int j = cols[r];
        const double *wj = W + (size_t)j * IN;
        double *y = out_cols;                  /* column r lives at y[b*ncols + r] */
        for (int b = 0; b < B; ++b) {
            const double *xb = x + (size_t)b * IN;
            double acc = 0.0;
            for (int i = 0; i < IN; ++i) acc += xb[i] * wj[i];
            y[(size_t)b * ncols + r] = acc + (b_lin ? b_lin[j] : 0.0);
        }
        double mu, var;
        if (training) {
            double s = 0.0;
            for (int b = 0; b < B; ++b) s += y[(size_t)b * ncols + r];
            mu = s / B;
            double ss = 0.0;
            for (int b = 0; b < B; ++b) {
                const double dv = y[(size_t)b * ncols + r] - mu;
                ss += dv * dv;
            }
            var = ss / B;
            if (running_mean)
                running_mean[j] = (1.0 - momentum) * running_mean[j] + momentum * mu;
            if (running_var)
                running_var[j] = (1.0 - momentum) * running_var[j] +
                                 momentum * var * (double)B / (double)(B - 1);
        } else {
            mu = running_mean[j];
            var = running_var[j];
        }
        if (batch_mean_var) { batch_mean_var[2 * r] = mu; batch_mean_var[2 * r + 1] = var; }
        const double inv = 1.0 / sqrt(var + eps);
        const double g = gamma ? gamma[j] : 1.0, be = beta ? beta[j] : 0.0;
        for (int b = 0; b < B; ++b) {
            double v = (y[(size_t)b * ncols + r] - mu) * inv * g + be;
            double u = (v + add_bias) / divide_value;
            y[(size_t)b * ncols + r] = u * sigmoid(u);
        }
    }
    return 0;
}
