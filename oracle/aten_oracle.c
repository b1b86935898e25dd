/*
 * The unfused form of softmax cross-entropy: CPU float64 oracle.
 *
 * TEST INFRASTRUCTURE ONLY, like ce_oracle.c: only the tests, the smoke
 * check and the benchmark's CPU baseline may call it, and it shares no code
 * with the CUDA library.
 *
 * Source (page title, section): "[tt-crank] fuse cross entropy onto the
 * ttml cross_entropy_fw/bw composites", tenstorrent/tt-mlir pull request
 * #9324: the table of aten ops the cross-entropy decomposes to
 * (_log_softmax on [1023, 128256] f32, nll_loss_forward; backward
 * nll_loss_backward and _log_softmax_backward_data), and the #9339
 * description quoted there (log-probabilities of [rows x C], integer
 * targets with ignore_index, mean/sum/none; _log_softmax as a max-shifted
 * log-sum-exp; an all-ignored batch gets zero gradients). Class weights,
 * which that lowering leaves out, follow the aten operators' own
 * definitions (weight w[c] per class, total_weight = sum of w[t_i] over
 * the rows that are not ignored).
 *
 * Inputs are double arrays (a caller converts its storage exactly); sums
 * use Neumaier's compensated summation.
 */
#include <math.h>
#include <stdint.h>

enum { AO_NONE = 0, AO_SUM = 1, AO_MEAN = 2 };
enum { AO_OK = 0, AO_BAD_ARG = 1, AO_TARGET_RANGE = 2 };

typedef struct { double s, c; } asum;

static void aadd(asum* a, double v) {
    double t = a->s + v;
    if (fabs(a->s) >= fabs(v)) a->c += (a->s - t) + v;
    else a->c += (v - t) + a->s;
    a->s = t;
}

static double aval(const asum* a) { return a->s + a->c; }

static double wt(const double* weight, int64_t c) { return weight ? weight[c] : 1.0; }

/*
 * _log_softmax over the last dimension: out[i, j] = x[i, j] - m_i - log S_i
 * with m_i = max_j x[i, j] and S_i = sum_j exp(x[i, j] - m_i).
 */
int ao_log_softmax(const double* x, int64_t rows, int64_t C, double* out) {
    if (rows < 0 || C <= 0) return AO_BAD_ARG;
    for (int64_t i = 0; i < rows; ++i) {
        const double* xr = x + i * C;
        double m = -INFINITY;
        for (int64_t j = 0; j < C; ++j)
            if (xr[j] > m) m = xr[j];
        asum s = {0.0, 0.0};
        for (int64_t j = 0; j < C; ++j) aadd(&s, exp(xr[j] - m));
        const double lse = m + log(aval(&s));
        for (int64_t j = 0; j < C; ++j) out[i * C + j] = xr[j] - lse;
    }
    return AO_OK;
}

/*
 * nll_loss_forward: per row l_i = -w[t_i] * logp[i, t_i] (0 when t_i is
 * ignore_index). "none" writes the rows' l_i to out[0 .. rows-1] and
 * total_weight 0; "sum" writes sum l_i; "mean" writes sum l_i / W with
 * W = sum of w[t_i] over the counted rows (NaN when W is 0). total_weight
 * receives W for "sum" and "mean". A target outside [0, C) that is not
 * ignore_index is an error.
 */
int ao_nll_forward(const double* logp, const int64_t* target, const double* weight,
                   int64_t rows, int64_t C, int64_t ignore_index, int reduction,
                   double* out, double* total_weight) {
    if (rows < 0 || C <= 0) return AO_BAD_ARG;
    if (reduction != AO_NONE && reduction != AO_SUM && reduction != AO_MEAN) return AO_BAD_ARG;
    asum L = {0.0, 0.0}, W = {0.0, 0.0};
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t t = target[i];
        double l = 0.0;
        if (t != ignore_index) {
            if (t < 0 || t >= C) return AO_TARGET_RANGE;
            l = -wt(weight, t) * logp[i * C + t];
            aadd(&L, l);
            aadd(&W, wt(weight, t));
        }
        if (reduction == AO_NONE) out[i] = l;
    }
    if (reduction == AO_NONE) {
        *total_weight = 0.0;
    } else {
        *total_weight = aval(&W);
        out[0] = reduction == AO_SUM ? aval(&L) : aval(&L) / aval(&W);
    }
    return AO_OK;
}

/*
 * nll_loss_backward: grad[i, j] = 0 except grad[i, t_i] = -w[t_i] * g_i for
 * counted rows, with g_i = grad_output[i] ("none"), grad_output[0] ("sum")
 * or grad_output[0] / total_weight ("mean"). An all-ignored batch has no
 * counted row, so every gradient is zero whatever total_weight is.
 */
int ao_nll_backward(const double* grad_output, const int64_t* target, const double* weight,
                    int64_t rows, int64_t C, int64_t ignore_index, int reduction,
                    double total_weight, double* grad) {
    if (rows < 0 || C <= 0) return AO_BAD_ARG;
    if (reduction != AO_NONE && reduction != AO_SUM && reduction != AO_MEAN) return AO_BAD_ARG;
    for (int64_t k = 0; k < rows * C; ++k) grad[k] = 0.0;
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t t = target[i];
        if (t == ignore_index) continue;
        if (t < 0 || t >= C) return AO_TARGET_RANGE;
        double g = reduction == AO_NONE ? grad_output[i] : grad_output[0];
        if (reduction == AO_MEAN) g /= total_weight;
        grad[i * C + t] = -wt(weight, t) * g;
    }
    return AO_OK;
}

/*
 * _log_softmax_backward_data: with y = log_softmax(x) and dy the incoming
 * gradient, dx[i, j] = dy[i, j] - exp(y[i, j]) * sum_k dy[i, k] (the
 * Jacobian of log-softmax applied to dy).
 */
int ao_log_softmax_backward(const double* dy, const double* y, int64_t rows, int64_t C,
                            double* dx) {
    if (rows < 0 || C <= 0) return AO_BAD_ARG;
    for (int64_t i = 0; i < rows; ++i) {
        asum s = {0.0, 0.0};
        for (int64_t j = 0; j < C; ++j) aadd(&s, dy[i * C + j]);
        const double sd = aval(&s);
        for (int64_t j = 0; j < C; ++j)
            dx[i * C + j] = dy[i * C + j] - exp(y[i * C + j]) * sd;
    }
    return AO_OK;
}
