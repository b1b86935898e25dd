/*
 * Fused softmax cross-entropy: CPU float64 oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do. It shares no code, header, table or helper with the CUDA
 * library: it is a plain, slow, single-threaded restatement of what the
 * method computes, written so that a reader can check it against the pages
 * by eye.
 *
 * Sources followed (page title, section):
 *  - "Kernel Profile: CrossEntropy (Tier 3 - Fused/Complex)" (Liger-Kernel):
 *      §Forward Pass (inputs, outputs, reductions, softcap, ignore_index,
 *      class weights, label smoothing, z_loss, token accuracy, predicted
 *      tokens; exp and log are the precision-sensitive ops),
 *      §Backward Pass (the gradient is produced by the forward; backward
 *      only scales it by grad_output),
 *      §Module Parameters (ignore_index default -100, lse_square_scale),
 *      §Key Patterns (max-shifted log-sum-exp; loss = CE + label-smoothing
 *      loss + z-loss, each contributing to loss and gradient).
 *  - "[tt-crank] fuse cross entropy onto the ttml cross_entropy_fw/bw
 *      composites", tenstorrent/tt-mlir pull request #9324:
 *      review comments on the mean reduction (an all-ignored batch keeps the
 *      NaN forward loss and gets exactly zero gradients, as PyTorch does;
 *      the mean divides by total_weight), the checklist (non-finite logits
 *      in ignored rows must not leak), and the #9339 description
 *      (max-shifted log-sum-exp, because log(softmax) overflows past a
 *      logit gap of about 87).
 *
 * Readings where the pages are silent (each also listed in the design
 * notes): label smoothing takes PyTorch's form, with class weights inside
 * the smoothing sum; the weighted mean divides every term (NLL, smoothing,
 * z-loss) by D = sum of w[t_i] over non-ignored rows; z-loss is the
 * unweighted lse_square_scale * lse^2 of the softcapped logits; argmax runs
 * over the raw logits and the lowest index wins ties; an ignored row has
 * loss 0, gradient +0 and predicted token -1, and its logits are never
 * read; accuracy is n_correct / n_valid (a 0/1 value per row under "none").
 *
 * Arithmetic: every input element is converted exactly to double (bf16,
 * fp16 and fp32 embed exactly in binary64); sums use Neumaier's compensated
 * summation.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2, ORC_F16 = 3 };
enum { ORC_NONE = 0, ORC_SUM = 1, ORC_MEAN = 2 };
enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_TARGET_RANGE = 2 };

/* ---- exact storage decoding ------------------------------------------ */

/* A bf16 value is the upper half of an IEEE binary32 with the same bits;
 * widening it (then to binary64) is exact. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: sign bit, 5 exponent bits with bias 15, 10 fraction
 * bits. Exponent field 0 holds zero and the subnormals (fraction * 2^-24);
 * 31 holds the infinities (fraction 0) and NaN; otherwise the value is
 * (1024 + fraction) * 2^(exponent - 25). Every value is exact in double. */
static double f16_bits_to_double(uint16_t bits) {
    const int e = (bits >> 10) & 0x1F;
    const int f = bits & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return (bits & 0x8000) ? -v : v;
}

static double logit(const void* x, int dtype, int64_t k) {
    switch (dtype) {
    case ORC_F64: return ((const double*)x)[k];
    case ORC_F32: return (double)((const float*)x)[k];
    case ORC_F16: return f16_bits_to_double(((const uint16_t*)x)[k]);
    default: return bf16_bits_to_double(((const uint16_t*)x)[k]);
    }
}

/* ---- Neumaier compensated summation ---------------------------------- */

typedef struct { double s, c; } nsum;

static void nadd(nsum* a, double v) {
    double t = a->s + v;
    if (fabs(a->s) >= fabs(v)) a->c += (a->s - t) + v;
    else a->c += (v - t) + a->s;
    a->s = t;
}

static double nval(const nsum* a) { return a->s + a->c; }

/* ---- one row ---------------------------------------------------------- */

/* Softcap (Forward Pass: "softcap: float or None"): z = s * tanh(x / s)
 * when s > 0, otherwise z = x. Returns z and, through dzdx, its derivative
 * 1 - tanh^2(x / s). */
static double softcapped(double x, double s, double* dzdx) {
    if (s > 0.0) {
        double th = tanh(x / s);
        *dzdx = 1.0 - th * th;
        return s * th;
    }
    *dzdx = 1.0;
    return x;
}

typedef struct {
    int valid;       /* target != ignore_index */
    double loss;     /* l_i, before any reduction */
    double zloss;    /* lse_square_scale * lse^2 */
    double lse;
    int64_t pred;    /* argmax of the raw logits, lowest index; -1 if ignored */
    int correct;     /* pred == target */
    double w_t;      /* weight of the target class (1 without weights) */
} row_out;

static double class_weight(const double* weight, int64_t j) {
    return weight ? weight[j] : 1.0;
}

/*
 * Computes one row. xr points at the row's V logits. If grad_row is not
 * NULL it receives grad_scale * d l_i / d x_j for every j.
 *
 * With z = softcap(x), lse = log sum_j exp(z_j) (max-shifted),
 * p_j = exp(z_j - lse), t the target, w the class weights (all 1 when
 * absent), eps the label smoothing and lam the lse_square_scale:
 *
 *   l_i = (1 - eps) * w_t * (lse - z_t)             cross-entropy (NLL)
 *       + (eps / V) * sum_j w_j * (lse - z_j)       label smoothing
 *       + lam * lse^2                               z-loss
 *
 *   d l_i / d z_k = (1 - eps) * w_t * (p_k - [k == t])
 *                 + (eps / V) * (W * p_k - w_k),   W = sum_j w_j
 *                 + 2 * lam * lse * p_k
 *   d l_i / d x_k = d l_i / d z_k * dz_k / dx_k
 */
static int one_row(const void* x, int dtype, int64_t row, int64_t V, int64_t t,
                   const double* weight, int64_t ignore_index, double eps,
                   double lam, double softcap, double grad_scale,
                   double* grad_row, row_out* out) {
    const int64_t base = row * V;
    memset(out, 0, sizeof *out);
    out->pred = -1;

    if (t == ignore_index) {
        /* Ignored row: its logits are never read, so inf or NaN there
         * cannot reach any output; its gradient is exactly +0. */
        if (grad_row)
            for (int64_t j = 0; j < V; ++j) grad_row[j] = 0.0;
        return ORC_OK;
    }
    if (t < 0 || t >= V) return ORC_TARGET_RANGE;
    out->valid = 1;

    /* Max of z and argmax of the raw x (first occurrence wins). */
    double m = -INFINITY, xbest = -INFINITY;
    int64_t arg = 0;
    for (int64_t j = 0; j < V; ++j) {
        double d;
        double xj = logit(x, dtype, base + j);
        double zj = softcapped(xj, softcap, &d);
        if (zj > m) m = zj;
        if (j == 0 || xj > xbest) { xbest = xj; arg = j; }
    }

    /* lse = m + log sum_j exp(z_j - m): the max-shifted log-sum-exp. */
    nsum S = {0, 0};
    for (int64_t j = 0; j < V; ++j) {
        double d;
        double zj = softcapped(logit(x, dtype, base + j), softcap, &d);
        nadd(&S, exp(zj - m));
    }
    const double lse = m + log(nval(&S));

    double dzt;
    const double zt = softcapped(logit(x, dtype, base + t), softcap, &dzt);
    const double wt = class_weight(weight, t);

    /* Label-smoothing sum over all classes: sum_j w_j * (lse - z_j). */
    nsum smooth = {0, 0}, Wsum = {0, 0};
    for (int64_t j = 0; j < V; ++j) {
        double d;
        double zj = softcapped(logit(x, dtype, base + j), softcap, &d);
        double wj = class_weight(weight, j);
        nadd(&smooth, wj * (lse - zj));
        nadd(&Wsum, wj);
    }
    const double W = nval(&Wsum);

    out->lse = lse;
    out->zloss = lam * lse * lse;
    out->loss = (1.0 - eps) * wt * (lse - zt) + (eps / (double)V) * nval(&smooth) +
                out->zloss;
    out->pred = arg;
    out->correct = (arg == t);
    out->w_t = wt;

    if (grad_row) {
        for (int64_t k = 0; k < V; ++k) {
            double dzdx;
            double zk = softcapped(logit(x, dtype, base + k), softcap, &dzdx);
            double pk = exp(zk - lse);
            double wk = class_weight(weight, k);
            double g = (1.0 - eps) * wt * (pk - (k == t ? 1.0 : 0.0)) +
                       (eps / (double)V) * (W * pk - wk) + 2.0 * lam * lse * pk;
            grad_row[k] = grad_scale * g * dzdx;
        }
    }
    return ORC_OK;
}

/* ---- denominators ------------------------------------------------------ */

/* D = sum of w[t_i] over non-ignored rows (the count when unweighted): the
 * mean reduction's total_weight. Also returns the non-ignored row count. */
static int denominators(int64_t rows, int64_t V, const int64_t* target,
                        const double* weight, int64_t ignore_index, double* D,
                        int64_t* n_valid) {
    nsum d = {0, 0};
    int64_t n = 0;
    for (int64_t i = 0; i < rows; ++i) {
        int64_t t = target[i];
        if (t == ignore_index) continue;
        if (t < 0 || t >= V) return ORC_TARGET_RANGE;
        nadd(&d, class_weight(weight, t));
        ++n;
    }
    *D = nval(&d);
    *n_valid = n;
    return ORC_OK;
}

static int check_args(const void* x, int dtype, int64_t rows, int64_t V,
                      const int64_t* target, double eps, double softcap,
                      int reduction) {
    if (rows < 0 || V <= 0) return ORC_BAD_ARG;
    if (rows > 0 && (!x || !target)) return ORC_BAD_ARG;
    if (dtype != ORC_F64 && dtype != ORC_F32 && dtype != ORC_BF16 && dtype != ORC_F16)
        return ORC_BAD_ARG;
    if (!(eps >= 0.0 && eps <= 1.0)) return ORC_BAD_ARG;
    if (isnan(softcap) || isinf(softcap)) return ORC_BAD_ARG;
    if (reduction != ORC_NONE && reduction != ORC_SUM && reduction != ORC_MEAN)
        return ORC_BAD_ARG;
    return ORC_OK;
}

/* ---- public entry points ---------------------------------------------- */

/*
 * Whole batch. x is [rows, V] row-major in the storage type dtype; target is
 * [rows] int64; weight is [V] or NULL; softcap <= 0 means off.
 * Outputs (each may be NULL):
 *   loss, z_loss, acc : [rows] for reduction "none", else [1]
 *   pred              : [rows], -1 on ignored rows
 *   grad              : [rows, V], the gradient of the reduced loss with
 *                       respect to x (the mean divides it by D)
 * Reductions: "sum" adds the rows; "mean" divides the sums by D (so an
 * all-ignored batch gives 0/0 = NaN); accuracy is n_correct / n_valid for
 * "sum" and "mean", and 0/1 per row for "none".
 */
int orc_ce_forward(const void* x, int dtype, int64_t rows, int64_t V,
                   const int64_t* target, const double* weight,
                   int64_t ignore_index, double label_smoothing,
                   double lse_square_scale, double softcap, int reduction,
                   double* loss, double* z_loss, double* acc, int64_t* pred,
                   double* grad) {
    int rc = check_args(x, dtype, rows, V, target, label_smoothing, softcap, reduction);
    if (rc) return rc;

    double D;
    int64_t n_valid;
    rc = denominators(rows, V, target, weight, ignore_index, &D, &n_valid);
    if (rc) return rc;
    /* With no valid row every gradient row is an ignored row (exact zeros),
     * so the scale is never applied; 1 avoids forming 1/0. */
    const double scale = (reduction == ORC_MEAN && D != 0.0) ? 1.0 / D : 1.0;

    nsum L = {0, 0}, Z = {0, 0};
    int64_t n_correct = 0;
    for (int64_t i = 0; i < rows; ++i) {
        row_out r;
        rc = one_row(x, dtype, i, V, target[i], weight, ignore_index,
                     label_smoothing, lse_square_scale, softcap, scale,
                     grad ? grad + i * V : NULL, &r);
        if (rc) return rc;
        if (pred) pred[i] = r.pred;
        if (reduction == ORC_NONE) {
            if (loss) loss[i] = r.loss;
            if (z_loss) z_loss[i] = r.zloss;
            if (acc) acc[i] = r.correct ? 1.0 : 0.0;
        }
        nadd(&L, r.loss);
        nadd(&Z, r.zloss);
        n_correct += r.correct;
    }
    if (reduction != ORC_NONE) {
        double l = nval(&L), z = nval(&Z);
        if (reduction == ORC_MEAN) { l /= D; z /= D; }
        if (loss) loss[0] = l;
        if (z_loss) z_loss[0] = z;
        if (acc) acc[0] = (double)n_correct / (double)n_valid;
    }
    return ORC_OK;
}

/*
 * Selected rows only, for spot checks of batches too large to run whole.
 * The gradient scale of the reduction (1/D for "mean") is still taken over
 * all rows of the batch. For each of the n_idx rows listed in row_idx it
 * writes the unreduced row loss, z-loss, predicted token, 0/1 correctness
 * and (if grad_rows is not NULL) the scaled gradient row into grad_rows
 * [n_idx, V]. D and n_valid receive the batch's denominators.
 */
int orc_ce_rows(const void* x, int dtype, int64_t rows, int64_t V,
                const int64_t* target, const double* weight, int64_t ignore_index,
                double label_smoothing, double lse_square_scale, double softcap,
                int reduction, const int64_t* row_idx, int64_t n_idx,
                double* loss_rows, double* zloss_rows, int64_t* pred_rows,
                double* correct_rows, double* grad_rows, double* D_out,
                int64_t* n_valid_out) {
    int rc = check_args(x, dtype, rows, V, target, label_smoothing, softcap, reduction);
    if (rc) return rc;
    double D;
    int64_t n_valid;
    rc = denominators(rows, V, target, weight, ignore_index, &D, &n_valid);
    if (rc) return rc;
    if (D_out) *D_out = D;
    if (n_valid_out) *n_valid_out = n_valid;
    const double scale = (reduction == ORC_MEAN && D != 0.0) ? 1.0 / D : 1.0;
    for (int64_t k = 0; k < n_idx; ++k) {
        int64_t i = row_idx[k];
        if (i < 0 || i >= rows) return ORC_BAD_ARG;
        row_out r;
        rc = one_row(x, dtype, i, V, target[i], weight, ignore_index,
                     label_smoothing, lse_square_scale, softcap, scale,
                     grad_rows ? grad_rows + k * V : NULL, &r);
        if (rc) return rc;
        if (loss_rows) loss_rows[k] = r.loss;
        if (zloss_rows) zloss_rows[k] = r.zloss;
        if (pred_rows) pred_rows[k] = r.pred;
        if (correct_rows) correct_rows[k] = r.correct ? 1.0 : 0.0;
    }
    return ORC_OK;
}

/* Backward (Backward Pass: the stored gradient times grad_output): either
 * one scalar for the whole matrix or one value per row. */
void orc_ce_backward(double* grad, int64_t rows, int64_t V,
                     const double* grad_output, int per_row) {
    for (int64_t i = 0; i < rows; ++i) {
        double g = per_row ? grad_output[i] : grad_output[0];
        for (int64_t j = 0; j < V; ++j) grad[i * V + j] *= g;
    }
}

/* Exposes the bf16 decoding so that a test can pin it to known bit
 * patterns. */
double orc_bf16_to_double(uint16_t bits) { return bf16_bits_to_double(bits); }

/* Exposes the fp16 decoding so that a test can pin it against every bit
 * pattern. */
double orc_f16_to_double(uint16_t bits) { return f16_bits_to_double(bits); }

/* Decodes n stored values (dtype as for the logits) into doubles, exactly. */
void orc_decode(const void* x, int dtype, int64_t n, double* out) {
    for (int64_t k = 0; k < n; ++k) out[k] = logit(x, dtype, k);
}
