/*
 * oracle.c -- plain float64 CPU reference for the fused row reductions.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * kernels: it restates each operation from its definition, one row at a time,
 * in float64, with no blocking, fusion or reordering.
 *
 * Sources of each definition (page titles as published):
 *   [P1] "Engineering a CUDA Machine Learning Framework from Scratch"
 *        sec. 3.1 "Online FlashSoftmax": softmax is defined by three passes
 *        (row max, normaliser sum of exp(x - max), normalise); the online
 *        method reaches the same value in one pass.
 *        sec. 3.2 "Welford Single-Pass Normalization": LayerNorm moments.
 *        sec. 2.1: loss gradients fused with the normalisation.
 *        sec. 2.2: the analytic (pre-derived) backward.
 *   [P2] "gpu-ml-learning" README, Module 3: softmax and cross-entropy loss.
 *   [P3] "NexusGrad" README: the Softmax activation layer of the layer stack
 *        (its backward is the softmax vector-Jacobian product) and RMSNorm
 *        among the transformer components (no formula given).
 * The two recurrences the pages name but whose equations did not survive are
 * restated from their published sources:
 *   Milakov & Gimelshein (2018), "Online normalizer calculation for softmax";
 *   Welford (1962) update, and the pairwise merge of Chan, Golub & LeVeque
 *   (1979).  They are here only so tests can check that they reach the
 *   three-pass / two-pass definitions (oracle_online_*, oracle_welford*).
 *
 * Readings taken where the pages are silent:
 *   - variance is the biased (population) one, rstd = 1/sqrt(var + eps);
 *   - a softmax / cross-entropy row whose maximum is -inf (fully masked) gives
 *     zeros: y = 0, loss = 0, dlogits = 0;
 *   - a cross-entropy row whose label equals ignore_index gives loss 0 and an
 *     all-zero dlogits row;
 *   - a label outside [0, cols) that is not ignore_index gives loss NaN and
 *     dlogits equal to the plain softmax; it is counted in the return value;
 *   - a LayerNorm row whose mean is not finite is masked: y = 0, mean = 0,
 *     rstd = 0; in the backward a row with rstd == 0 is masked: dx = 0 and it
 *     adds nothing to dgamma / dbeta;
 *   - loss is per row (no reduction), dlogits is unscaled;
 *   - log-softmax of a fully masked row is 0 (as the softmax gives zeros);
 *   - RMSNorm is y = x / sqrt(mean(x^2) + eps) * gamma (no bias, no mean
 *     subtraction); a row whose mean square is not finite is masked like a
 *     LayerNorm row (y = 0, rstd = 0; rstd == 0 masks it in the backward).
 *
 * Storage types: dtype 0 = IEEE float32, dtype 1 = bfloat16 (the upper 16 bits
 * of a float32).  Inputs are widened exactly to double.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* Exact widening of one stored element to double (bf16 is the top half of an
 * IEEE float32 bit pattern). */
static double load_elem(const void *base, int dtype, int64_t i)
{
    if (dtype == ORACLE_F32) {
        float f;
        memcpy(&f, (const char *)base + 4 * i, 4);
        return (double)f;
    } else {
        uint16_t h;
        uint32_t u;
        float f;
        memcpy(&h, (const char *)base + 2 * i, 2);
        u = ((uint32_t)h) << 16;
        memcpy(&f, &u, 4);
        return (double)f;
    }
}

/* ---------------------------------------------------------------------- */
/* Softmax, three-pass definition [P1 sec. 3.1].                          */
/* y_j = exp(x_j - m) / d with m = max_j x_j and d = sum_j exp(x_j - m).  */
/* ---------------------------------------------------------------------- */
void oracle_softmax(const void *x, int dtype, int64_t rows, int64_t cols,
                    double *y)
{
    for (int64_t r = 0; r < rows; ++r) {
        int64_t off = r * cols;
        /* pass 1: row maximum */
        double m = -INFINITY;
        for (int64_t j = 0; j < cols; ++j) {
            double v = load_elem(x, dtype, off + j);
            if (v > m) m = v;
        }
        if (m == -INFINITY) { /* fully masked row: zeros (reading) */
            for (int64_t j = 0; j < cols; ++j) y[off + j] = 0.0;
            continue;
        }
        /* pass 2: normaliser */
        double d = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            d += exp(load_elem(x, dtype, off + j) - m);
        /* pass 3: normalise */
        for (int64_t j = 0; j < cols; ++j)
            y[off + j] = exp(load_elem(x, dtype, off + j) - m) / d;
    }
}

/* ---------------------------------------------------------------------- */
/* Softmax cross-entropy, forward and backward [P1 sec. 2.1, P2 Module 3].*/
/* loss = -log softmax(x)[label] = m + log d - x[label];                  */
/* dlogits_j = softmax(x)_j - [j == label].                               */
/* Returns the number of rows whose label is out of range (and not        */
/* ignore_index).  loss/dlogits may be NULL to skip writing them.         */
/* ---------------------------------------------------------------------- */
int64_t oracle_xent(const void *logits, const int32_t *labels, int dtype,
                    int64_t rows, int64_t cols, int32_t ignore_index,
                    double *loss, double *dlogits)
{
    int64_t bad = 0;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t off = r * cols;
        int32_t label = labels[r];
        if (label == ignore_index) {
            if (loss) loss[r] = 0.0;
            if (dlogits)
                for (int64_t j = 0; j < cols; ++j) dlogits[off + j] = 0.0;
            continue;
        }
        int valid = (label >= 0 && (int64_t)label < cols);
        if (!valid) bad += 1;
        double m = -INFINITY;
        for (int64_t j = 0; j < cols; ++j) {
            double v = load_elem(logits, dtype, off + j);
            if (v > m) m = v;
        }
        if (m == -INFINITY) { /* fully masked row: zeros (reading) */
            if (loss) loss[r] = 0.0;
            if (dlogits)
                for (int64_t j = 0; j < cols; ++j) dlogits[off + j] = 0.0;
            continue;
        }
        double d = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            d += exp(load_elem(logits, dtype, off + j) - m);
        if (loss) {
            if (valid)
                loss[r] = m + log(d) - load_elem(logits, dtype, off + label);
            else
                loss[r] = NAN;
        }
        if (dlogits) {
            for (int64_t j = 0; j < cols; ++j) {
                double p = exp(load_elem(logits, dtype, off + j) - m) / d;
                dlogits[off + j] = (valid && j == label) ? p - 1.0 : p;
            }
        }
    }
    return bad;
}

/* ---------------------------------------------------------------------- */
/* LayerNorm forward, two-pass moments [P1 sec. 3.2].                     */
/* mean = (1/C) sum x; var = (1/C) sum (x - mean)^2 (biased);             */
/* rstd = 1/sqrt(var + eps); y = (x - mean) * rstd * gamma + beta.        */
/* ---------------------------------------------------------------------- */
void oracle_ln_fwd(const void *x, const void *gamma, const void *beta,
                   int dtype, int64_t rows, int64_t cols, double eps,
                   double *y, double *mean, double *rstd)
{
    for (int64_t r = 0; r < rows; ++r) {
        int64_t off = r * cols;
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j) s += load_elem(x, dtype, off + j);
        double mu = s / (double)cols;
        if (!isfinite(mu)) { /* masked row (reading) */
            mean[r] = 0.0;
            rstd[r] = 0.0;
            if (y)
                for (int64_t j = 0; j < cols; ++j) y[off + j] = 0.0;
            continue;
        }
        double ss = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double c = load_elem(x, dtype, off + j) - mu;
            ss += c * c;
        }
        double var = ss / (double)cols;
        double rs = 1.0 / sqrt(var + eps);
        mean[r] = mu;
        rstd[r] = rs;
        if (y)
            for (int64_t j = 0; j < cols; ++j)
                y[off + j] = (load_elem(x, dtype, off + j) - mu) * rs *
                                 load_elem(gamma, dtype, j) +
                             load_elem(beta, dtype, j);
    }
}

/* ---------------------------------------------------------------------- */
/* LayerNorm backward, analytic derivative of y = xhat*gamma + beta with  */
/* xhat = (x - mean) * rstd [P1 sec. 2.2]:                                */
/*   g = dy * gamma;                                                      */
/*   dx = rstd * (g - mean_j(g) - xhat * mean_j(g * xhat));               */
/*   dgamma_j = sum_r dy * xhat;  dbeta_j = sum_r dy.                     */
/* mean/rstd are the forward's saved statistics (double).  dgamma_abs and */
/* dbeta_abs (nullable) receive sum_r |dy * xhat| and sum_r |dy|, used to */
/* scale the tolerance of the column sums.  dgamma/dbeta are overwritten. */
/* ---------------------------------------------------------------------- */
void oracle_ln_bwd(const void *dy, const void *x, const double *mean,
                   const double *rstd, const void *gamma, int dtype,
                   int64_t rows, int64_t cols, double *dx, double *dgamma,
                   double *dbeta, double *dgamma_abs, double *dbeta_abs)
{
    for (int64_t j = 0; j < cols; ++j) {
        dgamma[j] = 0.0;
        dbeta[j] = 0.0;
        if (dgamma_abs) dgamma_abs[j] = 0.0;
        if (dbeta_abs) dbeta_abs[j] = 0.0;
    }
    for (int64_t r = 0; r < rows; ++r) {
        int64_t off = r * cols;
        double mu = mean[r], rs = rstd[r];
        if (rs == 0.0) { /* masked row (reading) */
            if (dx)
                for (int64_t j = 0; j < cols; ++j) dx[off + j] = 0.0;
            continue;
        }
        double sg = 0.0, sgx = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double xh = (load_elem(x, dtype, off + j) - mu) * rs;
            double g = load_elem(dy, dtype, off + j) * load_elem(gamma, dtype, j);
            sg += g;
            sgx += g * xh;
        }
        double mg = sg / (double)cols, mgx = sgx / (double)cols;
        for (int64_t j = 0; j < cols; ++j) {
            double xh = (load_elem(x, dtype, off + j) - mu) * rs;
            double d = load_elem(dy, dtype, off + j);
            double g = d * load_elem(gamma, dtype, j);
            if (dx) dx[off + j] = rs * (g - mg - xh * mgx);
            dgamma[j] += d * xh;
            dbeta[j] += d;
            if (dgamma_abs) dgamma_abs[j] += fabs(d * xh);
            if (dbeta_abs) dbeta_abs[j] += fabs(d);
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Softmax backward (vector-Jacobian product of y = softmax(x), the       */
/* derivative behind the Softmax activation layer of [P3] "NexusGrad",    */
/* "Current main layer stack"): dx_j = y_j * (dy_j - sum_k y_k dy_k).      */
/* y is the forward output as stored; a fully masked row (y = 0) gets 0.  */
/* ---------------------------------------------------------------------- */
void oracle_softmax_bwd(const void *y, const void *dy, int dtype, int64_t rows,
                        int64_t cols, double *dx)
{
    for (int64_t r = 0; r < rows; ++r) {
        int64_t off = r * cols;
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            s += load_elem(y, dtype, off + j) * load_elem(dy, dtype, off + j);
        for (int64_t j = 0; j < cols; ++j)
            dx[off + j] = load_elem(y, dtype, off + j) * (load_elem(dy, dtype, off + j) - s);
    }
}

/* ---------------------------------------------------------------------- */
/* Log-softmax forward from the same three passes as the softmax [P1 sec. */
/* 3.1]: m = max_j x_j, d = sum_j exp(x_j - m), z_j = x_j - m - ln d.      */
/* Reading: a fully masked row (m = -inf) gives z = 0, like the zeros the */
/* softmax gives there (never NaN).                                       */
/* ---------------------------------------------------------------------- */
void oracle_log_softmax(const void *x, int dtype, int64_t rows, int64_t cols,
                        double *z)
{
    for (int64_t r = 0; r < rows; ++r) {
        int64_t off = r * cols;
        double m = -INFINITY;
        for (int64_t j = 0; j < cols; ++j) {
            double v = load_elem(x, dtype, off + j);
            if (v > m) m = v;
        }
        if (m == -INFINITY) {
            for (int64_t j = 0; j < cols; ++j) z[off + j] = 0.0;
            continue;
        }
        double d = 0.0;
        for (int64_t j = 0; j < cols; ++j) d += exp(load_elem(x, dtype, off + j) - m);
        double lse = m + log(d);
        for (int64_t j = 0; j < cols; ++j) z[off + j] = load_elem(x, dtype, off + j) - lse;
    }
}

/* ---------------------------------------------------------------------- */
/* Log-softmax backward (VJP of z = log_softmax(x)):                      */
/*   dx_j = dz_j - exp(z_j) * sum_k dz_k,  exp(z) being the softmax.      */
/* The forward output z is taken as stored and the formula is applied to */
/* every row (a fully masked row, z = 0 from the forward, has no          */
/* derivative of its own; it gets dx = dz - sum dz like any row of equal  */
/* logits).                                                               */
/* ---------------------------------------------------------------------- */
void oracle_log_softmax_bwd(const void *z, const void *dz, int dtype, int64_t rows,
                            int64_t cols, double *dx)
{
    for (int64_t r = 0; r < rows; ++r) {
        int64_t off = r * cols;
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j) s += load_elem(dz, dtype, off + j);
        for (int64_t j = 0; j < cols; ++j)
            dx[off + j] = load_elem(dz, dtype, off + j) - exp(load_elem(z, dtype, off + j)) * s;
    }
}

/* ---------------------------------------------------------------------- */
/* RMSNorm forward ([P3] "NexusGrad", "Core Capabilities" lists RMSNorm   */
/* without a formula; reading: the standard definition of Zhang &         */
/* Sennrich (2019)): ms = (1/C) sum_j x_j^2, rstd = 1/sqrt(ms + eps),      */
/* y_j = x_j * rstd * gamma_j.  A row whose ms is not finite is masked:   */
/* y = 0, rstd = 0 (the LayerNorm convention).                            */
/* ---------------------------------------------------------------------- */
void oracle_rms_fwd(const void *x, const void *gamma, int dtype, int64_t rows,
                    int64_t cols, double eps, double *y, double *rstd)
{
    for (int64_t r = 0; r < rows; ++r) {
        int64_t off = r * cols;
        double ss = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double v = load_elem(x, dtype, off + j);
            ss += v * v;
        }
        double ms = ss / (double)cols;
        if (!isfinite(ms)) {
            rstd[r] = 0.0;
            if (y)
                for (int64_t j = 0; j < cols; ++j) y[off + j] = 0.0;
            continue;
        }
        double rs = 1.0 / sqrt(ms + eps);
        rstd[r] = rs;
        if (y)
            for (int64_t j = 0; j < cols; ++j)
                y[off + j] = load_elem(x, dtype, off + j) * rs * load_elem(gamma, dtype, j);
    }
}

/* ---------------------------------------------------------------------- */
/* RMSNorm backward, the analytic derivative of the forward above: with   */
/* xhat = x * rstd and g = dy * gamma,                                    */
/*   dx = rstd * (g - xhat * mean_j(g * xhat)),  dgamma_j = sum_r dy*xhat. */
/* rstd == 0 marks a masked row (dx = 0, nothing added to dgamma).        */
/* dgamma_abs (nullable) receives sum_r |dy * xhat|.                      */
/* ---------------------------------------------------------------------- */
void oracle_rms_bwd(const void *dy, const void *x, const double *rstd,
                    const void *gamma, int dtype, int64_t rows, int64_t cols,
                    double *dx, double *dgamma, double *dgamma_abs)
{
    for (int64_t j = 0; j < cols; ++j) {
        dgamma[j] = 0.0;
        if (dgamma_abs) dgamma_abs[j] = 0.0;
    }
    for (int64_t r = 0; r < rows; ++r) {
        int64_t off = r * cols;
        double rs = rstd[r];
        if (rs == 0.0) {
            if (dx)
                for (int64_t j = 0; j < cols; ++j) dx[off + j] = 0.0;
            continue;
        }
        double sgx = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double xh = load_elem(x, dtype, off + j) * rs;
            sgx += load_elem(dy, dtype, off + j) * load_elem(gamma, dtype, j) * xh;
        }
        double mgx = sgx / (double)cols;
        for (int64_t j = 0; j < cols; ++j) {
            double xh = load_elem(x, dtype, off + j) * rs;
            double d = load_elem(dy, dtype, off + j);
            double g = d * load_elem(gamma, dtype, j);
            if (dx) dx[off + j] = rs * (g - xh * mgx);
            dgamma[j] += d * xh;
            if (dgamma_abs) dgamma_abs[j] += fabs(d * xh);
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Self-check helpers: the recurrences the GPU path uses, in float64, so  */
/* tests can show they reach the definitions above.                       */
/* ---------------------------------------------------------------------- */

/* Online normaliser (Milakov & Gimelshein 2018): one pass keeps the
 * running maximum m and the sum d of exp(x - m) rescaled whenever m grows:
 *   m' = max(m, x);  d' = d * exp(m - m') + exp(x - m').
 * A state with m = -inf has d = 0 and contributes nothing. */
void oracle_online_softmax_stats(const double *x, int64_t n, double *m_out,
                                 double *d_out)
{
    double m = -INFINITY, d = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double mn = x[i] > m ? x[i] : m;
        if (mn == -INFINITY) continue; /* nothing seen yet but -inf */
        double scale = (m == -INFINITY) ? 0.0 : exp(m - mn);
        d = d * scale + exp(x[i] - mn);
        m = mn;
    }
    *m_out = m;
    *d_out = d;
}

/* Merge of two online states (same paper):
 *   m = max(ma, mb);  d = da * exp(ma - m) + db * exp(mb - m). */
void oracle_online_merge(double ma, double da, double mb, double db,
                         double *m_out, double *d_out)
{
    double m = ma > mb ? ma : mb;
    if (m == -INFINITY) {
        *m_out = m;
        *d_out = 0.0;
        return;
    }
    double d = 0.0;
    if (ma != -INFINITY) d += da * exp(ma - m);
    if (mb != -INFINITY) d += db * exp(mb - m);
    *m_out = m;
    *d_out = d;
}

/* Welford (1962): n += 1; delta = x - mean; mean += delta / n;
 * M2 += delta * (x - mean).  var = M2 / n (biased). */
void oracle_welford(const double *x, int64_t n, double *mean_out,
                    double *m2_out)
{
    double mean = 0.0, m2 = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double delta = x[i] - mean;
        mean += delta / (double)(i + 1);
        m2 += delta * (x[i] - mean);
    }
    *mean_out = mean;
    *m2_out = m2;
}

/* Chan, Golub & LeVeque (1979) pairwise merge of (n, mean, M2):
 * n = na + nb; delta = mean_b - mean_a; mean = mean_a + delta * nb / n;
 * M2 = M2a + M2b + delta^2 * na * nb / n. */
void oracle_chan_merge(double na, double mean_a, double m2a, double nb,
                       double mean_b, double m2b, double *n_out,
                       double *mean_out, double *m2_out)
{
    double n = na + nb;
    if (n == 0.0) {
        *n_out = 0.0;
        *mean_out = 0.0;
        *m2_out = 0.0;
        return;
    }
    double delta = mean_b - mean_a;
    *n_out = n;
    *mean_out = mean_a + delta * nb / n;
    *m2_out = m2a + m2b + delta * delta * na * nb / n;
}

/* ---------------------------------------------------------------------- */
/* Scaled dot-product attention, forward [P1 sec. 6.4 and P3: the          */
/* FlashAttention-style extension of the online softmax; the attention     */
/* itself as defined by Vaswani et al. (2017)].  For each head b and query */
/* row i: s_j = scale * sum_c q_ic k_jc over the keys j it may see (j <= i */
/* when causal, all j otherwise), o_i = sum_j softmax(s)_j v_j and         */
/* lse_i = m + log sum_j exp(s_j - m), m = max_j s_j.  The plain           */
/* three-pass definition per row (scores, maximum and normaliser, output); */
/* no tiling.  q, k, v: [bh][s][d] stored dtype; o: [bh][s][d] and         */
/* lse: [bh][s] float64; scores: caller's scratch of s doubles.            */
/* ---------------------------------------------------------------------- */
void oracle_attention(const void *q, const void *k, const void *v, int dtype,
                      int64_t bh, int64_t s, int64_t d, double scale, int causal,
                      double *o, double *lse, double *scores)
{
    for (int64_t b = 0; b < bh; ++b) {
        const int64_t base = b * s * d;
        for (int64_t i = 0; i < s; ++i) {
            const int64_t nk = causal ? i + 1 : s;
            /* pass 1: scores and their maximum */
            double m = -INFINITY;
            for (int64_t j = 0; j < nk; ++j) {
                double acc = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    acc += load_elem(q, dtype, base + i * d + c) *
                           load_elem(k, dtype, base + j * d + c);
                scores[j] = scale * acc;
                if (scores[j] > m) m = scores[j];
            }
            /* pass 2: normaliser */
            double l = 0.0;
            for (int64_t j = 0; j < nk; ++j) l += exp(scores[j] - m);
            /* pass 3: output row */
            for (int64_t c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int64_t j = 0; j < nk; ++j)
                    acc += exp(scores[j] - m) * load_elem(v, dtype, base + j * d + c);
                o[base + i * d + c] = acc / l;
            }
            lse[b * s + i] = m + log(l);
        }
    }
}
