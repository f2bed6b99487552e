/*
 * CPU oracle for per-token log-probabilities.  TEST INFRASTRUCTURE ONLY: this
 * file is built and called by the tests, by the package's smoke check and by
 * the CPU-baseline leg of the benchmark; the product path never links or runs
 * it.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (PreSTO, Appendix B.1 last paragraph and Appendix D.3):
 * for every scored row r with logits l_0..l_{V-1} and token tok,
 *     lp0 = log p0(tok)    = log softmax(l)[tok]        (temperature 1)
 *     lq  = log q_tau(tok) = log softmax(l / tau)[tok]  (temperature tau)
 * both from the same logits.  It is the plain definition written out in
 * float64: with m = max_j l_j and j* its first index,
 *     log softmax(l / t)[tok] = (l_tok - m) / t - log(1 + sum_{j != j*} exp((l_j - m) / t)).
 * The max term is kept out of the sum so that log1p stays accurate when one
 * token holds nearly all the mass.
 *
 * Logits rows are read as stored: bf16 (dtype 0, bit pattern in the high half
 * of a float32) or float32 (dtype 1).  A NaN logit, a token outside [0, V) or
 * a row whose logits are all -inf gives NaN for that row.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static double elem(const void *row, int dtype, int64_t j)
{
    float f;
    if (dtype == 0) {
        uint32_t bits = (uint32_t)((const uint16_t *)row)[j] << 16;
        memcpy(&f, &bits, sizeof f);
    } else {
        f = ((const float *)row)[j];
    }
    return (double)f;
}

/*
 * Full-vocabulary entropy of p0 = softmax(l) in nats (PreSTO Appendix D.3,
 * the quantity (iii) of the patched sampler): H = -sum_j p_j log p_j, written
 * with m = max_j l_j (first index j*), E = sum_{j != j*} exp(l_j - m) and
 * Z = 1 + E as
 *     H = log1p(E) - sum_{j != j*} exp(l_j - m) (l_j - m) / Z
 * (the max term has l_j - m = 0).  Keeping the max term out of the sums keeps
 * the result accurate when one token holds nearly all the mass.  A -inf
 * logit has probability 0 and contributes nothing.
 */
static double row_entropy(const void *row, int dtype, int64_t V, double m, int64_t jstar)
{
    double e_sum = 0.0, a = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        if (j == jstar)
            continue;
        double d = elem(row, dtype, j) - m;
        if (d == -INFINITY)
            continue;
        double e = exp(d);
        e_sum += e;
        a += e * d;
    }
    return log1p(e_sum) - a / (1.0 + e_sum);
}

static void one_row(const void *row, int dtype, int64_t V, int32_t tok, double tau,
                    double *lp0, double *lq, double *ent)
{
    if (tok < 0 || (int64_t)tok >= V) {
        *lp0 = NAN;
        *lq = NAN;
        if (ent)
            *ent = NAN;
        return;
    }
    double m = -INFINITY;
    int64_t jstar = -1;
    for (int64_t j = 0; j < V; ++j) {
        double l = elem(row, dtype, j);
        if (isnan(l)) {
            *lp0 = NAN;
            *lq = NAN;
            if (ent)
                *ent = NAN;
            return;
        }
        if (l > m) {
            m = l;
            jstar = j;
        }
    }
    if (jstar < 0) {            /* every logit is -inf */
        *lp0 = NAN;
        *lq = NAN;
        if (ent)
            *ent = NAN;
        return;
    }
    double e1 = 0.0, et = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        if (j == jstar)
            continue;
        double d = elem(row, dtype, j) - m;
        e1 += exp(d);
        et += exp(d / tau);
    }
    double dt = elem(row, dtype, tok) - m;
    *lp0 = dt - log1p(e1);
    *lq = dt / tau - log1p(et);
    if (ent)
        *ent = row_entropy(row, dtype, V, m, jstar);
}

/*
 * Score n_rows rows.  Row r reads logits row row_index[r] (or r when row_index
 * is NULL), at byte offset row * ld * element size from `logits`.  `entropy`
 * may be NULL; otherwise it receives H of p0 for every row.
 */
void oracle_row_logprobs(const void *logits, int dtype, int64_t V, int64_t ld,
                         int64_t n_rows, const int64_t *row_index,
                         const int32_t *tokens, double tau, double *lp0, double *lq,
                         double *entropy, int n_threads)
{
    const size_t esz = dtype == 0 ? 2 : 4;
#pragma omp parallel for schedule(dynamic, 16) num_threads(n_threads > 0 ? n_threads : 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t src = row_index ? row_index[r] : r;
        const char *row = (const char *)logits + (size_t)src * (size_t)ld * esz;
        one_row(row, dtype, V, tokens[r], tau, &lp0[r], &lq[r], entropy ? &entropy[r] : 0);
    }
}

/* Number of OpenMP threads the oracle would use by default (for reporting). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
