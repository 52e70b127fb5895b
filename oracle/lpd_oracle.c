/*
 * Float64 CPU oracle for selected-token logprob drift scoring.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * restatement of what the scorer computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA library: every definition below is
 * written out again from the method's text.
 *
 * Sources (page title, section):
 *   [MC]  "WS2 Cross-Config Logprob Drift Contract", section "Measurement
 *         Contract": dlogp = train_recomputed_logp - rollout_old_logp, taken
 *         only on active response/action tokens; teacher forcing on the
 *         already-sampled sequence (no resampling).
 *   [DG]  same page, section "Diagnostics": ratio0 = exp(dlogp); clipfrac0 =
 *         mean indicator that ratio0 is outside the clip range; approx_kl0 =
 *         masked mean of exp(dlogp) - 1 - dlogp; mean/p95/p99/max of
 *         abs(dlogp), all over active tokens only.
 *   [B1]  same page, section "Revised Modular PR Roadmap", item B1: the zero
 *         active-token case and worst-token metadata are part of the contract.
 *   [LP]  "[WS2] Framework for ablation experiment", LogProb knobs table,
 *         rows 3-5 and 8: per-shard (vocab_start, vocab_end) ownership, the
 *         per-shard partial logsumexp merged in global vocab-shard order, and
 *         the single-owner selected-logit gather on pre-shifted rows.
 *   [HD]  same table, rows 9-10: the LM-head GEMM that produces the logits.
 *   [TC]  same table, row 7: an ordered chain of logit transforms (temperature,
 *         soft-cap, logit scale) applied to every logit before the softmax.
 *   [TS]  same table, row 11: training-only state, i.e. the entropy of the
 *         softmax and the logprob's gradient with respect to the logits.
 *   [AM]  "Attention Debug Matrix", row A7 (merge_order), and the Attention
 *         knobs table of "[WS2] Framework for ablation experiment", rows 6-7:
 *         split-KV / context-parallel partial results (out_k, lse_k) merged
 *         into one (out, lse) in a given block order; lse in base e or 2.
 *
 * Readings where the pages are silent (each is also listed with the design
 * notes): percentiles are nearest-rank (1-based rank ceil(p*A/100) of the
 * ascending |dlogp|); the ratio0 aggregate is the masked mean; the clip range
 * is given as absolute bounds [lo, hi] and a ratio equal to a bound is inside;
 * with zero active tokens every metric is 0 and the NO_ACTIVE flag is set;
 * the worst token is the lowest row index among ties of max |dlogp|.
 *
 * Arithmetic: every logit is widened to double (exact for bf16 and fp32);
 * sums run serially in column order; exp/log/expm1 are the C library's.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { LPDO_BF16 = 0, LPDO_F32 = 1 };

/* status bits (per call, OR-ed over active rows) */
#define LPDO_STATUS_TOKEN_OOB 1u
#define LPDO_STATUS_NONFINITE 2u
/* result flags */
#define LPDO_FLAG_NO_ACTIVE 1u

typedef struct {
    int64_t n_active;
    int64_t argmax_row;
    uint32_t flags;
    uint32_t status;
    double ratio0_mean;
    double clipfrac0;
    double approx_kl0;
    double mean_abs_dlogp;
    double p95_abs_dlogp;
    double p99_abs_dlogp;
    double max_abs_dlogp;
} lpdo_metrics;

/* One stored logit, widened to double.  A bf16 value is the upper half of the
 * fp32 with the same bits, so the widening is exact. */
static double logit_at(const void *row, int dtype, int64_t j)
{
    if (dtype == LPDO_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)row)[j] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)row)[j];
}

static const void *row_ptr(const void *base, int dtype, int64_t stride, int64_t r)
{
    size_t elt = dtype == LPDO_BF16 ? 2 : 4;
    return (const char *)base + (size_t)r * (size_t)stride * elt;
}

/* Partial log-sum-exp of columns [c0, c1) of one row, as the pair
 * (m, s) with m = max_j x_j and s = sum_j exp(x_j - m), serial in j.
 * An empty or all -inf range gives (-inf, 0). */
void lpdo_partial(const void *row, int dtype, int64_t c0, int64_t c1,
                  double *m_out, double *s_out)
{
    double m = -INFINITY;
    int has_nan = 0;
    for (int64_t j = c0; j < c1; ++j) {
        double x = logit_at(row, dtype, j);
        if (x > m)
            m = x;
        if (isnan(x))
            has_nan = 1;
    }
    double s = 0.0;
    if (m != -INFINITY) {
        for (int64_t j = c0; j < c1; ++j)
            s += exp(logit_at(row, dtype, j) - m);
    }
    /* a NaN anywhere in the range makes the sum NaN, which the caller flags */
    if (has_nan)
        s = NAN;
    *m_out = m;
    *s_out = s;
}

/* log(sum_j exp(x_j)) from a partial pair. */
static double lse_of(double m, double s)
{
    if (m == -INFINITY && s == 0.0)
        return -INFINITY;
    return m + log(s);
}

/* Selected-token log-probability of one row [MC]:
 *   logp = x[id] - log(sum_j exp(x_j)).
 * Returns the status bits this row raises. */
uint32_t lpdo_row_logp(const void *row, int dtype, int64_t vocab, int64_t id,
                       double *logp_out)
{
    if (id < 0 || id >= vocab) {
        *logp_out = NAN;
        return LPDO_STATUS_TOKEN_OOB;
    }
    double m, s;
    lpdo_partial(row, dtype, 0, vocab, &m, &s);
    double lse = lse_of(m, s);
    double xs = logit_at(row, dtype, id);
    *logp_out = xs - lse;
    return (isfinite(lse) && isfinite(xs)) ? 0u : LPDO_STATUS_NONFINITE;
}

static int cmp_double(const void *a, const void *b)
{
    double x = *(const double *)a, y = *(const double *)b;
    return (x > y) - (x < y);
}

/* Drift diagnostics over active rows [DG], [B1].  d[r] is read only where
 * mask[r] != 0. */
void lpdo_metrics_from_dlogp(const double *d, const uint8_t *mask, int64_t n_rows,
                             double clip_lo, double clip_hi, lpdo_metrics *out)
{
    memset(out, 0, sizeof *out);
    out->argmax_row = -1;
    int64_t a = 0;
    for (int64_t r = 0; r < n_rows; ++r)
        a += mask[r] != 0;
    out->n_active = a;
    if (a == 0) {
        out->flags |= LPDO_FLAG_NO_ACTIVE;
        return;
    }
    double *absd = (double *)malloc((size_t)a * sizeof(double));
    double sum_ratio = 0.0, sum_k3 = 0.0, sum_abs = 0.0;
    int64_t n_clip = 0, k = 0;
    double best = -1.0;
    for (int64_t r = 0; r < n_rows; ++r) {
        if (!mask[r])
            continue;
        double x = d[r];
        double ratio = exp(x);                 /* ratio0 */
        sum_ratio += ratio;
        sum_k3 += expm1(x) - x;                /* exp(d) - 1 - d */
        sum_abs += fabs(x);
        if (ratio < clip_lo || ratio > clip_hi)
            ++n_clip;
        if (fabs(x) > best) {                  /* strict: lowest row wins ties */
            best = fabs(x);
            out->argmax_row = r;
        }
        absd[k++] = fabs(x);
    }
    qsort(absd, (size_t)a, sizeof(double), cmp_double);
    /* nearest rank: 1-based rank ceil(p * A / 100), integer arithmetic */
    int64_t k95 = (95 * a + 99) / 100, k99 = (99 * a + 99) / 100;
    out->ratio0_mean = sum_ratio / (double)a;
    out->clipfrac0 = (double)n_clip / (double)a;
    out->approx_kl0 = sum_k3 / (double)a;
    out->mean_abs_dlogp = sum_abs / (double)a;
    out->p95_abs_dlogp = absd[k95 - 1];
    out->p99_abs_dlogp = absd[k99 - 1];
    out->max_abs_dlogp = absd[a - 1];
    free(absd);
}

/* Teacher-forced scoring of both sides over all rows [MC].
 * Row r of each logits tensor scores token_ids[r] (pre-shifted rows [LP]);
 * only rows with mask[r] != 0 are read.  Per-row outputs are written for every
 * row (0 where inactive).  Returns the status bits. */
uint32_t lpdo_score(const void *train, int train_dtype, int64_t train_stride,
                    const void *rollout, int rollout_dtype, int64_t rollout_stride,
                    int64_t n_rows, int64_t vocab, const int32_t *token_ids,
                    const uint8_t *mask, double clip_lo, double clip_hi,
                    double *logp_train, double *logp_rollout, double *dlogp,
                    lpdo_metrics *metrics)
{
    uint32_t status = 0;
    for (int64_t r = 0; r < n_rows; ++r) {
        logp_train[r] = logp_rollout[r] = dlogp[r] = 0.0;
        if (!mask[r])
            continue;
        status |= lpdo_row_logp(row_ptr(train, train_dtype, train_stride, r),
                                train_dtype, vocab, token_ids[r], &logp_train[r]);
        status |= lpdo_row_logp(row_ptr(rollout, rollout_dtype, rollout_stride, r),
                                rollout_dtype, vocab, token_ids[r], &logp_rollout[r]);
        dlogp[r] = logp_train[r] - logp_rollout[r];
    }
    if (metrics) {
        lpdo_metrics_from_dlogp(dlogp, mask, n_rows, clip_lo, clip_hi, metrics);
        metrics->status = status;
    }
    return status;
}

/* Score a selected list of rows only (for sampled checks on inputs too large
 * to score whole).  rows[i] names the row; outputs are indexed by i. */
uint32_t lpdo_score_rows(const void *train, int train_dtype, int64_t train_stride,
                         const void *rollout, int rollout_dtype, int64_t rollout_stride,
                         int64_t vocab, const int32_t *token_ids, const int64_t *rows,
                         int64_t n_sel, double *logp_train, double *logp_rollout,
                         double *dlogp)
{
    uint32_t status = 0;
    for (int64_t i = 0; i < n_sel; ++i) {
        int64_t r = rows[i];
        status |= lpdo_row_logp(row_ptr(train, train_dtype, train_stride, r),
                                train_dtype, vocab, token_ids[r], &logp_train[i]);
        status |= lpdo_row_logp(row_ptr(rollout, rollout_dtype, rollout_stride, r),
                                rollout_dtype, vocab, token_ids[r], &logp_rollout[i]);
        dlogp[i] = logp_train[i] - logp_rollout[i];
    }
    return status;
}

/* ---- vocab-sharded form [LP] ------------------------------------------- */

typedef struct {
    const void *ptr;      /* [n_rows, stride] logits of this shard's columns */
    int32_t dtype;
    int32_t pad_;
    int64_t stride;       /* elements between rows */
    int64_t v_start;      /* global vocab range [v_start, v_end) */
    int64_t v_end;
} lpdo_shard;

/* One side, one row, vocab split over shards.  Each shard yields its own
 * partial (m_k, s_k) over its columns; the partials are merged one at a time
 * in the order given by `order` (a permutation of shard indices):
 *   m = max(m, m_k);  s = s * exp(m_old - m) + s_k * exp(m_k - m).
 * The selected logit comes from the single shard whose range holds id. */
static uint32_t sharded_row_logp(const lpdo_shard *sh, int n_shards, const int32_t *order,
                                 int64_t r, int64_t vocab, int64_t id, double *logp_out)
{
    if (id < 0 || id >= vocab) {
        *logp_out = NAN;
        return LPDO_STATUS_TOKEN_OOB;
    }
    double m = -INFINITY, s = 0.0, xs = NAN;
    int owners = 0;
    for (int i = 0; i < n_shards; ++i) {
        const lpdo_shard *k = &sh[order[i]];
        const void *row = row_ptr(k->ptr, k->dtype, k->stride, r);
        double mk, sk;
        lpdo_partial(row, k->dtype, 0, k->v_end - k->v_start, &mk, &sk);
        double mn = mk > m ? mk : m;
        if (mn != -INFINITY)
            s = (m == -INFINITY ? 0.0 : s * exp(m - mn)) +
                (mk == -INFINITY ? 0.0 : sk * exp(mk - mn));
        if (isnan(sk))
            s = NAN;
        m = mn;
        if (id >= k->v_start && id < k->v_end) {
            xs = logit_at(row, k->dtype, id - k->v_start);
            ++owners;
        }
    }
    double lse = lse_of(m, s);
    *logp_out = xs - lse;
    if (owners != 1)
        return LPDO_STATUS_TOKEN_OOB;
    return (isfinite(lse) && isfinite(xs)) ? 0u : LPDO_STATUS_NONFINITE;
}

/* Exact-tiling check of a shard map [LP] ("fail closed on missing vocab-shard
 * bounds"): the ranges must cover [0, vocab) with no gap and no overlap.
 * Returns 0 if valid. */
int lpdo_check_tiling(const lpdo_shard *sh, int n_shards, int64_t vocab)
{
    if (n_shards <= 0)
        return -1;
    int64_t covered = 0;
    for (int i = 0; i < n_shards; ++i) {
        if (sh[i].v_start < 0 || sh[i].v_end <= sh[i].v_start || sh[i].v_end > vocab)
            return -1;
        covered += sh[i].v_end - sh[i].v_start;
        for (int j = 0; j < i; ++j)
            if (sh[i].v_start < sh[j].v_end && sh[j].v_start < sh[i].v_end)
                return -1;
    }
    return covered == vocab ? 0 : -1;
}

uint32_t lpdo_score_sharded(const lpdo_shard *train, const lpdo_shard *rollout, int n_shards,
                            const int32_t *order, int64_t n_rows, int64_t vocab,
                            const int32_t *token_ids, const uint8_t *mask,
                            double clip_lo, double clip_hi,
                            double *logp_train, double *logp_rollout, double *dlogp,
                            lpdo_metrics *metrics)
{
    uint32_t status = 0;
    for (int64_t r = 0; r < n_rows; ++r) {
        logp_train[r] = logp_rollout[r] = dlogp[r] = 0.0;
        if (!mask[r])
            continue;
        status |= sharded_row_logp(train, n_shards, order, r, vocab, token_ids[r], &logp_train[r]);
        status |= sharded_row_logp(rollout, n_shards, order, r, vocab, token_ids[r], &logp_rollout[r]);
        dlogp[r] = logp_train[r] - logp_rollout[r];
    }
    if (metrics) {
        lpdo_metrics_from_dlogp(dlogp, mask, n_rows, clip_lo, clip_hi, metrics);
        metrics->status = status;
    }
    return status;
}

/* ---- LM-head form [HD] -------------------------------------------------- */

/* Logits of one token from its hidden state: x_v = sum_k h_k * W[v, k],
 * serial in k, in double.  h is [hidden] bf16, W is [vocab, hidden] bf16
 * row-major.  Each bf16 x bf16 product is exact in double. */
void lpdo_head_logits(const uint16_t *h, const uint16_t *W, int64_t hidden, int64_t vocab,
                      double *x_out)
{
    for (int64_t v = 0; v < vocab; ++v) {
        const uint16_t *w = W + (size_t)v * (size_t)hidden;
        double acc = 0.0;
        for (int64_t k = 0; k < hidden; ++k)
            acc += logit_at(h, LPDO_BF16, k) * logit_at(w, LPDO_BF16, k);
        x_out[v] = acc;
    }
}

/* Selected-token logp of the listed rows through the LM head: materialise
 * the row's logits in double, then the same logsumexp and gather as
 * lpdo_row_logp.  hidden_t / hidden_r are [n_rows, hidden] bf16. */
uint32_t lpdo_score_head_rows(const uint16_t *hidden_t, const uint16_t *hidden_r,
                              const uint16_t *W, int64_t hidden, int64_t vocab,
                              const int32_t *token_ids, const int64_t *rows, int64_t n_sel,
                              double *logp_train, double *logp_rollout, double *dlogp)
{
    uint32_t status = 0;
    double *x = (double *)malloc((size_t)vocab * sizeof(double));
    for (int64_t i = 0; i < n_sel; ++i) {
        int64_t r = rows[i];
        const uint16_t *hs[2] = {hidden_t + (size_t)r * (size_t)hidden,
                                 hidden_r + (size_t)r * (size_t)hidden};
        double *outs[2] = {&logp_train[i], &logp_rollout[i]};
        for (int side = 0; side < 2; ++side) {
            lpdo_head_logits(hs[side], W, hidden, vocab, x);
            int64_t id = token_ids[r];
            if (id < 0 || id >= vocab) {
                *outs[side] = NAN;
                status |= LPDO_STATUS_TOKEN_OOB;
                continue;
            }
            double m = -INFINITY, s = 0.0;
            for (int64_t j = 0; j < vocab; ++j)
                if (x[j] > m)
                    m = x[j];
            for (int64_t j = 0; j < vocab; ++j)
                s += exp(x[j] - m);
            double lse = m + log(s);
            *outs[side] = x[id] - lse;
            if (!isfinite(lse))
                status |= LPDO_STATUS_NONFINITE;
        }
        dlogp[i] = logp_train[i] - logp_rollout[i];
    }
    free(x);
    return status;
}

/* ---- logit transform chain [TC] ----------------------------------------- */

#define LPDO_OP_SCALE 1   /* x <- x * p          (temperature 1/T, logit scale) */
#define LPDO_OP_SOFTCAP 2 /* x <- p * tanh(x / p) */

typedef struct {
    int32_t n_ops;
    int32_t kind[4];
    float param[4];
} lpdo_transform;

/* The chain applied to one logit, in order, in double. */
static double apply_chain(const lpdo_transform *c, double x)
{
    if (!c)
        return x;
    for (int k = 0; k < c->n_ops; ++k) {
        double p = (double)c->param[k];
        if (c->kind[k] == LPDO_OP_SCALE)
            x = x * p;
        else if (c->kind[k] == LPDO_OP_SOFTCAP)
            x = p * tanh(x / p);
    }
    return x;
}

/* Selected-token logp of one row after the chain: every logit (the selected
 * one included) is transformed, then the plain definition is applied. */
static uint32_t row_logp_chain(const void *row, int dtype, int64_t vocab, int64_t id,
                               const lpdo_transform *c, double *logp_out)
{
    if (id < 0 || id >= vocab) {
        *logp_out = NAN;
        return LPDO_STATUS_TOKEN_OOB;
    }
    double m = -INFINITY;
    int has_nan = 0;
    for (int64_t j = 0; j < vocab; ++j) {
        double x = apply_chain(c, logit_at(row, dtype, j));
        if (x > m)
            m = x;
        if (isnan(x))
            has_nan = 1;
    }
    double s = 0.0;
    if (m != -INFINITY)
        for (int64_t j = 0; j < vocab; ++j)
            s += exp(apply_chain(c, logit_at(row, dtype, j)) - m);
    if (has_nan)
        s = NAN;
    double lse = lse_of(m, s);
    double xs = apply_chain(c, logit_at(row, dtype, id));
    *logp_out = xs - lse;
    return (isfinite(lse) && isfinite(xs)) ? 0u : LPDO_STATUS_NONFINITE;
}

uint32_t lpdo_score_transformed(const void *train, int train_dtype, int64_t train_stride,
                                const void *rollout, int rollout_dtype, int64_t rollout_stride,
                                const lpdo_transform *train_chain, const lpdo_transform *rollout_chain,
                                int64_t n_rows, int64_t vocab, const int32_t *token_ids,
                                const uint8_t *mask, double clip_lo, double clip_hi,
                                double *logp_train, double *logp_rollout, double *dlogp,
                                lpdo_metrics *metrics)
{
    uint32_t status = 0;
    for (int64_t r = 0; r < n_rows; ++r) {
        logp_train[r] = logp_rollout[r] = dlogp[r] = 0.0;
        if (!mask[r])
            continue;
        status |= row_logp_chain(row_ptr(train, train_dtype, train_stride, r), train_dtype, vocab,
                                 token_ids[r], train_chain, &logp_train[r]);
        status |= row_logp_chain(row_ptr(rollout, rollout_dtype, rollout_stride, r), rollout_dtype,
                                 vocab, token_ids[r], rollout_chain, &logp_rollout[r]);
        dlogp[r] = logp_train[r] - logp_rollout[r];
    }
    if (metrics) {
        lpdo_metrics_from_dlogp(dlogp, mask, n_rows, clip_lo, clip_hi, metrics);
        metrics->status = status;
    }
    return status;
}

/* ---- training-only state [TS] ------------------------------------------- */

/* Entropy of the softmax of one row: H = -sum_j p_j log p_j with
 * p_j = exp(x_j - lse), written as H = lse - sum_j p_j x_j (serial in j). */
double lpdo_row_entropy(const void *row, int dtype, int64_t vocab)
{
    double m, s;
    lpdo_partial(row, dtype, 0, vocab, &m, &s);
    double lse = lse_of(m, s);
    double px = 0.0;
    for (int64_t j = 0; j < vocab; ++j) {
        double x = logit_at(row, dtype, j);
        double p = exp(x - lse);
        if (p > 0.0)
            px += p * x;
    }
    return lse - px;
}

/* Entropies of both sides for every active row (0 where inactive). */
void lpdo_entropy(const void *train, int train_dtype, int64_t train_stride,
                  const void *rollout, int rollout_dtype, int64_t rollout_stride,
                  int64_t n_rows, int64_t vocab, const uint8_t *mask,
                  double *ent_train, double *ent_rollout)
{
    for (int64_t r = 0; r < n_rows; ++r) {
        ent_train[r] = ent_rollout[r] = 0.0;
        if (!mask[r])
            continue;
        ent_train[r] = lpdo_row_entropy(row_ptr(train, train_dtype, train_stride, r), train_dtype, vocab);
        ent_rollout[r] = lpdo_row_entropy(row_ptr(rollout, rollout_dtype, rollout_stride, r),
                                          rollout_dtype, vocab);
    }
}

/* Gradient of grad * logp(x)[id] with respect to the row's logits:
 *   d/dx_j = grad * (1[j == id] - p_j),  p_j = exp(x_j - lse). */
void lpdo_logprob_backward_row(const void *row, int dtype, int64_t vocab, int64_t id, double grad,
                               double *out)
{
    double m, s;
    lpdo_partial(row, dtype, 0, vocab, &m, &s);
    double lse = lse_of(m, s);
    for (int64_t j = 0; j < vocab; ++j) {
        double p = exp(logit_at(row, dtype, j) - lse);
        out[j] = grad * ((j == id ? 1.0 : 0.0) - p);
    }
}

/* ---- attention partial merge [AM] ---------------------------------------- */

/* Merge K partial attention results for each of n rows, visiting the parts in
 * `order` (a permutation of 0..K-1):
 *   lse = log(sum_k exp(lse_k)),  out = sum_k exp(lse_k - lse) * out_k.
 * out_parts: [K][n][d] (f32), lse_parts: [K][n]; with lse_base2 the lse values
 * are log2-sum-exp2 and are converted to natural log first (and back for the
 * merged lse).  A part whose lse is -inf saw no keys for that row: it carries
 * no weight and its out values are not read (a backend may leave them 0 or
 * NaN).  A row no part saw merges to out = 0, lse = -inf. */
void lpdo_attn_merge(const float *out_parts, const float *lse_parts, int K, int64_t n, int d,
                     int lse_base2, const int32_t *order, double *out, double *out_lse)
{
    const double ln2 = log(2.0);
    for (int64_t i = 0; i < n; ++i) {
        double *oi = out + (size_t)i * (size_t)d;
        for (int j = 0; j < d; ++j)
            oi[j] = 0.0;
        double m = -INFINITY;
        for (int k = 0; k < K; ++k) {
            double l = lse_parts[(size_t)order[k] * (size_t)n + (size_t)i];
            if (lse_base2)
                l *= ln2;
            if (l > m)
                m = l;
        }
        if (m == -INFINITY) {
            out_lse[i] = -INFINITY;
            continue;
        }
        double s = 0.0;
        for (int k = 0; k < K; ++k) {
            double l = lse_parts[(size_t)order[k] * (size_t)n + (size_t)i];
            if (lse_base2)
                l *= ln2;
            s += exp(l - m);
        }
        double lse = m + log(s);
        for (int k = 0; k < K; ++k) {
            int kk = order[k];
            double l = lse_parts[(size_t)kk * (size_t)n + (size_t)i];
            if (l == -INFINITY)
                continue;
            if (lse_base2)
                l *= ln2;
            double w = exp(l - lse);
            const float *o = out_parts + ((size_t)kk * (size_t)n + (size_t)i) * (size_t)d;
            for (int j = 0; j < d; ++j)
                oi[j] += w * (double)o[j];
        }
        out_lse[i] = lse_base2 ? lse / ln2 : lse;
    }
}

/* ---- merge-order drift summary [LP] ---------------------------------------
 * The LogProb knobs table (row 5) names the merge order of the per-shard
 * partials as a drift source; the summary of that diagnostic compares two
 * per-token results of the same rows, a (the fixed global shard order) and b
 * (another merge order), over the active rows only:
 *   max_abs_t / max_abs_r  the largest |b - a| of each side, formed in double
 *                          from the float32 values; a NaN difference (either
 *                          value NaN) counts as larger than any number;
 *   row_t / row_r          the lowest active row attaining it (-1 with no
 *                          active row);
 *   n_differ               active rows where a and b are different numbers on
 *                          either side (+0 and -0 are the same number, and two
 *                          NaNs count as the same);
 *   frac_differ            n_differ / n_active (0 with no active row). */
typedef struct {
    double max_abs_t;
    double max_abs_r;
    int64_t row_t;
    int64_t row_r;
    int64_t n_active;
    int64_t n_differ;
    double frac_differ;
} lpdo_drift_summary;

/* 1 when |b - a| of this row beats the best so far (ties keep the lower row,
 * which was seen first) */
static int drift_beats(double diff, double best, int have)
{
    if (!have)
        return 1;
    if (isnan(best))
        return 0;
    if (isnan(diff))
        return 1;
    return diff > best;
}

static int same_number(float a, float b)
{
    if (isnan(a) && isnan(b))
        return 1;
    return a == b;
}

void lpdo_logp_drift(int64_t n_rows, const float *a_t, const float *a_r, const float *b_t,
                     const float *b_r, const uint8_t *mask, lpdo_drift_summary *out)
{
    out->max_abs_t = 0.0;
    out->max_abs_r = 0.0;
    out->row_t = -1;
    out->row_r = -1;
    out->n_active = 0;
    out->n_differ = 0;
    out->frac_differ = 0.0;
    for (int64_t r = 0; r < n_rows; ++r) {
        if (!mask[r])
            continue;
        double dt = fabs((double)b_t[r] - (double)a_t[r]);
        double dr = fabs((double)b_r[r] - (double)a_r[r]);
        if (drift_beats(dt, out->max_abs_t, out->row_t >= 0)) {
            out->max_abs_t = dt;
            out->row_t = r;
        }
        if (drift_beats(dr, out->max_abs_r, out->row_r >= 0)) {
            out->max_abs_r = dr;
            out->row_r = r;
        }
        out->n_active += 1;
        if (!same_number(a_t[r], b_t[r]) || !same_number(a_r[r], b_r[r]))
            out->n_differ += 1;
    }
    if (out->n_active > 0)
        out->frac_differ = (double)out->n_differ / (double)out->n_active;
}
