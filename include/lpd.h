/*
 * lpd.h - selected-token logprob drift scoring on one GB300 (sm_103a).
 *
 * C ABI of liblpd.so.  Plain pointers and sizes only; no C++ or torch types.
 *
 * What it computes ("WS2 Cross-Config Logprob Drift Contract", section
 * "Measurement Contract"): the already-sampled sequence is teacher-forced
 * through both the training-side and the rollout-side logits; for every
 * active response/action token r
 *
 *     logp_side[r] = x_side[r, id[r]] - log(sum_j exp(x_side[r, j]))
 *     dlogp[r]     = logp_train[r] - logp_rollout[r]
 *
 * and, over active tokens only (section "Diagnostics"): ratio0 = exp(dlogp)
 * (reported as its mean), clipfrac0 (fraction of ratio0 outside the clip
 * range), approx_kl0 = mean of exp(dlogp) - 1 - dlogp, and the mean, 95th and
 * 99th percentile and maximum of |dlogp|.  Percentiles are nearest-rank: the
 * value of 1-based rank ceil(p * A / 100) among the A ascending |dlogp|.
 *
 * Row convention ("[WS2] Framework for ablation experiment", LogProb knobs
 * table, row 8, "pre-shifted input convention"): logits row r scores
 * token_ids[r]; the caller does the shift.  action_mask[r] != 0 marks an
 * active token; prompt and padding rows carry 0, so left and right padding
 * look the same to the library.  Inactive rows are never read: their logits
 * and token ids may hold anything.
 *
 * Determinism: each row's arithmetic order depends only on the vocabulary
 * size and the logical column index, never on the row's position, the batch,
 * the grid or the storage dtype, so the same row gives bitwise-identical
 * results whatever batch it is scored in (the batch-composition control of
 * "Attention Debug Matrix", section "Metrics", must be bitwise zero).  No
 * floating-point atomics are used anywhere.
 *
 * Memory: the caller owns every buffer.  Logits, ids, mask, per-token outputs,
 * the metrics record and the workspace are DEVICE pointers (lpd_score_host
 * alone takes its logits, ids and mask in host memory); nothing is allocated
 * or retained by the library between calls.  All calls are asynchronous on
 * the given stream (a cudaStream_t passed as void*, NULL for the legacy
 * default stream) and, all but lpd_score_host, may be captured in a CUDA
 * graph.
 *
 * Errors: invalid arguments are detected on the host before anything is
 * launched and returned as a negative LPD_ERR_* code.  Problems that only the
 * device can see are reported in lpd_metrics.status (LPD_STATUS_* bits) and
 * never trap: a token id outside [0, vocab) on an active row, or a non-finite
 * log-sum-exp or selected logit on an active row.  When status != 0 the
 * metric values are unspecified; per-token outputs of the offending rows are
 * NaN or non-finite.
 *
 * Bounded waits: no kernel waits without a limit.  The streaming row pass
 * gives up a pipeline wait after 2 s (4 s in the fused LM-head kernel), sets
 * LPD_STATUS_TIMEOUT, lets its in-flight copies land and returns; the context
 * stays usable.  For tests of that path, the environment variable
 * LPD_STALL_ROW_PASS=1 (read at each call) makes one CTA of the row pass
 * withhold its first copy: the call then takes about 4 s and returns with
 * LPD_STATUS_TIMEOUT.
 */
#ifndef LPD_H
#define LPD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- element types --------------------------------------------------- */
#define LPD_BF16 0 /* bfloat16, 2 bytes */
#define LPD_F32 1  /* IEEE float32, 4 bytes */

/* ---- return codes ----------------------------------------------------- */
#define LPD_OK 0
#define LPD_ERR_NULL_POINTER (-1) /* a required pointer is NULL */
#define LPD_ERR_BAD_SIZE (-2)     /* n_rows < 0, vocab <= 0, hidden <= 0, ... */
#define LPD_ERR_BAD_DTYPE (-3)    /* dtype not LPD_BF16 / LPD_F32, or mixed within a side */
#define LPD_ERR_BAD_STRIDE (-4)   /* row_stride < columns of that tensor */
#define LPD_ERR_BAD_CLIP (-5)     /* clip bounds not 0 < lo <= hi (finite) */
#define LPD_ERR_BAD_SHARDS (-6)   /* shard ranges do not tile [0, vocab) exactly */
#define LPD_ERR_WORKSPACE (-7)    /* workspace NULL or smaller than lpd_workspace_size() */
#define LPD_ERR_CUDA (-8)         /* a CUDA runtime call failed (launch, attribute) */
#define LPD_ERR_ALIGNMENT (-9)    /* a pointer or stride breaks a stated alignment rule */
#define LPD_ERR_UNSUPPORTED (-10) /* a size outside what this library supports */
#define LPD_ERR_BAD_TRANSFORM (-11) /* transform chain: bad op count, kind or parameter */
#define LPD_ERR_BAD_MEMORY (-12)    /* a host-side argument points to device memory */

/* ---- device-reported status bits (lpd_metrics.status) ------------------ */
#define LPD_STATUS_TOKEN_OOB 1u /* an active row's token id is outside [0, vocab) */
#define LPD_STATUS_NONFINITE 2u /* non-finite log-sum-exp or selected logit on an active row */
#define LPD_STATUS_TIMEOUT 4u   /* an internal pipeline wait gave up (never expected) */

/* ---- result flags (lpd_metrics.flags) --------------------------------- */
#define LPD_FLAG_NO_ACTIVE 1u /* zero active tokens: every metric is 0 */
#define LPD_FLAG_NO_PERCENTILES 2u /* p95 / p99 not available (a record merged from
                                    * per-rank records): NaN */

/* ---- workspace kinds --------------------------------------------------- */
#define LPD_KIND_SCORE 0   /* lpd_score and its stages */
#define LPD_KIND_SHARDED 1 /* lpd_score_sharded */

/* One side's logits: [n_rows, row_stride] row-major, columns [0, vocab) used. */
typedef struct {
    const void *ptr;    /* device pointer to row 0, column 0 */
    int32_t dtype;      /* LPD_BF16 or LPD_F32 */
    int32_t reserved;   /* set to 0 */
    int64_t row_stride; /* elements between consecutive rows, >= vocab */
} lpd_logits;

/* One vocab shard of one side: [n_rows, row_stride] holding global columns
 * [v_start, v_end) as local columns [0, v_end - v_start), as a tensor-parallel
 * vocab split would produce ("[WS2] Framework for ablation experiment",
 * LogProb knobs table, row 3: per-rank (vocab_start, vocab_end)). */
typedef struct {
    const void *ptr;
    int32_t dtype;
    int32_t reserved;
    int64_t row_stride; /* >= v_end - v_start */
    int64_t v_start;
    int64_t v_end;
} lpd_shard;

/* Drift diagnostics over active tokens (device-resident, written by the
 * library).  Field meaning: "WS2 Cross-Config Logprob Drift Contract",
 * section "Diagnostics"; n_active and argmax_row are the active-token count
 * and worst-token metadata of roadmap item B1 (argmax_row is the lowest row
 * index among ties of max |dlogp|, -1 when there is no active token). */
typedef struct {
    int64_t n_active;
    int64_t argmax_row;
    uint32_t flags;  /* LPD_FLAG_* */
    uint32_t status; /* LPD_STATUS_* bits, 0 when every active row was valid */
    double ratio0_mean;
    double clipfrac0;
    double approx_kl0;
    double mean_abs_dlogp;
    double p95_abs_dlogp;
    double p99_abs_dlogp;
    double max_abs_dlogp;
} lpd_metrics;

/* Kernel backend descriptor ("WS2 Cross-Config Logprob Drift Contract",
 * section "Kernel Integration Contract": stable id, semantic operator name,
 * architectures, dtypes, determinism properties, build-time flags, fallback
 * behaviour, build fingerprint; section "Mapping to Current Code": the
 * fast-math and architecture build knobs). */
typedef struct {
    char backend_id[32];   /* "lpd.sm103a.v1" */
    char op_name[48];      /* "selected_logprob_drift" */
    char arch[16];         /* "sm_103a" */
    char dtypes[32];       /* "bf16,f32" (per side, may differ) */
    int32_t deterministic; /* 1: bitwise repeatable run to run */
    int32_t batch_invariant; /* 1: a row's result is independent of its batch */
    int32_t fast_math;     /* 0: built without --use_fast_math */
    int32_t has_fallback;  /* 0: no CPU or library fallback exists */
    char fingerprint[96];  /* compiler version and build date */
} lpd_backend_info_t;

/* Logit transform chain of one side ("[WS2] Framework for ablation
 * experiment", LogProb knobs table, row 7): ops applied in order to every logit
 * before the softmax.  LPD_OP_SCALE: x <- x * param (temperature T is param =
 * 1/T; logit scale); LPD_OP_SOFTCAP: x <- param * tanh(x / param).  Parameters
 * must be finite and > 0.  n_ops = 0 is the identity. */
#define LPD_OP_SCALE 1
#define LPD_OP_SOFTCAP 2
#define LPD_MAX_TRANSFORM_OPS 4
typedef struct {
    int32_t n_ops;
    int32_t kind[LPD_MAX_TRANSFORM_OPS];
    float param[LPD_MAX_TRANSFORM_OPS];
} lpd_transform;

/* ---- sizing and introspection ----------------------------------------- */

/* Bytes of device workspace that a call of the given kind needs for n_rows
 * rows (vocab and n_shards are used by the sharded kind; pass 0
 * otherwise).  Returns 0 for invalid arguments. */
size_t lpd_workspace_size(int32_t kind, int64_t n_rows, int64_t vocab, int32_t n_shards);

/* Fills *info.  Returns LPD_OK, or LPD_ERR_NULL_POINTER. */
int lpd_backend_info(lpd_backend_info_t *info);

/* Static English text for a return code or a single status bit. */
const char *lpd_strerror(int code);

/* ---- the scoring path --------------------------------------------------- */

/* Whole path ("Measurement Contract" and "Diagnostics" sections): select
 * active rows, score both sides, then the metrics.  Equivalent to
 * lpd_select_active + lpd_token_logp + lpd_drift_metrics on one stream.
 *
 * train, rollout   host structs describing device logits [n_rows, vocab];
 *                  dtypes may differ between the sides.
 * token_ids        device int32[n_rows].
 * action_mask      device uint8[n_rows].
 * clip_lo, clip_hi ratio0 bounds; a ratio equal to a bound is inside.
 * out_logp_train, out_logp_rollout, out_dlogp
 *                  device float32[n_rows] each, or NULL to skip; inactive rows
 *                  receive 0.
 * out_metrics      device lpd_metrics (required).
 * workspace        device buffer of at least
 *                  lpd_workspace_size(LPD_KIND_SCORE, n_rows, 0, 0) bytes,
 *                  256-byte aligned.
 * stream           cudaStream_t or NULL.
 * n_rows may be 0 (then out_metrics reports zero active tokens). */
int lpd_score(const lpd_logits *train, const lpd_logits *rollout, int64_t n_rows,
              int64_t vocab, const int32_t *token_ids, const uint8_t *action_mask,
              double clip_lo, double clip_hi, float *out_logp_train,
              float *out_logp_rollout, float *out_dlogp, lpd_metrics *out_metrics,
              void *workspace, size_t workspace_bytes, void *stream);

/* lpd_score on logits held in HOST memory (page-locked for full link speed).
 * The scorer never reads an inactive row ("Measurement Contract": prompt and
 * padding positions are excluded), so only active rows cross the host-device
 * link: the host reads action_mask_host during the call and, for every run of
 * consecutive active rows, issues one 2-D copy per side into the same rows of
 * the caller's device staging buffers; ids and mask are copied whole.  Then
 * lpd_score runs on the staged rows.  Everything is ordered on `stream`.
 * Inactive rows of the staging buffers keep whatever they held.
 *
 * train_host, rollout_host   lpd_logits over host memory [n_rows, vocab].
 * train_dev, rollout_dev     lpd_logits over device memory [n_rows, vocab]
 *                            (row_stride >= vocab), each with the dtype of
 *                            its host side, else LPD_ERR_BAD_DTYPE.
 * token_ids_host, action_mask_host   host int32[n_rows], uint8[n_rows].
 * token_ids_dev, action_mask_dev     device int32[n_rows], uint8[n_rows].
 * out_h2d_bytes   host int64, or NULL: the bytes this call copies to the
 *                 device (active rows of both sides, ids and mask).
 * The host reads action_mask_host itself: a pointer the CUDA runtime reports
 * as device memory returns LPD_ERR_BAD_MEMORY before anything is copied.
 * Other arguments, outputs and errors as lpd_score.  As with any
 * asynchronous copy, the host buffers must not change until the copies have
 * completed on `stream`.  The copies issued depend on the mask's contents at
 * call time, so the call is not meant for CUDA-graph capture. */
int lpd_score_host(const lpd_logits *train_host, const lpd_logits *rollout_host,
                   const lpd_logits *train_dev, const lpd_logits *rollout_dev,
                   int64_t n_rows, int64_t vocab, const int32_t *token_ids_host,
                   const uint8_t *action_mask_host, int32_t *token_ids_dev,
                   uint8_t *action_mask_dev, double clip_lo, double clip_hi,
                   float *out_logp_train, float *out_logp_rollout, float *out_dlogp,
                   lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes,
                   int64_t *out_h2d_bytes, void *stream);

/* Stage 1 of lpd_score ("Measurement Contract": prompt, padding and masked
 * positions are excluded): the order-preserving list of active rows with
 * their token ids, and their count, into the workspace; zeroes the per-token
 * outputs of inactive rows and clears out_metrics->status.  The three stages
 * must run in order on one stream with the same workspace, n_rows and output
 * pointers. */
int lpd_select_active(int64_t n_rows, const int32_t *token_ids, const uint8_t *action_mask,
                      float *out_logp_train, float *out_logp_rollout, float *out_dlogp,
                      lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes,
                      void *stream);

/* Stage 2 of lpd_score: the streaming row pass over the rows stage 1 listed.
 * For each active row, both sides' log-sum-exp in one read of each logits row,
 * the selected-logit gather, and the per-token logp_train, logp_rollout and
 * dlogp (plus the per-row values stage 3 reduces). */
int lpd_token_logp(const lpd_logits *train, const lpd_logits *rollout, int64_t n_rows,
                   int64_t vocab, float *out_logp_train, float *out_logp_rollout,
                   float *out_dlogp, lpd_metrics *out_metrics, void *workspace,
                   size_t workspace_bytes, void *stream);

/* Stage 3 of lpd_score ("Diagnostics"): metrics over the active rows scored
 * by stage 2, into out_metrics (everything but status, which stages 1-2
 * own). */
int lpd_drift_metrics(int64_t n_rows, double clip_lo, double clip_hi,
                      lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes,
                      void *stream);

/* Global metrics of a data-parallel run from its per-rank records ("WS2
 * Cross-Config Logprob Drift Contract", "Diagnostics": the same metrics per
 * rank and globally), where only the small records are exchanged.  HOST call,
 * no GPU work: per_rank is a host array of n_ranks lpd_metrics in rank order
 * (each rank's lpd_score record, copied to the host), row_offsets an optional
 * host int64[n_ranks] mapping each rank's local rows to global ones (NULL: all
 * 0), out a host record.  Combined exactly, visiting ranks in rank order so
 * the result does not depend on the collective that gathered them:
 *   n_active    the sum;  status  the OR;
 *   ratio0_mean, clipfrac0, approx_kl0, mean_abs_dlogp
 *               means weighted by each rank's n_active (sum of a_k m_k in rank
 *               order, divided by the total);
 *   max_abs_dlogp, argmax_row
 *               the largest per-rank maximum; ties go to the earlier rank,
 *               whose rows come first; argmax_row + that rank's offset;
 *   p95 / p99   NaN, with LPD_FLAG_NO_PERCENTILES: percentiles of the union are
 *               not a function of per-rank ones (gather the per-token dlogp and
 *               use lpd_drift_metrics_from_dlogp for them);
 *   flags       LPD_FLAG_NO_ACTIVE when the total is 0 (every mean 0, argmax -1).
 * Ranks with n_active == 0 contribute only their status.  Returns
 * LPD_ERR_NULL_POINTER / LPD_ERR_BAD_SIZE (n_ranks < 1 or a negative count). */
int lpd_merge_rank_metrics(const lpd_metrics *per_rank, const int64_t *row_offsets, int32_t n_ranks,
                           lpd_metrics *out);

/* Stage 3 over caller-given per-token values: the metrics record of the
 * rows with action_mask != 0, with d = dlogp[r] (float32, widened exactly) in
 * place of the scorer's own values.  For data-parallel runs: the ranks'
 * out_dlogp and masks gathered in rank order give the exact metrics of the
 * union, percentiles included ("WS2 Cross-Config Logprob Drift Contract",
 * "Diagnostics": the same metrics globally and per rank).  A non-finite value
 * on an active row sets LPD_STATUS_NONFINITE.
 * dlogp        device float32[n_rows]; action_mask device uint8[n_rows].
 * workspace    lpd_workspace_size(LPD_KIND_SCORE, n_rows, 0, 0) bytes. */
int lpd_drift_metrics_from_dlogp(int64_t n_rows, const float *dlogp, const uint8_t *action_mask,
                                 double clip_lo, double clip_hi, lpd_metrics *out_metrics,
                                 void *workspace, size_t workspace_bytes, void *stream);

/* lpd_score with a logit transform chain per side (each may be NULL for the
 * identity).  The chains are part of what is compared: different chains on the
 * two sides show up as drift, which the pages treat as a correctness bug rather
 * than noise.  Same workspace kind and outputs as lpd_score; a chain that is
 * not valid returns LPD_ERR_BAD_TRANSFORM before any launch. */
int lpd_score_transformed(const lpd_logits *train, const lpd_logits *rollout,
                          const lpd_transform *train_chain, const lpd_transform *rollout_chain,
                          int64_t n_rows, int64_t vocab, const int32_t *token_ids,
                          const uint8_t *action_mask, double clip_lo, double clip_hi,
                          float *out_logp_train, float *out_logp_rollout, float *out_dlogp,
                          lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes,
                          void *stream);

/* lpd_score plus the entropy of each side's softmax per active token
 * ("[WS2] Framework for ablation experiment", LogProb knobs table, row 11:
 * training-only state), H = -sum_j p_j log p_j, accumulated in the same single
 * read of each row.  out_entropy_train / out_entropy_rollout are device
 * float32[n_rows] (at least one non-NULL; inactive rows receive 0). */
int lpd_score_entropy(const lpd_logits *train, const lpd_logits *rollout, int64_t n_rows,
                      int64_t vocab, const int32_t *token_ids, const uint8_t *action_mask,
                      double clip_lo, double clip_hi, float *out_logp_train,
                      float *out_logp_rollout, float *out_dlogp, float *out_entropy_train,
                      float *out_entropy_rollout, lpd_metrics *out_metrics, void *workspace,
                      size_t workspace_bytes, void *stream);

/* Gradient of the selected-token logprob with respect to the logits, for one
 * side (row 11 of the same table): for every active row r and column j,
 *   out[r, j] = grad_logp[r] * (1[j == token_ids[r]] - exp(x[r, j] - lse[r])),
 * with lse[r] = x[r, token_ids[r]] - logp[r] taken from this row's logp as
 * returned by the scoring calls; inactive rows receive 0.  One read of the
 * logits and one write of the gradient.
 * logits       the side's lpd_logits [n_rows, vocab] (any row stride).
 * logp         device float32[n_rows], grad_logp device float32[n_rows].
 * out_dlogits  device [n_rows, out_row_stride] of out_dtype (LPD_BF16 or
 *              LPD_F32), columns [0, vocab) written.
 * An active row whose id is outside [0, vocab) receives NaN. */
int lpd_logprob_backward(const lpd_logits *logits, int64_t n_rows, int64_t vocab,
                         const int32_t *token_ids, const uint8_t *action_mask, const float *logp,
                         const float *grad_logp, void *out_dlogits, int32_t out_dtype,
                         int64_t out_row_stride, void *stream);

/* Vocab-sharded scoring ("[WS2] Framework for ablation experiment", LogProb
 * knobs table, rows 3-5 and 8).  Each side's vocabulary arrives as n_shards
 * tensors whose [v_start, v_end) ranges must tile [0, vocab) exactly, in any
 * array order (else LPD_ERR_BAD_SHARDS, "fail closed on missing vocab-shard
 * bounds").  Each shard gives its own partial (max, sum exp); the partials are
 * merged in global vocab-shard order (ascending v_start), and the selected
 * logit comes from the single shard that owns the id.  All shards of a side
 * share one dtype.  1 <= n_shards <= 16.
 *
 * merge_perm       optional HOST int32[n_shards]: a permutation of the shard
 *                  positions in vocab order.  When given, each row is merged a
 *                  second time in that order and the resulting logp is written
 *                  to out_perm_logp_train / out_perm_logp_rollout (device
 *                  float32[n_rows] each, may be NULL) as a merge-order drift
 *                  diagnostic (row 5: merge order as a drift source).
 * The fixed-order result is what out_logp_* / out_dlogp / out_metrics carry.
 * workspace        lpd_workspace_size(LPD_KIND_SHARDED, n_rows, vocab, n_shards). */
int lpd_score_sharded(const lpd_shard *train, const lpd_shard *rollout, int32_t n_shards,
                      int64_t n_rows, int64_t vocab, const int32_t *token_ids,
                      const uint8_t *action_mask, double clip_lo, double clip_hi,
                      const int32_t *merge_perm, float *out_logp_train,
                      float *out_logp_rollout, float *out_dlogp,
                      float *out_perm_logp_train, float *out_perm_logp_rollout,
                      lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes,
                      void *stream);

/* Summary of the merge-order diagnostic ("[WS2] Framework for ablation
 * experiment", LogProb knobs table, row 5: the merge order of the per-shard
 * partials as a drift source), next to the per-token outputs it summarises.
 * Two per-token results of the same rows are compared over the active rows:
 * a = the fixed global shard order (out_logp_* of lpd_score_sharded), b = the
 * permuted order (out_perm_logp_*), or any other pair of per-token logp results.
 *   max_abs_dlogp_train / _rollout  largest |b - a| of each side (float32
 *                        difference widened to double; a NaN difference, i.e.
 *                        either value NaN, ranks above every number);
 *   row_train / row_rollout  lowest active row attaining it (-1: no active row);
 *   n_active             active rows (action_mask != 0);
 *   n_differ             active rows where either side's b is a different
 *                        number from a (+0 equals -0; two NaNs count as equal);
 *   frac_differ          n_differ / n_active (0 with no active row).
 * `scratch` is working space of the call; its contents afterwards mean
 * nothing. */
typedef struct {
    double max_abs_dlogp_train;
    double max_abs_dlogp_rollout;
    int64_t row_train;
    int64_t row_rollout;
    int64_t n_active;
    int64_t n_differ;
    double frac_differ;
    uint64_t scratch[4];
} lpd_logp_drift;

/* logp_train_a, logp_rollout_a, logp_train_b, logp_rollout_b: device float32
 * [n_rows]; action_mask: device uint8 [n_rows]; out: device lpd_logp_drift
 * (8-byte aligned), written asynchronously on `stream`.  Inactive rows are never
 * read.  0 <= n_rows < 2^32 - 1 (else LPD_ERR_BAD_SIZE / LPD_ERR_UNSUPPORTED);
 * NULL pointers give LPD_ERR_NULL_POINTER (the row arrays may be NULL when
 * n_rows == 0).  No workspace; nothing is allocated. */
int lpd_logp_drift_summary(int64_t n_rows, const float *logp_train_a, const float *logp_rollout_a,
                           const float *logp_train_b, const float *logp_rollout_b,
                           const uint8_t *action_mask, lpd_logp_drift *out, void *stream);

/* ---- reduction topology arms ------------------------------------------------- */

/* The three ways a vocab-parallel logprob can combine its shards
 * ("[WS2] Framework for ablation experiment", LogProb knobs table, row 4:
 * reduction topology), run on the same shards so that their drift against
 * each other is pure arithmetic.  All three compute the same logp exactly; they
 * differ in rounding only.
 *   LPD_TOPO_ALLGATHER_PARTIALS_FIXED_MERGE  every shard's (m, s) partial,
 *       merged pairwise (online softmax) in shard order or `reduce_order`:
 *       the main result of lpd_score_sharded.
 *   LPD_TOPO_ALLREDUCE_PARTIALS  a max reduction M = max_k m_k, then a sum
 *       reduction S = sum_k s_k exp(m_k - M) in fp32, in shard order or
 *       `reduce_order` (the order an all-reduce adds in); lse = M + log S per
 *       side, and dlogp is the difference of the two sides' logp.
 *   LPD_TOPO_ALLGATHER_LOGITS  the shards gathered into full rows in the
 *       workspace (a copy kernel), then one pass over each row: bitwise what
 *       lpd_score gives on the concatenated logits.
 *       `reduce_order` is ignored. */
#define LPD_TOPO_ALLGATHER_PARTIALS_FIXED_MERGE 0
#define LPD_TOPO_ALLREDUCE_PARTIALS 1
#define LPD_TOPO_ALLGATHER_LOGITS 2

/* Workspace bytes for lpd_score_sharded_topology (0 for invalid arguments).
 * The gather arm also holds both sides' gathered logits: n_rows rows of
 * vocab elements of each side's dtype, each row padded to 16 bytes. */
size_t lpd_topology_workspace_size(int32_t topology, int64_t n_rows, int64_t vocab,
                                   int32_t n_shards, int32_t dtype_train,
                                   int32_t dtype_rollout);

/* lpd_score_sharded with a chosen reduction topology.  Arguments, outputs,
 * status and errors are those of lpd_score_sharded without its permuted-merge
 * outputs; `reduce_order` is a HOST int32[n_shards] permutation (else
 * LPD_ERR_BAD_SHARDS) or NULL for ascending shard order.  An unknown topology
 * returns LPD_ERR_UNSUPPORTED.  workspace: lpd_topology_workspace_size(...)
 * bytes with the shards' dtypes, 256-byte aligned. */
int lpd_score_sharded_topology(const lpd_shard *train, const lpd_shard *rollout,
                               int32_t n_shards, int64_t n_rows, int64_t vocab,
                               const int32_t *token_ids, const uint8_t *action_mask,
                               double clip_lo, double clip_hi, int32_t topology,
                               const int32_t *reduce_order, float *out_logp_train,
                               float *out_logp_rollout, float *out_dlogp,
                               lpd_metrics *out_metrics, void *workspace,
                               size_t workspace_bytes, void *stream);

/* Fused LM-head scoring ("[WS2] Framework for ablation experiment", LogProb
 * knobs table, rows 9-10: the head GEMM and its fusion tiling).  The logits
 * x_side[r, v] = sum_k hidden_side[r, k] * W[v, k] are formed tile by tile on
 * the tensor cores (bf16 inputs, fp32 accumulation in a fixed k order, no
 * split-K) and folded into an online log-sum-exp as they are produced; they are
 * never written to memory.  Per-token outputs, metrics, status and errors are
 * those of lpd_score.
 *
 * hidden_train, hidden_rollout  device bf16 [n_rows, hidden], row-major, dense.
 * W                             device bf16 [vocab, hidden], row-major, dense.
 * hidden must be a multiple of 64 and the three pointers 16-byte aligned, else
 * LPD_ERR_ALIGNMENT.
 * workspace        lpd_fused_workspace_size(n_rows, hidden, vocab) bytes,
 *                  256-byte aligned (holds the active hidden rows of both sides
 *                  densely and one 20-byte partial per active row and 256-wide
 *                  vocab tile). */
size_t lpd_fused_workspace_size(int64_t n_rows, int64_t hidden, int64_t vocab);

int lpd_score_fused(const void *hidden_train, const void *hidden_rollout, const void *W,
                    int64_t n_rows, int64_t hidden, int64_t vocab, const int32_t *token_ids,
                    const uint8_t *action_mask, double clip_lo, double clip_hi,
                    float *out_logp_train, float *out_logp_rollout, float *out_dlogp,
                    lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes,
                    void *stream);

/* lpd_score_fused with a logit transform chain per side (each may be NULL for
 * the identity; "[WS2] Framework for ablation experiment", LogProb knobs table,
 * row 7).  Each fp32 logit out of the tensor cores goes through its side's
 * chain, with the same arithmetic as lpd_score_transformed, before the online
 * log-sum-exp sees it and before the selected logit is taken; the columns past
 * `vocab` in the last tile stay out of the sum.  Arguments, workspace, outputs
 * and errors are those of lpd_score_fused; a chain that is not valid returns
 * LPD_ERR_BAD_TRANSFORM before any launch. */
int lpd_score_fused_transformed(const void *hidden_train, const void *hidden_rollout,
                                const void *W, const lpd_transform *train_chain,
                                const lpd_transform *rollout_chain, int64_t n_rows,
                                int64_t hidden, int64_t vocab, const int32_t *token_ids,
                                const uint8_t *action_mask, double clip_lo, double clip_hi,
                                float *out_logp_train, float *out_logp_rollout,
                                float *out_dlogp, lpd_metrics *out_metrics, void *workspace,
                                size_t workspace_bytes, void *stream);

/* ---- attention (out, lse) merge --------------------------------------------- */

/* Split-KV / context-parallel attention partials are merged with the same
 * online-softmax algebra as the vocab shards above ("Attention Debug Matrix",
 * row A7 merge_order; "[WS2] Framework for ablation experiment", Attention
 * knobs table, rows 6-7: LSE domain/base and the CP / split-K merge order).
 * Part k computed attention of each query row over one block of keys and
 * returned its normalised output out_k[r, :] and its log-sum-exp lse_k[r].
 * For every row r the merge gives
 *
 *     lse[r] = log(sum_k exp(lse_k[r])),   out[r, :] = sum_k exp(lse_k[r] - lse[r]) out_k[r, :]
 *
 * folding the parts one at a time, in `order`, into a running state
 * (max m, sum s, unnormalised acc): a part above the running max rescales the
 * state by exp(m - lse_k), the others add exp(lse_k - m) out_k; the result is
 * acc / s and m + log(s).  Arithmetic is fp32 with a fixed per-row order, so
 * the result depends on `order` only through rounding: which order is taken is
 * the A7 diagnostic knob.  A part with lse_k[r] = -inf saw no keys for row r:
 * it carries no weight and its out values are not read (they may be NaN).  A
 * row no part saw gets out = 0 and lse = -inf.
 *
 * out_parts   device [n_parts][n_rows][head_dim], dense, dtype LPD_F32 or
 *             LPD_BF16 (a partial state downcast to bf16, Attention knobs row
 *             8), 16-byte aligned; head_dim * element size must be a multiple
 *             of 16 bytes (head_dim % 4 == 0 for f32, % 8 for bf16), else
 *             LPD_ERR_ALIGNMENT.
 * lse_parts   device float [n_parts][n_rows], dense.
 * lse_base2   0: lse values are natural-log (log-sum-exp); 1: base 2
 *             (log2-sum-exp2, as some kernels export).  Inputs and the merged
 *             lse use the same base.  Other values: LPD_ERR_BAD_SIZE.
 * order       HOST int32[n_parts], a permutation of 0..n_parts-1 (else
 *             LPD_ERR_BAD_SHARDS); NULL means ascending global block index
 *             0, 1, ..., n_parts-1, the fixed order.
 * out         device float [n_rows][head_dim], 16-byte aligned.
 * out_lse     device float [n_rows].
 * 1 <= n_parts <= LPD_ATTN_MAX_PARTS and one part at most 2^32 - 2 16-byte
 * chunks (n_rows * head_dim * element size < 64 GB), else LPD_ERR_UNSUPPORTED;
 * 0 <= n_rows < 2^32 - 1 and head_dim >= 1 (else LPD_ERR_BAD_SIZE).  No
 * workspace; nothing is allocated. */
#define LPD_ATTN_MAX_PARTS 64

int lpd_attn_merge(const void *out_parts, int32_t parts_dtype, const float *lse_parts,
                   int32_t n_parts, int64_t n_rows, int32_t head_dim, int32_t lse_base2,
                   const int32_t *order, float *out, float *out_lse, void *stream);

/* Summary of an order-drift run.  max_abs_dout is the largest |out_a - out_b|
 * over all rows and columns, max_abs_dlse the largest |lse_a - lse_b| (0 where
 * both are -inf); row_dout / row_dlse the lowest row attaining each (NaN ranks
 * above every number, so a NaN anywhere is what gets reported).  With
 * n_rows == 0 both maxima are 0 and both rows -1.  `scratch` is working
 * space of the call; its contents afterwards mean nothing. */
typedef struct {
    double max_abs_dout;
    double max_abs_dlse;
    int64_t row_dout;
    int64_t row_dlse;
    uint64_t scratch[2];
} lpd_merge_drift;

/* The merge-order diagnostic itself: merges the same partials in order_a and
 * in order_b in one pass over them and reports how far the two results are
 * apart.  Arguments are those of lpd_attn_merge; out / out_lse receive the
 * order_a result (bitwise what lpd_attn_merge gives for order_a), and
 *   row_dout   device float [n_rows]: max over the row's columns of |out_a - out_b|,
 *   row_dlse   device float [n_rows]: |lse_a - lse_b| (0 where both are -inf),
 *   drift      device lpd_merge_drift, the summary above.
 * order_a and order_b are host permutations; NULL means ascending order. */
int lpd_attn_merge_order_drift(const void *out_parts, int32_t parts_dtype, const float *lse_parts,
                               int32_t n_parts, int64_t n_rows, int32_t head_dim,
                               int32_t lse_base2, const int32_t *order_a, const int32_t *order_b,
                               float *out, float *out_lse, float *row_dout, float *row_dlse,
                               lpd_merge_drift *drift, void *stream);

/* ---- scoring without a caller-provided workspace -------------------------- */

/* Largest n_rows lpd_score_noalloc accepts: its built-in scratch is sized for
 * this many rows (about 25 MB of device memory per GPU that loads the
 * library, held until the process exits). */
#define LPD_NOALLOC_MAX_ROWS 32768

/* lpd_score without the workspace argument, for callers that cannot allocate
 * device memory (for example code running inside another engine whose caching
 * allocator owns the device, or a plugin host that hands out only a stream and
 * the tensors).  The pages have no counterpart to this entry point.
 *
 * Arguments, outputs and results are those of lpd_score; the workspace comes
 * from a fixed array inside the library.  Returns LPD_ERR_UNSUPPORTED when
 * n_rows > LPD_NOALLOC_MAX_ROWS, before touching the GPU.  It allocates
 * nothing.  The first call on each device (with that device current) looks up
 * the array's address, so make that first call before any stream capture on
 * the device; the address is cached per device context, so the first call
 * after a device reset looks it up again.  All calls on a device share the
 * array and it keeps the previous call's contents (nothing in it needs to
 * start at zero).  The library does not serialise callers: calls whose work
 * overlaps on the GPU race on the array, so the caller orders them (one
 * stream, or events between streams). */
int lpd_score_noalloc(const lpd_logits *train, const lpd_logits *rollout, int64_t n_rows,
                      int64_t vocab, const int32_t *token_ids, const uint8_t *action_mask,
                      double clip_lo, double clip_hi, float *out_logp_train,
                      float *out_logp_rollout, float *out_dlogp, lpd_metrics *out_metrics,
                      void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LPD_H */
