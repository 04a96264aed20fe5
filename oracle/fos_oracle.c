/*
 * fos_oracle.c -- plain, slow FP64 CPU oracle for the fixed-order row softmax.
 *
 * TEST INFRASTRUCTURE ONLY.  The product library never links, includes or calls this file.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline / reference legs use
 * it.  It shares no header, helper or constant with the CUDA library.
 *
 * What it computes is the plain mathematical definition, in double precision, one row at a
 * time, keys in ascending order, with no tiling, blocking, fusion or reordering:
 *
 *   forward  ("[WS1][kernels] Add fixed-order joint-attention softmax for Qwen-Image",
 *             Summary: softmax of the QK scores along the key dimension; LSE as in
 *             "Batch-invariant attention (standard softmax--cuda version)", Implementation:
 *             masked softmax + LSE; sink as in "[ROCm] Jax Add softmax sink (learnable
 *             off-by-one) support", Description: one extra logit per head in the normaliser)
 *
 *       V    = valid keys of the row (mask definition below)
 *       M    = max({x_j : j in V} U {sink_h if a sink is given})
 *       Z    = sum_{j in V} exp(x_j - M)  +  [sink] exp(sink_h - M)
 *       LSE  = M + log Z,     P_j = exp(x_j - M) / Z  (j in V),   P_j = 0  (j not in V)
 *       A row with no valid key and no (finite) sink has P = 0 and LSE = -inf.
 *
 *   backward (same first page, "Fixed-order backward": the standard softmax VJP)
 *
 *       delta = sum_{j in V} P_j dP_j,     dS_j = P_j (dP_j - delta)  (j in V),  0 otherwise
 *
 *     applied to the P the caller passes in (the backward receives P; it does not recompute it).
 *
 *   sink gradient (third page above, the d_sink reduction; derivative of the row losses with
 *   respect to the per-head sink logit, dP_j/dsink = -P_j * P_sink, P_sink = exp(sink - LSE)):
 *
 *       d_sink[h] = - sum_{rows r of head h} exp(sink_h - LSE_r) * delta_r
 *
 * Mask definition (one definition for every step).  Rows are ordered [batch][heads][q_len];
 * row r has b = r / (heads*q_len), h = (r / q_len) % heads, i = r % q_len.  Key j (< L) of
 * row r is valid iff
 *   - causal:        j <= L - q_len + i   ("Batch-invariant attention", Prefill / Decode /
 *                                           KV-cache Contract: the causal condition)
 *   - kv_valid_len:  j <  kv_valid_len[b] (key padding, "Path Status": key_padding_mask)
 *   - key_mask:      key_mask[b*L + j] != 0
 *   - forward only:  x_j != -inf          (an input -inf acts as masked)
 * Every condition applies only when its input is given.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Row coordinates for the [batch][heads][q_len] row order. */
static void row_coords(int64_t r, int32_t heads, int32_t q_len, int64_t *b, int64_t *h,
                       int64_t *i) {
  *b = r / ((int64_t)heads * q_len);
  *h = (r / q_len) % heads;
  *i = r % q_len;
}

/* The mask definition above, without the forward-only -inf rule. */
static int key_valid(int64_t r, int64_t j, int32_t L, int32_t heads, int32_t q_len,
                     int32_t causal, const int32_t *kv_valid_len, const uint8_t *key_mask) {
  int64_t b, h, i;
  row_coords(r, heads, q_len, &b, &h, &i);
  if (causal && j > (int64_t)L - q_len + i) return 0;
  if (kv_valid_len && j >= (int64_t)kv_valid_len[b]) return 0;
  if (key_mask && key_mask[b * L + j] == 0) return 0;
  return 1;
}

static int check_common(int64_t n, int32_t L, int32_t batch, int32_t heads, int32_t q_len,
                        int32_t causal) {
  if (n < 0 || L < 1 || batch < 1 || heads < 1 || q_len < 1) return 1;
  if (causal && q_len > L) return 1;
  return 0;
}

static void set_threads(int32_t nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

/* Number of threads the parallel loops use (1 without OpenMP). */
int fos_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Forward.  scores/probs are n x L row-major doubles (the exact stored values, widened);
 * row k of the arrays is global row row_ids[k] (row k when row_ids is NULL), which fixes
 * b, h, i for the masks and the sink.  sink is [heads] or NULL.  Returns 0, or 1 on bad sizes.
 */
int fos_oracle_fwd(int64_t n, const int64_t *row_ids, int32_t L, int32_t batch, int32_t heads,
                   int32_t q_len, int32_t causal, const int32_t *kv_valid_len,
                   const uint8_t *key_mask, const double *sink, const double *scores,
                   double *probs, double *lse, int32_t nthreads) {
  if (check_common(n, L, batch, heads, q_len, causal)) return 1;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t k = 0; k < n; ++k) {
    const int64_t r = row_ids ? row_ids[k] : k;
    const double *x = scores + k * (int64_t)L;
    double *p = probs + k * (int64_t)L;
    int64_t b, h, i;
    row_coords(r, heads, q_len, &b, &h, &i);

    /* M: the largest logit taking part in the normaliser. */
    double M = -INFINITY;
    for (int64_t j = 0; j < L; ++j)
      if (key_valid(r, j, L, heads, q_len, causal, kv_valid_len, key_mask) && x[j] > M) M = x[j];
    if (sink && sink[h] > M) M = sink[h];

    if (M == -INFINITY) { /* nothing takes part: P = 0, LSE = -inf */
      for (int64_t j = 0; j < L; ++j) p[j] = 0.0;
      lse[k] = -INFINITY;
      continue;
    }

    /* Z: the normaliser, scaled by exp(-M). */
    double Z = 0.0;
    for (int64_t j = 0; j < L; ++j)
      if (key_valid(r, j, L, heads, q_len, causal, kv_valid_len, key_mask) && x[j] != -INFINITY)
        Z += exp(x[j] - M);
    if (sink) Z += exp(sink[h] - M);

    for (int64_t j = 0; j < L; ++j) {
      const int v = key_valid(r, j, L, heads, q_len, causal, kv_valid_len, key_mask) &&
                    x[j] != -INFINITY;
      p[j] = v ? exp(x[j] - M) / Z : 0.0;
    }
    lse[k] = M + log(Z);
  }
  return 0;
}

/*
 * Backward (softmax VJP applied to the given P).  probs/dprobs/dscores are n x L doubles;
 * delta is [n].  Row ids as in the forward.  Returns 0, or 1 on bad sizes.
 */
int fos_oracle_bwd(int64_t n, const int64_t *row_ids, int32_t L, int32_t batch, int32_t heads,
                   int32_t q_len, int32_t causal, const int32_t *kv_valid_len,
                   const uint8_t *key_mask, const double *probs, const double *dprobs,
                   double *dscores, double *delta, int32_t nthreads) {
  if (check_common(n, L, batch, heads, q_len, causal)) return 1;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t k = 0; k < n; ++k) {
    const int64_t r = row_ids ? row_ids[k] : k;
    const double *p = probs + k * (int64_t)L;
    const double *dp = dprobs + k * (int64_t)L;
    double *ds = dscores + k * (int64_t)L;

    double d = 0.0;
    for (int64_t j = 0; j < L; ++j)
      if (key_valid(r, j, L, heads, q_len, causal, kv_valid_len, key_mask)) d += p[j] * dp[j];

    for (int64_t j = 0; j < L; ++j)
      ds[j] = key_valid(r, j, L, heads, q_len, causal, kv_valid_len, key_mask)
                  ? p[j] * (dp[j] - d)
                  : 0.0;
    delta[k] = d;
  }
  return 0;
}

/*
 * Sink gradient.  lse and delta hold all rows = batch*heads*q_len, in row order; sink and
 * d_sink are [heads].  A head whose sink is -inf has no sink probability and gets 0.
 * Returns 0, or 1 on bad sizes.
 */
int fos_oracle_sink_grad(int32_t batch, int32_t heads, int32_t q_len, const double *sink,
                         const double *lse, const double *delta, double *d_sink) {
  if (batch < 1 || heads < 1 || q_len < 1) return 1;
  for (int32_t h = 0; h < heads; ++h) {
    double acc = 0.0;
    if (sink[h] != -INFINITY) {
      for (int64_t b = 0; b < batch; ++b)
        for (int64_t i = 0; i < q_len; ++i) {
          const int64_t r = (b * heads + h) * q_len + i;
          acc += exp(sink[h] - lse[r]) * delta[r];
        }
    }
    d_sink[h] = -acc;
  }
  return 0;
}
