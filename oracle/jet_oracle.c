/*
 * jet_oracle.c -- plain fp64 CPU oracle of the candidate-set scoring head.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the test suite, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * It is deliberately slow and literal: every quantity is computed in double
 * precision straight from its definition, one row / one candidate / one set at
 * a time, with no blocking, fusion or reordering.  Inputs arrive as bf16 bit
 * patterns (the values the GPU sees) and are widened exactly to double.
 *
 * Sources (titles and sections of the pages the method is described on):
 *   [JET]  "JET: Justification Evaluation in Transformer"
 *          Eq. 1  candidate-token probability, full-vocabulary denominator,
 *                 teacher forcing, no temperature and no top-k/top-p;
 *          Eq. 2  its stable logarithm l = z_y - logsumexp_v z_v;
 *          Eq. 3  chain rule s(c) = sum_t l_{c,t} (no length normalisation,
 *                 no end-of-turn token, no sum over alternative phrasings);
 *          Eq. 4  q(c) = P(c) / sum_c' P(c'), worked example 0.06, 0.02 ->
 *                 0.75, 0.25; duplicating a candidate changes q;
 *          Eq. 5  argmax decision, ties broken by a fixed ordering; binary sets
 *                 {false, true} return q(true); ordinal sets return the expected
 *                 index sum_i i q(i); labels with identical text get identical
 *                 likelihoods and their probabilities are summed.
 *   [ARCH] Gemma/MLX "architecture.md", sections "Candidate likelihoods"
 *          (s(c), p(c) = exp(s/T) / sum exp(s/T), default T = 1) and "Output
 *          contracts" (confidence = one minus normalised entropy;
 *          allowed_token_mass = probability on allowed tokens, or summed
 *          complete candidate-sequence probabilities).
 *   [PAR]  "PARALLEL_SCORING.md", section "Execution" steps 5-6 (restricted
 *          head: project hidden states onto the gathered union of allowed code
 *          tokens, each field takes its subset, softmax(logits / T)) and
 *          "V2 probability default" (T scales candidate logits once, before the
 *          softmax; argmax does not change).
 *
 * Readings where the pages are silent (all stated in the design notes):
 *   - ties: the supplied candidate order, lowest index wins (decided on s,
 *     which is T-independent);
 *   - T scales only s before the set softmax: l, s, mass and decision do not
 *     depend on T; q, q_equiv, expected and confidence do;
 *   - allowed_token_mass = sum of exp(s) at T = 1 over DISTINCT token sequences;
 *   - confidence of a K = 1 set is 1; 0 * ln 0 = 0;
 *   - restricted mode replaces the vocabulary V by the union U in the
 *     denominator of Eq. 1; every candidate is one token of U.
 *
 * Parity pins: the test suite checks every function here against values the
 * pages print, closed forms, library routines and brute force.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_TOKEN (-2)
#define ORC_ERR_OFFSETS (-3)
#define ORC_ERR_UNION (-5)
#define ORC_ERR_NOMEM (-9)

int orc_version(void) { return 1; }
int orc_max_threads(void);

/* bf16 bit pattern -> double, exactly (bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* z_v = sum_k h_k * W[v, k]: the logit of token v for hidden row h ([JET] Eq. 1,
 * the logits z_{c,t,v}).  One dot product per vocabulary entry. */
static void row_logits(const double *h, const uint16_t *W, int64_t d, int64_t v_count,
                       const int32_t *v_ids, double *z) {
  for (int64_t i = 0; i < v_count; ++i) {
    const int64_t v = v_ids ? (int64_t)v_ids[i] : i;
    const uint16_t *w = W + v * d;
    double acc = 0.0;
    for (int64_t k = 0; k < d; ++k) acc += h[k] * bf16_to_double(w[k]);
    z[i] = acc;
  }
}

/* logsumexp_v z_v = M + log sum_v exp(z_v - M), M = max_v z_v ([JET] Eq. 2). */
static double logsumexp(const double *z, int64_t n) {
  double M = -INFINITY;
  for (int64_t i = 0; i < n; ++i)
    if (z[i] > M) M = z[i];
  double sum = 0.0;
  for (int64_t i = 0; i < n; ++i) sum += exp(z[i] - M);
  return M + log(sum);
}

/* l = z_tok - logsumexp(z) on a given logit vector ([JET] Eq. 2). */
int orc_log_softmax_at(const double *z, int64_t n, int64_t tok, double *out) {
  if (!z || !out || n <= 0 || tok < 0 || tok >= n) return ORC_ERR_ARG;
  *out = z[tok] - logsumexp(z, n);
  return ORC_OK;
}

/* Full logit vector of the listed rows (for tests; n_rows x V doubles). */
int orc_logits(const uint16_t *H, const uint16_t *W, int64_t N, int64_t d, int64_t V,
               const int64_t *rows, int64_t n_rows, double *z_out) {
  if (!H || !W || !rows || !z_out || d <= 0 || V <= 0) return ORC_ERR_ARG;
  double *h = (double *)malloc((size_t)d * sizeof(double));
  if (!h) return ORC_ERR_NOMEM;
  for (int64_t i = 0; i < n_rows; ++i) {
    if (rows[i] < 0 || rows[i] >= N) { free(h); return ORC_ERR_ARG; }
    for (int64_t k = 0; k < d; ++k) h[k] = bf16_to_double(H[rows[i] * d + k]);
    row_logits(h, W, d, V, NULL, z_out + i * V);
  }
  free(h);
  return ORC_OK;
}

/*
 * Per-token log-probabilities ([JET] Eq. 1-2).  For every wanted token j:
 *   l_j = z[tok_row_j, tok_ids_j] - lse[tok_row_j],
 *   lse_r = logsumexp over the normaliser set of z[r, .].
 * The normaliser set is the full vocabulary (union == NULL) or the union of
 * allowed code tokens ([PAR] Execution step 5); in the latter case each wanted
 * token must be a member of the union.
 *
 * want:   NULL = all tokens, else want[j] != 0 selects token j.
 * logp:   [n_tok]  written for wanted tokens, NAN elsewhere.
 * lse:    [N] or NULL, written for rows of wanted tokens, NAN elsewhere.
 */
static int score_tokens_impl(const uint16_t *H, const uint16_t *W, int64_t N, int64_t d, int64_t V,
                             const int32_t *union_ids, int64_t n_union,
                             const int32_t *tok_row, const int32_t *tok_ids, int64_t n_tok,
                             const uint8_t *want, double *logp, double *lse, int threads) {
  if (!H || !W || !tok_row || !tok_ids || !logp || d <= 0 || V <= 0 || N < 0 || n_tok < 0)
    return ORC_ERR_ARG;
  for (int64_t j = 0; j < n_tok; ++j) {
    logp[j] = NAN;
    if (want && !want[j]) continue;
    if (tok_row[j] < 0 || tok_row[j] >= N || tok_ids[j] < 0 || tok_ids[j] >= V) return ORC_ERR_TOKEN;
  }
  if (union_ids) {
    if (n_union <= 0) return ORC_ERR_ARG;
    for (int64_t u = 0; u < n_union; ++u) {
      if (union_ids[u] < 0 || union_ids[u] >= V) return ORC_ERR_TOKEN;
      for (int64_t w = 0; w < u; ++w)
        if (union_ids[w] == union_ids[u]) return ORC_ERR_UNION;
    }
    for (int64_t j = 0; j < n_tok; ++j) {
      if (want && !want[j]) continue;
      int found = 0;
      for (int64_t u = 0; u < n_union; ++u) found |= (union_ids[u] == tok_ids[j]);
      if (!found) return ORC_ERR_UNION;
    }
  }
  if (lse)
    for (int64_t r = 0; r < N; ++r) lse[r] = NAN;

  /* rows that some wanted token needs, and the tokens of each row (CSR) */
  int64_t *cnt = (int64_t *)calloc((size_t)N + 1, sizeof(int64_t));
  int64_t *idx = (int64_t *)malloc(((size_t)n_tok + 1) * sizeof(int64_t));
  if (!cnt || !idx) { free(cnt); free(idx); return ORC_ERR_NOMEM; }
  for (int64_t j = 0; j < n_tok; ++j)
    if (!want || want[j]) cnt[tok_row[j] + 1]++;
  for (int64_t r = 0; r < N; ++r) cnt[r + 1] += cnt[r];
  {
    int64_t *fill = (int64_t *)malloc(((size_t)N + 1) * sizeof(int64_t));
    if (!fill) { free(cnt); free(idx); return ORC_ERR_NOMEM; }
    memcpy(fill, cnt, ((size_t)N + 1) * sizeof(int64_t));
    for (int64_t j = 0; j < n_tok; ++j)
      if (!want || want[j]) idx[fill[tok_row[j]]++] = j;
    free(fill);
  }
  const int64_t n_norm = union_ids ? n_union : V;
  int err = ORC_OK;
  const int nt = threads > 0 ? threads : orc_max_threads();

#pragma omp parallel num_threads(nt)
  {
    double *h = (double *)malloc((size_t)d * sizeof(double));
    double *z = (double *)malloc((size_t)n_norm * sizeof(double));
    if (!h || !z) {
#pragma omp atomic write
      err = ORC_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < N; ++r) {
      if (!h || !z || cnt[r + 1] == cnt[r]) continue;
      for (int64_t k = 0; k < d; ++k) h[k] = bf16_to_double(H[r * d + k]);
      row_logits(h, W, d, n_norm, union_ids, z);
      const double lse_r = logsumexp(z, n_norm);
      if (lse) lse[r] = lse_r;
      for (int64_t e = cnt[r]; e < cnt[r + 1]; ++e) {
        const int64_t j = idx[e];
        int64_t pos = tok_ids[j];
        if (union_ids) {
          pos = -1;
          for (int64_t u = 0; u < n_union; ++u)
            if (union_ids[u] == tok_ids[j]) pos = u;
        }
        logp[j] = z[pos] - lse_r;
      }
    }
    free(h);
    free(z);
  }
  free(cnt);
  free(idx);
  return err;
}

int orc_score_tokens(const uint16_t *H, const uint16_t *W, int64_t N, int64_t d, int64_t V,
                     const int32_t *tok_row, const int32_t *tok_ids, int64_t n_tok,
                     const uint8_t *want, double *logp, double *lse, int threads) {
  return score_tokens_impl(H, W, N, d, V, NULL, 0, tok_row, tok_ids, n_tok, want, logp, lse, threads);
}

int orc_score_tokens_restricted(const uint16_t *H, const uint16_t *W, int64_t N, int64_t d, int64_t V,
                                const int32_t *union_ids, int64_t n_union,
                                const int32_t *tok_row, const int32_t *tok_ids, int64_t n_tok,
                                const uint8_t *want, double *logp, double *lse, int threads) {
  if (!union_ids) return ORC_ERR_ARG;
  return score_tokens_impl(H, W, N, d, V, union_ids, n_union, tok_row, tok_ids, n_tok, want, logp,
                           lse, threads);
}

/* Candidates a and b have identical token sequences (identical answer text,
 * [JET] Eq. 5 discussion of labels versus text). */
static int same_sequence(const int32_t *tok_ids, const int32_t *cand_offsets, int64_t a, int64_t b) {
  const int64_t la = cand_offsets[a + 1] - cand_offsets[a];
  const int64_t lb = cand_offsets[b + 1] - cand_offsets[b];
  if (la != lb) return 0;
  for (int64_t t = 0; t < la; ++t)
    if (tok_ids[cand_offsets[a] + t] != tok_ids[cand_offsets[b] + t]) return 0;
  return 1;
}

/*
 * Candidate-set rules, one set at a time, candidates in supplied order.
 *   s(c)        = sum of l over the candidate's tokens               [JET] Eq. 3
 *   a_i         = s_i / T
 *   q_i         = exp(a_i - max a) / sum_k exp(a_k - max a)          [JET] Eq. 4, [ARCH]
 *   decision    = smallest i with s_i = max s                        [JET] Eq. 5
 *   expected    = sum_i i q_i  (binary {false,true}: q(true))        [JET] Eq. 5
 *   confidence  = 1 - H(q) / ln K, H = -sum_{q_i>0} q_i ln q_i; K=1: 1   [ARCH]
 *   mass        = sum over distinct sequences of exp(s)  (T = 1)      [ARCH]
 *   q_equiv(c)  = sum of q over candidates with c's token sequence    [JET] Eq. 5
 *   margin      = q(decision) - max q over candidates whose sequence differs
 *                 from the winner's (INFINITY when there is none)
 * kind: 0 choice (K >= 1), 1 binary (K == 2), 2 ordinal (K >= 2).
 */
int orc_set_rules(const double *logp, const int32_t *tok_ids, int64_t n_tok,
                  const int32_t *cand_offsets, int64_t n_cand,
                  const int32_t *set_offsets, const uint8_t *kind, int64_t n_sets, double T,
                  double *s, double *q, double *q_equiv, int32_t *decision, double *expected,
                  double *confidence, double *mass, double *margin) {
  if (!logp || !tok_ids || !cand_offsets || !set_offsets || !kind || !s || !q || !q_equiv ||
      !decision || !expected || !confidence || !mass || !margin)
    return ORC_ERR_ARG;
  if (!(T > 0.0) || !isfinite(T)) return ORC_ERR_ARG;
  if (cand_offsets[0] != 0 || cand_offsets[n_cand] != n_tok) return ORC_ERR_OFFSETS;
  for (int64_t c = 0; c < n_cand; ++c)
    if (cand_offsets[c + 1] <= cand_offsets[c]) return ORC_ERR_OFFSETS;
  if (set_offsets[0] != 0 || set_offsets[n_sets] != n_cand) return ORC_ERR_OFFSETS;
  for (int64_t k = 0; k < n_sets; ++k) {
    const int64_t K = set_offsets[k + 1] - set_offsets[k];
    if (K < 1) return ORC_ERR_OFFSETS;
    if (kind[k] > 2) return ORC_ERR_ARG;
    if (kind[k] == 1 && K != 2) return ORC_ERR_OFFSETS;
    if (kind[k] == 2 && K < 2) return ORC_ERR_OFFSETS;
  }

  /* chain rule, token order */
  for (int64_t c = 0; c < n_cand; ++c) {
    double acc = 0.0;
    for (int64_t t = cand_offsets[c]; t < cand_offsets[c + 1]; ++t) acc += logp[t];
    s[c] = acc;
  }

  for (int64_t k = 0; k < n_sets; ++k) {
    const int64_t c0 = set_offsets[k], c1 = set_offsets[k + 1], K = c1 - c0;

    int64_t best = c0;
    for (int64_t c = c0 + 1; c < c1; ++c)
      if (s[c] > s[best]) best = c;          /* strict: the first maximum stays */
    decision[k] = (int32_t)(best - c0);

    const double amax = s[best] / T;
    double Z = 0.0;
    for (int64_t c = c0; c < c1; ++c) Z += exp(s[c] / T - amax);
    double ex = 0.0, ent = 0.0;
    for (int64_t c = c0; c < c1; ++c) {
      q[c] = exp(s[c] / T - amax) / Z;
      ex += (double)(c - c0) * q[c];
      if (q[c] > 0.0) ent -= q[c] * log(q[c]);
    }
    expected[k] = ex;
    confidence[k] = (K == 1) ? 1.0 : 1.0 - ent / log((double)K);

    double m = 0.0, other = -INFINITY;
    for (int64_t c = c0; c < c1; ++c) {
      double qe = 0.0;
      int first = 1;
      for (int64_t c2 = c0; c2 < c1; ++c2) {
        if (same_sequence(tok_ids, cand_offsets, c, c2)) {
          qe += q[c2];
          if (c2 < c) first = 0;
        }
      }
      q_equiv[c] = qe;
      if (first) m += exp(s[c]);
      if (!same_sequence(tok_ids, cand_offsets, c, best) && q[c] > other) other = q[c];
    }
    mass[k] = m;
    margin[k] = (other == -INFINITY) ? INFINITY : q[best] - other;
  }
  return ORC_OK;
}

/* Number of OpenMP threads a parallel region would use (for reporting). */
int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Whole path for one batch: per-token log-probabilities (full vocabulary, or
 * the union in restricted mode, where every candidate must be a single token),
 * then the set rules.  Outputs as in orc_score_tokens and orc_set_rules.
 */
int orc_score_sets(const uint16_t *H, const uint16_t *W, int64_t N, int64_t d, int64_t V,
                   const int32_t *tok_row, const int32_t *tok_ids, int64_t n_tok,
                   const int32_t *cand_offsets, int64_t n_cand,
                   const int32_t *set_offsets, const uint8_t *kind, int64_t n_sets,
                   double T, int mode, const int32_t *union_ids, int64_t n_union,
                   double *logp, double *lse, double *s, double *q, double *q_equiv,
                   int32_t *decision, double *expected, double *confidence, double *mass,
                   double *margin, int threads) {
  int rc;
  if (mode == 0) {
    rc = orc_score_tokens(H, W, N, d, V, tok_row, tok_ids, n_tok, NULL, logp, lse, threads);
  } else if (mode == 1) {
    if (!cand_offsets) return ORC_ERR_ARG;
    for (int64_t c = 0; c < n_cand; ++c)
      if (cand_offsets[c + 1] - cand_offsets[c] != 1) return ORC_ERR_OFFSETS;
    rc = orc_score_tokens_restricted(H, W, N, d, V, union_ids, n_union, tok_row, tok_ids, n_tok,
                                     NULL, logp, lse, threads);
  } else {
    return ORC_ERR_ARG;
  }
  if (rc != ORC_OK) return rc;
  return orc_set_rules(logp, tok_ids, n_tok, cand_offsets, n_cand, set_offsets, kind, n_sets, T, s,
                       q, q_equiv, decision, expected, confidence, mass, margin);
}
