/*
 * jetscore.h -- C ABI of libjetscore, the candidate-set scoring head on one
 * NVIDIA GB300 (sm_103a).
 *
 * What it computes (method: "JET: Justification Evaluation in Transformer";
 * contracts: Gemma/MLX architecture page, "Candidate likelihoods" and "Output
 * contracts"; restricted head: PARALLEL_SCORING page, "Execution" steps 5-6):
 *
 *   z[r, v]  = H[r, :] . W[v, :]                       logits of hidden row r
 *   lse[r]   = log sum_v exp z[r, v]                   full-vocabulary denominator (JET Eq. 1)
 *   l_j      = z[tok_row_j, tok_ids_j] - lse[tok_row_j]                        (JET Eq. 2)
 *   s(c)     = sum over the candidate's tokens of l    sequence log-likelihood  (JET Eq. 3)
 *   q(c)     = exp(s(c)/T) / sum_{c' in set} exp(s(c')/T)                       (JET Eq. 4)
 *   decision = first index of max s (fixed-order tie-break)                    (JET Eq. 5)
 *   expected = sum_i i q_i  (binary {false,true}: = q(true); ordinal: level mean)
 *   confidence = 1 - H(q)/ln K;  mass = sum of exp(s) at T=1 over distinct token
 *   sequences (allowed_token_mass);  q_equiv(c) = q summed over candidates with
 *   c's token sequence (labels with identical text).
 *
 * The [N, V] logit matrix is never written to memory: the projection, the
 * running max / sum-exp over vocabulary tiles and the gather of the supplied
 * token's logit happen in one kernel.
 *
 * Conventions shared by every call:
 *   - All array arguments are DEVICE pointers on the context's device, except
 *     in jet_score_sets_host, where they are HOST pointers.  The caller owns
 *     every input and output buffer; the library never frees or retains them.
 *   - H is bf16 row-major [n_rows, d]; W is bf16 row-major [V, d] (the output
 *     embedding / tied input embedding).  Both base addresses must be 16-byte
 *     aligned.  d must be a multiple of 64, 64 <= d <= 16384; 1 <= V < 2^31.
 *   - Index arrays are int32; kind is uint8; outputs are fp32 (decision int32).
 *   - Calls are stream-ordered on `cuda_stream` (a cudaStream_t, or NULL for
 *     the legacy default stream).  A context serves one stream at a time and
 *     is not thread-safe.
 *   - Return value: JET_OK or a negative status.  Host checks (sizes, T,
 *     mode, alignment) fail before anything is launched.  Index checks run in
 *     a device pre-pass that writes an error word; the synchronous calls wait
 *     for the stream once at the end and return that word.  On any error the
 *     outputs are unspecified.  Nothing in the library traps or asserts on the
 *     device; every device-side wait is bounded and reports JET_ERR_TIMEOUT.
 *
 * Diagnostic environment variables (read once per process; NOT part of the
 * ABI, for measuring and testing the library's own variants; every setting
 * gives results within the library's stated tolerances):
 *   JETSCORE_NO_PDL=1     launch every kernel with plain stream ordering
 *                         instead of programmatic dependent launch;
 *   JETSCORE_HEAD_PAIR=0|1 force the one-CTA (0) or the paired 2-SM (1)
 *                         full-vocabulary head for every batch size;
 *   JETSCORE_HEAD_DYN=0   paired head with several waves of units: take
 *                         units in a fixed stride order instead of from the
 *                         device counter;
 *   JETSCORE_RESTRICTED_TC=0|1 restricted mode: the mma.sync union kernel
 *                         (0) or the tcgen05 head over the staged union (1)
 *                         for every union size (default: by union size).
 */
#ifndef JETSCORE_H
#define JETSCORE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct jet_ctx jet_ctx; /* opaque: device workspace + schedule cache */

enum {
  JET_OK = 0,
  JET_ERR_ARG = -1,          /* bad size, pointer, alignment, T, kind value, or context */
  JET_ERR_TOKEN_RANGE = -2,  /* a token id outside [0, V) or a row outside [0, n_rows) */
  JET_ERR_OFFSETS = -3,      /* CSR offsets not monotone / not covering, empty candidate
                                or set, binary set with K != 2, ordinal set with K < 2 */
  JET_ERR_MODE = -4,         /* mode not FULL/RESTRICTED, or restricted-mode candidate
                                longer than one token */
  JET_ERR_NOT_IN_UNION = -5, /* restricted mode: candidate token not in union_ids, or a
                                union id repeated */
  JET_ERR_WORKSPACE = -6,    /* n_rows / n_tok beyond the sizes given to jet_create */
  JET_ERR_UNSUPPORTED = -7,  /* device is not sm_103 (GB300) or lacks the features used */
  JET_ERR_CUDA = -8,         /* a CUDA runtime call failed */
  JET_ERR_TIMEOUT = -9       /* a bounded device-side wait gave up (kernel returned early) */
};

enum { JET_KIND_CHOICE = 0, JET_KIND_BINARY = 1, JET_KIND_ORDINAL = 2 };
enum { JET_MODE_FULL = 0, JET_MODE_RESTRICTED = 1 };

#define JET_MAX_UNION 4096 /* restricted mode: largest accepted union */

/*
 * jet_create: make a context on CUDA device `device` for an output embedding of
 * shape [V, d], and allocate its device workspace for up to `max_rows` hidden
 * rows and `max_tokens` scored tokens per call (candidates and sets are bounded
 * by max_tokens as every candidate has >= 1 token).  Also allocates device
 * staging buffers of that size for jet_score_sets_host, and one of
 * min(V, JET_MAX_UNION) rows of W for restricted mode over large unions.
 * Errors: JET_ERR_ARG (sizes), JET_ERR_UNSUPPORTED (not sm_103), JET_ERR_CUDA.
 * On success *out owns the workspace until jet_destroy.
 */
int jet_create(jet_ctx **out, int d, int V, int max_rows, int max_tokens, int device);

/*
 * Tiled weights.  The head streams W in 128-row x 64-column boxes; stored
 * row-major each box is 128 pieces of 128 bytes, 2*d bytes apart.  A tiled copy
 * puts every box in 16 contiguous KB: element (v, k) of W sits at
 *   ((floor(v/128) * (d/64) + floor(k/64)) * 128 + v mod 128) * 64 + k mod 64
 * of a [ceil(V/128) * 128, d] bf16 array (rows past V are zero).  Results are
 * bit-identical to the row-major layout; the head reads it slightly faster.
 *
 * jet_tiled_weights_bytes: size of the tiled copy.
 * jet_tile_weights: write the tiled copy of W (device, row-major [V, d]) to
 *   W_tiled (device, jet_tiled_weights_bytes bytes, 16-byte aligned, not
 *   overlapping W).  Enqueued on `cuda_stream`; returns after enqueueing.
 * jet_set_weights_layout: how this context's later calls read their W
 *   argument: JET_W_ROWMAJOR (default) or JET_W_TILED (a jet_tile_weights copy).
 *   jet_score_tokens_noalloc always reads row-major W.
 * Errors: JET_ERR_ARG (NULL, alignment, overlap, unknown layout), JET_ERR_CUDA.
 */
enum { JET_W_ROWMAJOR = 0, JET_W_TILED = 1 };
size_t jet_tiled_weights_bytes(const jet_ctx *ctx);
int jet_tile_weights(jet_ctx *ctx, const void *W_bf16, void *W_tiled_bf16, void *cuda_stream);
int jet_set_weights_layout(jet_ctx *ctx, int layout);

/* Free the context and its workspace (waits for the device).  NULL is a no-op. */
void jet_destroy(jet_ctx *ctx);

/* Static, human-readable text for a status code. */
const char *jet_status_string(int status);

/*
 * jet_score_tokens: one scored token per hidden row (JET Eq. 1-2, the
 * per-position log-probability of a supplied token under teacher forcing):
 *   logp[i] = z[i, tok_ids[i]] - lse[i],   0 <= i < n_pos.
 * H [n_pos, d] bf16; W [V, d] bf16; tok_ids [n_pos] int32.
 * logp [n_pos] fp32 (required); lse [n_pos] fp32 or NULL.
 * n_pos == 0 returns JET_OK without launching.  Synchronous.
 */
int jet_score_tokens(jet_ctx *ctx, const void *H_bf16, const void *W_bf16, const int32_t *tok_ids,
                     int n_pos, float *logp, float *lse, void *cuda_stream);

/* Caller-owned device output buffers of jet_score_sets; NULL = not wanted. */
typedef struct {
  float *logp;       /* [n_tok]  l_j (full vocabulary) or z - lse over the union (restricted) */
  float *lse;        /* [n_rows] per-row log-sum-exp over the normaliser set */
  float *s;          /* [n_cand] sequence log-likelihood s(c) */
  float *q;          /* [n_cand] q(c) = softmax over the set of s/T */
  float *q_equiv;    /* [n_cand] q summed over candidates with an identical token sequence */
  int32_t *decision; /* [n_sets] index within the set of the first maximum of s */
  float *expected;   /* [n_sets] sum_i i q_i (binary sets: q(true)) */
  float *confidence; /* [n_sets] 1 - H(q)/ln K (K = 1: 1) */
  float *mass;       /* [n_sets] sum of exp(s) at T = 1 over distinct token sequences */
} jet_set_out;

/*
 * jet_score_sets: the whole scoring head for a batch of candidate sets.
 * Layout (CSR):
 *   H [n_rows, d] bf16 -- final hidden state at each teacher-forced position
 *       (JET, candidate evaluation under teacher forcing; Gemma/MLX page: one
 *       vocabulary vector per field for single-token candidates, one row per
 *       predicted token for multi-token candidates).  A row may serve several
 *       tokens.
 *   tok_row[n_tok], tok_ids[n_tok] -- for scored token j, the row predicting it
 *       and its id; a candidate's tokens are contiguous and in order.
 *   cand_offsets[n_cand+1] -- tokens of candidate c are [cand_offsets[c],
 *       cand_offsets[c+1]); cand_offsets[0] = 0, cand_offsets[n_cand] = n_tok.
 *   set_offsets[n_sets+1] -- candidates of set k, same convention over n_cand.
 *   kind[n_sets] -- JET_KIND_*: binary sets have K = 2 in order {false, true};
 *       ordinal sets K >= 2 levels in order; choice sets K >= 1.
 *   T > 0, finite -- temperature applied once to s before the set softmax
 *       (PARALLEL_SCORING page, "V2 probability default"); l, s, decision and
 *       mass do not depend on it.
 *   mode -- JET_MODE_FULL: normalise over the full vocabulary.
 *       JET_MODE_RESTRICTED: normalise over union_ids[n_union] (distinct ids,
 *       1 <= n_union <= JET_MAX_UNION); every candidate is one token of the
 *       union (PARALLEL_SCORING page, "Execution" step 5).  union_ids is ignored
 *       in full mode.  Unions of fewer than 192 codes are projected by a small
 *       tensor-core kernel (mma.sync); larger ones are copied into the
 *       context's staging rows and projected by the full-vocabulary tcgen05
 *       head with the union as its vocabulary (JETSCORE_RESTRICTED_TC=0|1
 *       forces either, for diagnostics).
 * out -- host struct of device pointers; any member may be NULL.
 * Empty batches (n_tok == 0 with n_cand == n_sets == 0) return JET_OK.
 * Synchronous: waits for `cuda_stream` once, then returns the device status.
 */
int jet_score_sets(jet_ctx *ctx, const void *H_bf16, const void *W_bf16, int n_rows,
                   const int32_t *tok_row, const int32_t *tok_ids, int n_tok,
                   const int32_t *cand_offsets, int n_cand, const int32_t *set_offsets,
                   const uint8_t *kind, int n_sets, float T, int mode, const int32_t *union_ids,
                   int n_union, const jet_set_out *out, void *cuda_stream);

/*
 * jet_score_sets_gather: jet_score_sets with the hidden rows read in place from
 * a larger source array, such as a right-padded backbone output [B * L, d]
 * whose scored rows sit at each sequence's answer (last valid) position
 * (Gemma/MLX architecture page, "Backbone and precision": right padding and
 * row-specific answer positions; PARALLEL_SCORING page, "Execution" step 4:
 * scores use each row's last valid position).  Row i of the problem is
 * H_src[row_index[i]].  Full mode copies the gathered rows once into the
 * context's staging buffer (one warp per row) and streams them from there
 * with tiled loads, as does restricted mode over unions on the tcgen05 head;
 * restricted mode over smaller unions reads them in place.
 *   H_src_bf16 [n_src_rows, d] bf16 (device, 16-byte aligned);
 *   row_index [n_rows] int32 (device), each in
 *   [0, n_src_rows); rows may repeat.  Every other argument is as in
 *   jet_score_sets, with n_rows the number of gathered rows and tok_row
 *   indexing them.
 * Errors: as jet_score_sets; a row_index outside [0, n_src_rows) gives
 * JET_ERR_TOKEN_RANGE.  Synchronous; jet_score_sets_gather_async returns
 * after enqueueing, like jet_score_sets_async (status via jet_sync_status).
 */
int jet_score_sets_gather(jet_ctx *ctx, const void *H_src_bf16, int n_src_rows, const int32_t *row_index,
                          int n_rows, const void *W_bf16, const int32_t *tok_row, const int32_t *tok_ids,
                          int n_tok, const int32_t *cand_offsets, int n_cand, const int32_t *set_offsets,
                          const uint8_t *kind, int n_sets, float T, int mode, const int32_t *union_ids,
                          int n_union, const jet_set_out *out, void *cuda_stream);
int jet_score_sets_gather_async(jet_ctx *ctx, const void *H_src_bf16, int n_src_rows, const int32_t *row_index,
                                int n_rows, const void *W_bf16, const int32_t *tok_row, const int32_t *tok_ids,
                                int n_tok, const int32_t *cand_offsets, int n_cand, const int32_t *set_offsets,
                                const uint8_t *kind, int n_sets, float T, int mode, const int32_t *union_ids,
                                int n_union, const jet_set_out *out, void *cuda_stream);

/*
 * jet_score_sets_async: as jet_score_sets but returns after enqueueing (host
 * checks only).  The device status of the last enqueued call is returned by
 * jet_sync_status, which waits for `cuda_stream`.  For benchmarking and
 * pipelining; results are valid once the stream has reached them.
 */
int jet_score_sets_async(jet_ctx *ctx, const void *H_bf16, const void *W_bf16, int n_rows,
                         const int32_t *tok_row, const int32_t *tok_ids, int n_tok,
                         const int32_t *cand_offsets, int n_cand, const int32_t *set_offsets,
                         const uint8_t *kind, int n_sets, float T, int mode,
                         const int32_t *union_ids, int n_union, const jet_set_out *out,
                         void *cuda_stream);
int jet_sync_status(jet_ctx *ctx, void *cuda_stream);

/*
 * jet_score_sets_host: end-to-end entry for callers holding HOST buffers.
 * W_bf16 is a DEVICE pointer (the output embedding stays resident, like any
 * model weight); every other array (H, the index arrays, union_ids, and the
 * members of *out_host) is a HOST pointer (pinned memory gives full copy
 * speed; pageable memory works).  The call copies the inputs into the
 * context's device staging buffers, runs jet_score_sets on them, copies the
 * requested outputs back and waits for `cuda_stream`.
 * Errors: as jet_score_sets.
 */
int jet_score_sets_host(jet_ctx *ctx, const void *H_bf16_host, const void *W_bf16_dev, int n_rows,
                        const int32_t *tok_row, const int32_t *tok_ids, int n_tok,
                        const int32_t *cand_offsets, int n_cand, const int32_t *set_offsets,
                        const uint8_t *kind, int n_sets, float T, int mode,
                        const int32_t *union_ids, int n_union, const jet_set_out *out_host,
                        void *cuda_stream);

/*
 * jet_score_sets_host_async / jet_host_wait: jet_score_sets_host for a stream
 * of batches, returning after enqueueing so that consecutive calls overlap:
 * each call copies its inputs into one of two device staging slots on the
 * context's own copy stream (the copy of batch k+1 runs while the kernels of
 * batch k run on `cuda_stream`), then enqueues the kernels and the copies of
 * the requested outputs (and of the call's status) back into the caller's
 * host buffers on `cuda_stream`.  Arguments as jet_score_sets_host, except:
 *   - every host buffer (H, the index arrays, union_ids, the members of
 *     *out_host) must be page-locked (cudaHostAlloc / cudaHostRegister);
 *   - inputs must stay unmodified, and outputs unread, until jet_host_wait
 *     returns; every call between two waits uses the same `cuda_stream`, and
 *     no other call uses the context until the wait (the slots are its
 *     staging buffers).
 * The first call allocates the second staging slot (max_rows x d bf16 plus
 * the index arrays) and creates the copy stream.  Host checks fail at once,
 * with nothing enqueued; device-side statuses are collected by the wait.
 * After 4096 calls without a wait, a call waits for the earlier ones first.
 * jet_host_wait: waits for `cuda_stream` and returns the first non-zero status
 * of the calls enqueued since the previous wait (JET_OK if none).
 */
int jet_score_sets_host_async(jet_ctx *ctx, const void *H_bf16_host, const void *W_bf16_dev, int n_rows,
                              const int32_t *tok_row, const int32_t *tok_ids, int n_tok,
                              const int32_t *cand_offsets, int n_cand, const int32_t *set_offsets,
                              const uint8_t *kind, int n_sets, float T, int mode,
                              const int32_t *union_ids, int n_union, const jet_set_out *out_host,
                              void *cuda_stream);
int jet_host_wait(jet_ctx *ctx, void *cuda_stream);

/*
 * jet_dedup_rows: project each distinct predictor state once -- the
 * candidate-preserving readout of FastJEV (section 3.3: project each required
 * predictor node once, normalise over the full vocabulary, gather the token
 * log-probabilities along each candidate path).  Finds bitwise-identical rows
 * of H (candidates sharing a token history carry identical hidden states) and
 * writes the distinct rows, in order of first occurrence, to H_unique; each
 * token's row is remapped so that scoring (H_unique, tok_row_unique) gives the
 * same results as scoring (H, tok_row).  Rows are compared by content (a
 * 64-bit hash, confirmed byte by byte), so different rows are never merged.
 *   H [n_rows, d] bf16 (device, 16-byte aligned); tok_row [n_tok] int32
 *     (n_tok may be 0: the rows are compacted and no token is remapped).
 *   H_unique [n_rows, d] bf16 (device, caller-owned, must not overlap H):
 *     rows 0 .. *n_unique-1 are written.
 *   tok_row_unique [n_tok] int32 (device): row of each token in H_unique.
 *   row_map [n_rows] int32 (device) or NULL: H_unique row of each input row.
 *   *n_unique (host): number of distinct rows.
 * Errors: JET_ERR_ARG (pointers, alignment, overlap, sizes), JET_ERR_WORKSPACE
 * (beyond jet_create's sizes), JET_ERR_TOKEN_RANGE (a tok_row outside
 * [0, n_rows)), JET_ERR_CUDA.  Synchronous.
 */
int jet_dedup_rows(jet_ctx *ctx, const void *H_bf16, int n_rows, const int32_t *tok_row, int n_tok,
                   void *H_unique_bf16, int32_t *tok_row_unique, int32_t *row_map, int *n_unique,
                   void *cuda_stream);

/*
 * jet_fit_temperature: fit the set-softmax temperature to labelled sets (the
 * calibration step of the Gemma/MLX architecture page, "Output contracts") by
 * minimising the mean gold negative log-likelihood
 *   NLL(T) = mean_k -log sum_{c in G_k} q_c(T),   q = softmax over the set of s/T,
 * where G_k holds the candidates of set k with the gold candidate's token
 * sequence (gold probability summed over labels with identical text, JET
 * Eq. 5 discussion).  NLL is convex in 1/T; the fit is a bracketed Newton
 * iteration on 1/T over [T_min, T_max] in one CTA.
 *   s [n_cand] fp32 (device): sequence log-likelihoods, e.g. jet_score_sets' s
 *   tok_ids [n_tok], cand_offsets [n_cand+1], set_offsets [n_sets+1]: as in
 *     jet_score_sets (device)
 *   gold [n_sets] int32 (device): index within each set of the gold candidate
 *   0 < T_min < T_max (finite)
 *   *T_out (host): fitted temperature (T_min or T_max when the optimum lies
 *     at the boundary); *nll_out (host) or NULL: mean NLL at *T_out
 * Errors: JET_ERR_ARG, JET_ERR_OFFSETS (offsets or a gold index out of
 * range), JET_ERR_WORKSPACE (n_tok beyond jet_create's max_tokens),
 * JET_ERR_CUDA.  Synchronous.
 */
int jet_fit_temperature(jet_ctx *ctx, const float *s, const int32_t *tok_ids, int n_tok,
                        const int32_t *cand_offsets, int n_cand, const int32_t *set_offsets, int n_sets,
                        const int32_t *gold, double T_min, double T_max, double *T_out, double *nll_out,
                        void *cuda_stream);

/*
 * jet_layer_sensitivity: decision-guided layer ranking ("FastJEV: Understanding
 * Redundancy for Compact JEV Inference", section 3.4, Eq. 5-6):
 *   d_l(x) = rms(ctr(z^(-l)(x) - z(x))) / max(1e-8, rms(ctr(z(x)))),
 *   J_l = mean over inputs x of d_l(x),  selected = the k layers with the
 *   smallest J_l, ties resolved by layer index,
 * with ctr(v) = v - mean(v) and rms(v) = ||v||_2 / sqrt(len v).
 *   z [total] fp32 (device): the decision logits of every calibration input,
 *     input x owning entries offsets[x] .. offsets[x+1]-1 (at least one)
 *   z_skip [L, total] fp32 (device): the same logits with layer l skipped
 *   offsets [n_inputs+1] int32 (device), offsets[0] = 0, offsets[n] = total
 *   d [L, n_inputs], J [L] fp32 (device, caller-owned); selected [k] int32
 *     (device; may be NULL when k == 0)
 * Errors: JET_ERR_ARG (sizes, k outside [0, L]), JET_ERR_OFFSETS.  Synchronous.
 */
int jet_layer_sensitivity(jet_ctx *ctx, const float *z, const float *z_skip, const int32_t *offsets,
                          int n_inputs, int total, int L, int k, float *d, float *J, int32_t *selected,
                          void *cuda_stream);

/*
 * jet_plan_info: the vocabulary-split schedule the full-vocabulary head uses
 * for `n_rows` rows (for reports and tests).  info[0..7] receive:
 *   row tiles, vocabulary tiles, splits per row tile, band height (row tiles
 *   whose units run together), units, CTAs launched, rows per tile, vocabulary
 *   columns per tile.
 * Returns JET_ERR_ARG for a NULL pointer or n_rows outside [1, max_rows].
 */
int jet_plan_info(jet_ctx *ctx, int n_rows, int *info8);

/*
 * Kernel timing.  jet_profile_enable(ctx, 1) makes the library record a CUDA
 * event pair on the launching stream around each of its kernel launches (no
 * extra synchronisation).  jet_profile_read waits for the recorded events and
 * writes, for kernel kind k in {0 pre-pass, 1 full-vocabulary head, 2 split
 * merge, 3 restricted head, 4 set rules}: out[2k] = launches, out[2k+1] =
 * total milliseconds; then clears the record.  n_out must be >= 10.  Up to
 * 65536 launches per kind are timed between reads; later ones are counted
 * only (out[2k] counts all, out[10] = launches that were not timed).
 */
int jet_profile_enable(jet_ctx *ctx, int enable);
int jet_profile_read(jet_ctx *ctx, double *out, int n_out);

/*
 * jet_selftest_wait_timeout: diagnostic of the library's failure handling.
 * Launches one CTA that waits, with the same bounded wait every kernel of the
 * library uses, on a barrier that nothing completes, giving up after
 * limit_us microseconds (1 .. 2,000,000).  Returns JET_ERR_TIMEOUT when the
 * wait ran out and reported itself through the context's error word as
 * designed (the expected result), JET_ERR_CUDA otherwise.  The context stays
 * usable afterwards.
 */
int jet_selftest_wait_timeout(jet_ctx *ctx, int limit_us, void *cuda_stream);

/*
 * jet_score_tokens_noalloc: the computation of jet_score_tokens (one scored
 * token per row, logp[i] = z[i, tok_ids[i]] - lse[i]) for callers that cannot
 * allocate device memory -- code running inside a process whose device memory
 * belongs to another framework's pool allocator (an inference server or a
 * plugin that reserves memory up front), where cudaMalloc may fail or stall
 * all streams with its implicit synchronisation mid-request.  It needs no
 * context and calls no allocating routine.  The pages describing the method
 * have no counterpart to this entry point.
 *
 * Arguments as jet_score_tokens, plus the embedding shape d, V (same limits as
 * jet_create); works on the CURRENT CUDA device.  Scratch lives in one static
 * device array of about 2.2 MB that every GPU loading the library keeps until
 * the process exits; it bounds a call to n_pos <= JET_NOALLOC_MAX_POS
 * (larger batches return JET_ERR_WORKSPACE).  All calls share that array:
 * calls whose GPU work overlaps (other streams or host threads) race on it.
 * The first call in each CUDA context on a device looks up the array's
 * device address (cudaGetSymbolAddress) and caches it for that context (a
 * context made after cudaDeviceReset looks it up again); make that first call
 * before any stream capture.  Synchronous; returns JET_OK or a status as
 * above.
 */
#define JET_NOALLOC_MAX_POS 4096
#define JET_NOALLOC_MAX_UNITS 1024
int jet_score_tokens_noalloc(const void *H_bf16, const void *W_bf16, int d, int V, const int32_t *tok_ids,
                             int n_pos, float *logp, float *lse, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* JETSCORE_H */
