// Internal declarations of libjetscore (GPU path) beyond the head's: the
// other kernels' arguments and launchers.  Not part of the C ABI.
#pragma once

#include "jet_head.cuh"

namespace jet {

// ---- launchers (each returns cudaGetLastError() of its launch) -------------
struct PrepArgs {
  int n_rows, n_tok, V;
  const int32_t* row_index = nullptr;   // gathered rows: each index must lie in [0, n_src); NULL: none
  int n_src = 0;
  const int32_t* tok_row;   // NULL: token i is predicted by row i
  const int32_t* tok_ids;
  const int32_t* cand_offsets; int n_cand;   // NULL when no sets (jet_score_tokens)
  const int32_t* set_offsets; const uint8_t* kind; int n_sets;
  int* row_ptr;    // [n_rows+1]
  int* row_cur;    // [n_rows+1] scratch counters
  int2* row_list;  // [n_tok]
  int* err;
  // restricted mode on the tensor-core head (launch_union_rows ran first):
  // the union is the vocabulary.  Adds the restricted checks (union ids in
  // range and distinct, one token per candidate, every token in the union)
  // and lists each token under its union position instead of its id.
  const int32_t* union_ids = nullptr;   // NULL: full vocabulary
  int n_union = 0;
  const int* umap = nullptr;            // [V] token id -> union position (launch_union_rows)
};
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st);

// Restricted mode on the tensor-core head: wU[u] = W[union_ids[u]] (row-major
// [n_union, d]; W row-major or tiled), and umap[union_ids[u]] = u.  Ids
// outside [0, V) give a zero row and no map entry (the pre-pass reports them).
cudaError_t launch_union_rows(const uint16_t* W, int V, int d, int w_tiled, const int32_t* union_ids, int n_union,
                              uint16_t* wU, int* umap, cudaStream_t st);

// Tiled copy of W (layout stated in jetscore.h, "Tiled weights").
cudaError_t launch_tile_weights(const uint16_t* W, int V, int d, uint16_t* W_tiled, cudaStream_t st);

// Copy rows src[row_index[i]] (i < n_rows) to dst[i]; indices outside
// [0, n_src) are skipped (the pre-pass reports them).  d % 8 == 0.
cudaError_t launch_gather_rows(const uint16_t* src, int n_src, const int32_t* row_index, int n_rows, int d,
                               uint16_t* dst, cudaStream_t st);

struct MergeArgs {
  int N = 0;
  Plan plan;
  const float2* part = nullptr;
  const float* zg = nullptr;
  float* lse = nullptr;       // [N] or NULL
  float* lse_row = nullptr;   // [N] per-row lse for the set kernel; NULL: token r of row r,
  float* logp = nullptr;      //     logp[r] = zg[r] - lse (one token per row)
  const int* err = nullptr;
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t st);

struct RestrictedArgs {
  int N, d, V, n_union, num_sms;
  const uint16_t* H; const uint16_t* W; const int32_t* union_ids;
  // NULL: row r is H[r]; else H[row_index[r]] with indices checked against
  // n_src (an index out of range is read as row 0 and reported by the set kernel)
  const int32_t* row_index = nullptr;
  int n_src = 0;
  int w_tiled = 0;  // W in the tiled layout (jet_tile_weights)
  float* zu;        // [N * n_union] logits over the union, or NULL (recomputed per token)
  float* lse_row;   // [N] log-sum-exp over the union
  float* lse;       // [N] caller's output or NULL
  int* umap;        // [V] union position of a token id (validated against union_ids)
  int* err;
};
cudaError_t launch_restricted(const RestrictedArgs& a, cudaStream_t st);

struct SetArgs {
  int n_sets;
  float* logp; const int32_t* tok_ids; const int32_t* cand_offsets;
  const int32_t* set_offsets; float T;
  float* s; float* q; float* q_equiv; int32_t* decision; float* expected;
  float* confidence; float* mass;
  unsigned long long* hash;   // [n_cand] scratch
  // full-vocabulary path: logp[t] = zg[t] - lse_row[tok_row[t]] is formed (and
  // stored) while the chain rule runs; NULL zg: logp is read as given
  const float* zg; const float* lse_row; const int32_t* tok_row;
  const int* err;
};
cudaError_t launch_sets(const SetArgs& a, cudaStream_t st);

// Validation, union lookup and set rules of the restricted path (after
// launch_restricted); n_cand, n_tok, r.N and r.V bound every index it follows.
struct RestrictedSetArgs {
  SetArgs s;
  RestrictedArgs r;
  int n_cand, n_tok;
  const int32_t* tok_row; const uint8_t* kind;
};
cudaError_t launch_restricted_sets(const RestrictedSetArgs& a, cudaStream_t st);

struct DedupArgs {
  int n_rows, d, n_tok;
  const uint16_t* H; const int32_t* tok_row;
  uint16_t* H_unique; int32_t* tok_row_unique; int32_t* row_map;   // row_map may be NULL
  unsigned long long* hash;   // [n_rows]
  unsigned long long* keys;   // [table]
  int* vals;                  // [table]
  int table;                  // power of two >= 2 * n_rows
  int* rep;                   // [n_rows]
  int* rank;                  // [n_rows + 1]; rank[n_rows] = distinct rows
  int* tile_count;            // [ceil(n_rows / 1024)] representatives per 1024-row tile
  int* err;
};
cudaError_t launch_dedup(const DedupArgs& a, cudaStream_t st);

struct FitArgs {
  int n_sets, n_cand, n_tok;
  const float* s; const int32_t* tok_ids; const int32_t* cand_offsets; const int32_t* set_offsets;
  const int32_t* gold;        // [n_sets] index within the set of the gold candidate
  double T_min, T_max;
  uint8_t* flags;             // [n_cand] scratch: member of its set's gold class
  double* result;             // [3]: T, mean NLL at T, iterations
  int* err;
};
cudaError_t launch_fit_temperature(const FitArgs& a, cudaStream_t st);

struct SensArgs {
  int n_inputs, L, total, k;
  const float* z;             // [total] logits of every input, CSR by offsets
  const float* z_skip;        // [L][total] the same with layer l skipped
  const int32_t* offsets;     // [n_inputs + 1]
  float* d;                   // [L][n_inputs]
  float* J;                   // [L]
  int32_t* selected;          // [k]
  int* err;
};
cudaError_t launch_sensitivity(const SensArgs& a, cudaStream_t st);

// One CTA waits on an mbarrier that nothing completes, with a limit of
// limit_ns; the bounded wait records JET_ERR_TIMEOUT (where = 99) in err.
cudaError_t launch_wait_selftest(int* err, unsigned long long limit_ns, cudaStream_t st);

}  // namespace jet
