// Internal declarations of libjetscore (GPU path).  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "jetscore.h"

namespace jet {

// ---- full-vocabulary head tile shape (tcgen05) ------------------------------
// One CTA owns 128 hidden rows (its TMEM lanes) and 256 vocabulary columns of
// a tile.  In the paired variant two CTAs of a cluster run one
// tcgen05.mma.cta_group::2 (M = 256): each stages its own 128 rows of H and
// half (128 rows) of the W tile.
constexpr int BM = 128;             // hidden rows per CTA tile = TMEM lanes
constexpr int BN = 256;             // vocabulary columns per tile = fp32 TMEM columns
constexpr int BK = 64;              // bf16 elements per k-block = one 128-byte swizzle row
constexpr int EPI_WARPS = 8;        // two warpgroups: column halves of a tile
constexpr int HEAD_THREADS = (2 + EPI_WARPS) * 32;
constexpr int TMEM_COLS = 2 * BN;   // two accumulators (double buffer)

template <bool PAIR>
struct HeadShape {
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;   // W rows this CTA stages per tile
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = PAIR ? 6 : 4;          // shared-memory ring depth (7 measured no faster)
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 512 /*barriers, unit ring*/;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// Device-side error word layout: err[0] = first status (0 = ok),
// err[1] = index of the offending element, err[2] = where a wait gave up.
constexpr int ERR_WORDS = 4;
// err[SCHED_WORD]: the head's unit counter when units are handed out
// dynamically; the pre-pass zeroes it together with the error words.
constexpr int SCHED_WORD = ERR_WORDS;

__device__ __forceinline__ void set_error(int* err, int code, int detail) {
  if (atomicCAS(err, 0, code) == 0) err[1] = detail;
}

// Programmatic dependent launch: kernels of one call are launched so that the
// next may be scheduled while the previous is still running.  A kernel calls
// pdl_wait() before it reads anything the previous kernel writes (including
// the error word); pdl_wait() returns at once when there is no dependency.
// pdl_trigger() lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Programmatic dependent launch is on unless the environment variable
// JETSCORE_NO_PDL is set (a diagnostic: launches then serialise normally).
bool pdl_enabled();

// Launch `kernel` on `st` as a programmatic dependent of the preceding kernel.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Vocabulary-split schedule of the head: unit u = (row tile m, split s) covers
// vocabulary tiles [s*n_vt/S, (s+1)*n_vt/S).  A row tile is 128 rows (one CTA)
// or, paired, 256 rows (a CTA pair).  Units are ordered band by band (Gm row
// tiles per band), split-major inside a band, so CTAs running together share
// W tiles through L2 while the band's H tiles stay L2-resident.
struct Plan {
  int n_mt = 0, n_vt = 0, S = 1, Gm = 1, n_full_bands = 0, r_last = 0, units = 0, grid = 0;
  int pair = 0;   // 1: units run on CTA pairs (cta_group::2)
};

__host__ __device__ __forceinline__ int plan_tile_rows(const Plan& p) { return p.pair ? 2 * BM : BM; }

// Slot of the (max, sum-exp) partial of (unit u, CTA sub of the pair, column
// half h, row lr of the CTA's 128).
__host__ __device__ __forceinline__ size_t part_slot(const Plan& p, int u, int sub, int h, int lr) {
  return (((size_t)u * (1 + p.pair) + sub) * 2 + h) * BM + lr;
}

struct HeadArgs {
  int N, V, d;
  Plan plan;
  const int* row_ptr;   // [N+1]   CSR over rows of the scored tokens
  const int2* row_list; // [n_tok] (token id, token index), sorted by id within a row
  float* zg;            // [n_tok] gathered logit of each scored token
  float2* part;         // per (unit, CTA of the pair, column half, row): (max, sum exp(z - max))
  int* err;
  int pf_kblocks;       // L2 prefetch distance for W, in k-blocks of the CTA's stream (0: off)
  int w_tiled = 0;      // tmW is the 4-D map of a tiled W (jet_tile_weights)
  int* sched = nullptr; // paired head, several waves of units: counter (zeroed by the pre-pass)
                        // from which pairs take units after their first; NULL: static stride
};

// Host: schedule for N rows on G SMs; units * (1 + pair) <= units_cap.
Plan make_plan(int N, int V, int d, int G, int units_cap, bool pair);
bool head_use_dynamic(const Plan& p);

// Host: whether the paired (2-SM) head serves N rows.
bool head_use_pair(int N);

// Host: L2 prefetch distance (k-blocks) for the head's W stream.  Off by
// default: measured on GB300 it slowed the W-streaming head (two CTAs share
// each W tile and both prefetch).  The environment variable
// JETSCORE_W_PREFETCH sets a distance for experiments.
int head_prefetch_kblocks(const Plan& p);

// Decode unit u of the plan into (row tile, first vocab tile, end vocab tile).
__host__ __device__ __forceinline__ void plan_unit(const Plan& p, int u, int& m, int& vt0, int& vt1) {
  const int main_units = p.n_full_bands * p.Gm * p.S;
  int split;
  if (u < main_units) {
    const int per_band = p.Gm * p.S;
    const int band = u / per_band, w = u - band * per_band;
    split = w / p.Gm;
    m = band * p.Gm + (w - split * p.Gm);
  } else {
    const int w = u - main_units;
    split = w / p.r_last;
    m = p.n_full_bands * p.Gm + (w - split * p.r_last);
  }
  vt0 = (int)((int64_t)split * p.n_vt / p.S);
  vt1 = (int)((int64_t)(split + 1) * p.n_vt / p.S);
}

// Unit index of (row tile m, split s): the inverse of plan_unit.
__host__ __device__ __forceinline__ int plan_unit_of(const Plan& p, int m, int split) {
  const int band = m / p.Gm;
  if (band < p.n_full_bands) return band * p.Gm * p.S + split * p.Gm + (m - band * p.Gm);
  return p.n_full_bands * p.Gm * p.S + split * p.r_last + (m - p.n_full_bands * p.Gm);
}

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
};
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st);

// Tiled copy of W (layout stated in jetscore.h, "Tiled weights").
cudaError_t launch_tile_weights(const uint16_t* W, int V, int d, uint16_t* W_tiled, cudaStream_t st);

// Copy rows src[row_index[i]] (i < n_rows) to dst[i]; indices outside
// [0, n_src) are skipped (the pre-pass reports them).  d % 8 == 0.
cudaError_t launch_gather_rows(const uint16_t* src, int n_src, const int32_t* row_index, int n_rows, int d,
                               uint16_t* dst, cudaStream_t st);

// tmW's box must have HeadShape<a.plan.pair>::B_ROWS rows; tmH's box BM rows.
cudaError_t launch_head(const CUtensorMap& tmH, const CUtensorMap& tmW, const HeadArgs& a,
                        cudaStream_t st);

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
