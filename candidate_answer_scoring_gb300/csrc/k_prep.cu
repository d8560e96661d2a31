// Device pre-pass: validates every index the rest of the path will use and
// builds, per hidden row, the list of scored tokens it predicts (sorted by
// token id), which the head's epilogue walks while it sweeps vocabulary tiles.
//
// One CTA of 1024 threads: the work is O(n_tok + n_rows + n_cand) integer
// operations, a few microseconds, and a single CTA needs no inter-CTA
// synchronisation.  Errors are reported through the error word (first error
// wins); nothing traps.
#include "jet_internal.cuh"

namespace jet {
namespace {

constexpr int PREP_THREADS = 1024;

__device__ __forceinline__ int row_of(const PrepArgs& a, int j) {
  return a.tok_row ? a.tok_row[j] : j;
}

__global__ void __launch_bounds__(PREP_THREADS) prep_kernel(PrepArgs a) {
  __shared__ int s_union[JET_MAX_UNION];
  __shared__ int s_scan[PREP_THREADS];
  const int tid = threadIdx.x, nth = blockDim.x;
  int* err = a.err;

  if (tid == 0) {
    for (int i = 0; i < ERR_WORDS; ++i) err[i] = 0;
  }
  for (int r = tid; r <= a.n_rows; r += nth) a.row_cur[r] = 0;
  __syncthreads();

  // scored tokens: id in [0, V), row in [0, n_rows); count tokens per row
  for (int j = tid; j < a.n_tok; j += nth) {
    const int t = a.tok_ids[j], r = row_of(a, j);
    if (t < 0 || t >= a.V || r < 0 || r >= a.n_rows) set_error(err, JET_ERR_TOKEN_RANGE, j);
    else atomicAdd(&a.row_cur[r], 1);
  }

  // candidate and set offsets (CSR), kind constraints
  if (a.cand_offsets) {
    if (tid == 0) {
      if (a.cand_offsets[0] != 0 || a.cand_offsets[a.n_cand] != a.n_tok)
        set_error(err, JET_ERR_OFFSETS, 0);
      if (a.set_offsets[0] != 0 || a.set_offsets[a.n_sets] != a.n_cand)
        set_error(err, JET_ERR_OFFSETS, 0);
    }
    for (int c = tid; c < a.n_cand; c += nth) {
      const int len = a.cand_offsets[c + 1] - a.cand_offsets[c];
      if (len < 1) set_error(err, JET_ERR_OFFSETS, c);
      else if (a.mode == JET_MODE_RESTRICTED && len != 1) set_error(err, JET_ERR_MODE, c);
    }
    for (int k = tid; k < a.n_sets; k += nth) {
      const int K = a.set_offsets[k + 1] - a.set_offsets[k];
      const int kd = a.kind[k];
      if (K < 1) set_error(err, JET_ERR_OFFSETS, k);
      else if (kd > JET_KIND_ORDINAL) set_error(err, JET_ERR_ARG, k);
      else if (kd == JET_KIND_BINARY && K != 2) set_error(err, JET_ERR_OFFSETS, k);
      else if (kd == JET_KIND_ORDINAL && K < 2) set_error(err, JET_ERR_OFFSETS, k);
    }
  }

  // restricted mode: union ids in range and distinct; every token in the union
  if (a.mode == JET_MODE_RESTRICTED) {
    for (int u = tid; u < a.n_union; u += nth) {
      const int t = a.union_ids[u];
      s_union[u] = t;
      if (t < 0 || t >= a.V) set_error(err, JET_ERR_TOKEN_RANGE, u);
    }
    __syncthreads();
    for (int u = tid; u < a.n_union; u += nth)
      for (int w = 0; w < u; ++w)
        if (s_union[w] == s_union[u]) set_error(err, JET_ERR_NOT_IN_UNION, u);
    for (int j = tid; j < a.n_tok; j += nth) {
      const int t = a.tok_ids[j];
      int pos = -1;
      for (int u = 0; u < a.n_union; ++u)
        if (s_union[u] == t) pos = u;
      if (pos < 0) set_error(err, JET_ERR_NOT_IN_UNION, j);
      a.upos[j] = pos;
    }
  }
  __syncthreads();
  if (*(volatile int*)err != 0) return;

  // exclusive scan of the per-row counts -> row_ptr; row_cur becomes the cursor
  const int chunk = (a.n_rows + nth - 1) / nth;
  const int r0 = min(a.n_rows, tid * chunk), r1 = min(a.n_rows, r0 + chunk);
  int local = 0;
  for (int r = r0; r < r1; ++r) local += a.row_cur[r];
  s_scan[tid] = local;
  __syncthreads();
  for (int off = 1; off < nth; off <<= 1) {        // Hillis-Steele inclusive scan
    const int v = (tid >= off) ? s_scan[tid - off] : 0;
    __syncthreads();
    s_scan[tid] += v;
    __syncthreads();
  }
  int run = s_scan[tid] - local;
  for (int r = r0; r < r1; ++r) {
    const int c = a.row_cur[r];
    a.row_ptr[r] = run;
    a.row_cur[r] = run;
    run += c;
  }
  if (tid == nth - 1) a.row_ptr[a.n_rows] = s_scan[nth - 1];
  __syncthreads();

  // scatter (token id, token index) into each row's slot range
  for (int j = tid; j < a.n_tok; j += nth) {
    const int r = row_of(a, j);
    const int pos = atomicAdd(&a.row_cur[r], 1);
    a.row_list[pos] = make_int2(a.tok_ids[j], j);
  }
  __syncthreads();

  // sort each row's list by (token id, token index): rows hold few tokens
  for (int r = tid; r < a.n_rows; r += nth) {
    const int b = a.row_ptr[r], e = a.row_ptr[r + 1];
    for (int i = b + 1; i < e; ++i) {
      const int2 x = a.row_list[i];
      int k = i - 1;
      while (k >= b && (a.row_list[k].x > x.x || (a.row_list[k].x == x.x && a.row_list[k].y > x.y))) {
        a.row_list[k + 1] = a.row_list[k];
        --k;
      }
      a.row_list[k + 1] = x;
    }
  }
}

}  // namespace

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st) {
  prep_kernel<<<1, PREP_THREADS, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace jet
