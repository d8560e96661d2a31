// Device pre-pass of the tcgen05 path: validates every index the rest of the
// path will use and builds, per hidden row, the list of scored tokens it
// predicts (sorted by the column each is gathered from: its token id, or in
// restricted mode over a staged union its union position, after the
// restricted checks), which the head's epilogue walks while it sweeps
// vocabulary tiles.
// Three layouts: one token per row (jet_score_tokens), tokens already grouped
// by row (tok_row non-decreasing: row pointers from run boundaries), and the
// general case (count, scan, scatter).
//
// One CTA of 1024 threads: the work is O(n_tok + n_rows + n_cand) integer
// operations, a few microseconds, and a single CTA needs no inter-CTA
// synchronisation.  Errors are reported through the error word (first error
// wins); nothing traps.
#include "jet_internal.cuh"

namespace jet {
namespace {

constexpr int PREP_THREADS = 1024;
constexpr int PREP_SMEM_ROWS = 6144;   // per-row counters in shared memory up to this many rows
constexpr int PREP_BATCH = 4;          // independent union lookups in flight per thread (restricted mode)

__device__ __forceinline__ int row_of(const PrepArgs& a, int j) {
  return a.tok_row ? a.tok_row[j] : j;
}

// The column token j is gathered from: its id, or in restricted mode its
// union position (read only after validation has passed).
__device__ __forceinline__ int list_key(const PrepArgs& a, int j) {
  return a.union_ids ? a.umap[a.tok_ids[j]] : a.tok_ids[j];
}

// Dynamic shared memory: [n_rows + 1] per-row counters when SMEM_COUNTS.
// Kept small so that the head kernel's CTA can share an SM with this one.
template <bool SMEM_COUNTS>
__global__ void __launch_bounds__(PREP_THREADS) prep_kernel(PrepArgs a) {
  extern __shared__ int s_cnt[];
  __shared__ int s_warp[PREP_THREADS / 32];
  __shared__ int s_unsorted;
  const int tid = threadIdx.x, nth = blockDim.x, lane = tid & 31, warp = tid >> 5;
  // Everything earlier on the stream has finished (and its writes are visible)
  // before this kernel touches memory, and before the head may start: the head
  // streams H and W as soon as it is scheduled and waits only for our outputs.
  pdl_wait();
  pdl_trigger();
  int* err = a.err;
  int* cnt = SMEM_COUNTS ? s_cnt : a.row_cur;
  const bool identity = a.tok_row == nullptr;    // token i is predicted by row i

  if (tid == 0) {
    for (int i = 0; i <= SCHED_WORD; ++i) err[i] = 0;   // error words and the head's unit counter
    s_unsorted = 0;
  }
  __syncthreads();

  // scored tokens: id in [0, V), row in [0, n_rows); is tok_row non-decreasing?
  for (int j = tid; j < a.n_tok; j += nth) {
    const int t = a.tok_ids[j], r = row_of(a, j);
    if (t < 0 || t >= a.V || r < 0 || r >= a.n_rows) set_error(err, JET_ERR_TOKEN_RANGE, j);
    if (!identity && j > 0 && a.tok_row[j - 1] > r) s_unsorted = 1;
  }
  if (a.union_ids) {
    // Restricted mode: each token's union position (a map entry is trusted
    // only where union_ids agrees, so entries left by earlier calls are
    // harmless), and the union ids in [0, V) and distinct (a repeated id
    // keeps one map position, so another of its positions does not map
    // back).  PREP_BATCH independent lookups in flight per thread.
    for (int j0 = tid; j0 < a.n_tok; j0 += nth * PREP_BATCH) {
      int t[PREP_BATCH], pos[PREP_BATCH];
#pragma unroll
      for (int i = 0; i < PREP_BATCH; ++i) {
        const int j = j0 + i * nth;
        t[i] = j < a.n_tok ? a.tok_ids[j] : -1;
      }
#pragma unroll
      for (int i = 0; i < PREP_BATCH; ++i) pos[i] = (t[i] >= 0 && t[i] < a.V) ? a.umap[t[i]] : -1;
#pragma unroll
      for (int i = 0; i < PREP_BATCH; ++i) {
        const int j = j0 + i * nth;
        if (t[i] < 0 || t[i] >= a.V) continue;          // out of range: reported above
        if (pos[i] < 0 || pos[i] >= a.n_union || a.union_ids[pos[i]] != t[i])
          set_error(err, JET_ERR_NOT_IN_UNION, j);
      }
    }
    for (int u0 = tid; u0 < a.n_union; u0 += nth * PREP_BATCH) {
      int t[PREP_BATCH], m[PREP_BATCH];
#pragma unroll
      for (int i = 0; i < PREP_BATCH; ++i) {
        const int u = u0 + i * nth;
        t[i] = u < a.n_union ? a.union_ids[u] : 0;
      }
#pragma unroll
      for (int i = 0; i < PREP_BATCH; ++i) m[i] = (t[i] >= 0 && t[i] < a.V) ? a.umap[t[i]] : -1;
#pragma unroll
      for (int i = 0; i < PREP_BATCH; ++i) {
        const int u = u0 + i * nth;
        if (u >= a.n_union) continue;
        if (t[i] < 0 || t[i] >= a.V) set_error(err, JET_ERR_TOKEN_RANGE, u);
        else if (m[i] != u) set_error(err, JET_ERR_NOT_IN_UNION, u);
      }
    }
  }

  // gathered rows: every index within the source array
  if (a.row_index)
    for (int i = tid; i < a.n_rows; i += nth) {
      const int idx = a.row_index[i];
      if (idx < 0 || idx >= a.n_src) set_error(err, JET_ERR_TOKEN_RANGE, i);
    }

  // candidate and set offsets (CSR), kind constraints
  if (a.cand_offsets) {
    if (tid == 0) {
      if (a.cand_offsets[0] != 0 || a.cand_offsets[a.n_cand] != a.n_tok) set_error(err, JET_ERR_OFFSETS, 0);
      if (a.set_offsets[0] != 0 || a.set_offsets[a.n_sets] != a.n_cand) set_error(err, JET_ERR_OFFSETS, 0);
    }
    for (int c = tid; c < a.n_cand; c += nth) {
      const int t0 = a.cand_offsets[c], t1 = a.cand_offsets[c + 1];
      if (!(t0 >= 0 && t0 < t1 && t1 <= a.n_tok)) set_error(err, JET_ERR_OFFSETS, c);
      else if (a.union_ids && t1 - t0 != 1) set_error(err, JET_ERR_MODE, c);   // restricted: one token each
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

  __syncthreads();
  if (*(volatile int*)err != 0) return;

  if (identity) {                                    // one token per row, in row order
    for (int i = tid; i < a.n_tok; i += nth) {
      a.row_ptr[i] = i;
      a.row_list[i] = make_int2(list_key(a, i), i);
    }
    if (tid == 0) a.row_ptr[a.n_rows] = a.n_tok;
    return;
  }

  if (!s_unsorted) {
    // tokens already grouped by row: row_ptr from the run boundaries of tok_row
    for (int j = tid; j < a.n_tok; j += nth) {
      const int r = a.tok_row[j];
      const int rp = (j == 0) ? -1 : a.tok_row[j - 1];
      for (int rr = rp + 1; rr <= r; ++rr) a.row_ptr[rr] = j;       // rows rp+1 .. r start at j
      if (j == a.n_tok - 1)
        for (int rr = r + 1; rr <= a.n_rows; ++rr) a.row_ptr[rr] = a.n_tok;
      a.row_list[j] = make_int2(list_key(a, j), j);
    }
    __syncthreads();
    for (int r = tid; r < a.n_rows; r += nth) {      // order each row's tokens by column
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
    return;
  }

  // general layout: count tokens per row
  for (int r = tid; r <= a.n_rows; r += nth) cnt[r] = 0;
  __syncthreads();
  for (int j = tid; j < a.n_tok; j += nth) atomicAdd(&cnt[a.tok_row[j]], 1);
  __syncthreads();

  // exclusive scan of the per-row counts -> row_ptr; the counters become cursors
  const int chunk = (a.n_rows + nth - 1) / nth;
  const int r0 = min(a.n_rows, tid * chunk), r1 = min(a.n_rows, r0 + chunk);
  int local = 0;
  for (int r = r0; r < r1; ++r) local += cnt[r];
  int incl = local;                                  // inclusive scan within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < nth / 32) ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    s_warp[lane] = w;                                // inclusive warp totals
  }
  __syncthreads();
  int run = incl - local + (warp > 0 ? s_warp[warp - 1] : 0);
  for (int r = r0; r < r1; ++r) {
    const int c = cnt[r];
    a.row_ptr[r] = run;
    cnt[r] = run;
    run += c;
  }
  if (tid == nth - 1) a.row_ptr[a.n_rows] = s_warp[nth / 32 - 1];
  __syncthreads();

  // scatter (token id, token index) into each row's slot range
  for (int j = tid; j < a.n_tok; j += nth) {
    const int pos = atomicAdd(&cnt[row_of(a, j)], 1);
    a.row_list[pos] = make_int2(list_key(a, j), j);
  }
  __syncthreads();

  // sort each row's list by (column, token index): rows hold few tokens
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

// Answer-position rows read in place from a larger source: one warp per row,
// 16-byte vectors, grid-stride.  The head then streams the compact copy with
// tiled TMA loads.  (Gathering inside the head's A-operand loads, four rows
// per TMA gather, was measured on GB300 at about four times the head's time:
// the A tile is fetched again for every vocabulary tile, and each 512-byte
// gather costs the TMA unit about as much as a 16 KB tile.)
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* src, int n_src, const int32_t* row_index,
                                                          int n_rows, int nvec, uint4* dst) {
  pdl_wait();      // earlier work on the stream is complete before any access
  pdl_trigger();   // the pre-pass may start; it waits for this grid before the head reads dst
  const int lane = threadIdx.x & 31;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < n_rows; r += (gridDim.x * blockDim.x) >> 5) {
    const int idx = row_index[r];
    if (idx < 0 || idx >= n_src) continue;
    const uint4* s = src + (size_t)idx * nvec;
    uint4* o = dst + (size_t)r * nvec;
    for (int k = lane; k < nvec; k += 32) o[k] = s[k];
  }
}

// Tiled copy of W: output vector o (8 bf16) of tile T, k-block kb, row r,
// vector j8 holds W[128 T + r][64 kb + 8 j8 .. +8], zero past row V.
__global__ void __launch_bounds__(256) tile_weights_kernel(const uint4* W, int V, int d, uint4* out,
                                                           long long n_vec) {
  const int kbs = d / 64;
  const int nvec_row = d / 8;
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < n_vec;
       o += (long long)gridDim.x * blockDim.x) {
    const int j8 = (int)(o & 7);
    const int r = (int)((o >> 3) & 127);
    const long long tk = o >> 10;               // tile * kbs + kb
    const int kb = (int)(tk % kbs);
    const long long row = (tk / kbs) * 128 + r;
    out[o] = row < V ? W[row * nvec_row + kb * 8 + j8] : make_uint4(0, 0, 0, 0);
  }
}

}  // namespace

cudaError_t launch_tile_weights(const uint16_t* W, int V, int d, uint16_t* W_tiled, cudaStream_t st) {
  const long long n_vec = (long long)((V + 127) / 128) * 128 * (d / 8);
  const long long want = (n_vec + 255) / 256;
  const int blocks = (int)(want < 4096 ? want : 4096);
  tile_weights_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(W), V, d,
                                              reinterpret_cast<uint4*>(W_tiled), n_vec);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const uint16_t* src, int n_src, const int32_t* row_index, int n_rows, int d,
                               uint16_t* dst, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  const int blocks = (n_rows + 7) / 8 < 1184 ? (n_rows + 7) / 8 : 1184;   // 8 rows per block, at most 8 per SM
  return launch_dependent(gather_rows_kernel, dim3(blocks), dim3(256), 0, st, reinterpret_cast<const uint4*>(src),
                          n_src, row_index, n_rows, d / 8, reinterpret_cast<uint4*>(dst));
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st) {
  if (a.tok_row != nullptr && a.n_rows + 1 <= PREP_SMEM_ROWS)
    return launch_dependent(prep_kernel<true>, dim3(1), dim3(PREP_THREADS), (a.n_rows + 1) * sizeof(int), st, a);
  return launch_dependent(prep_kernel<false>, dim3(1), dim3(PREP_THREADS), 0, st, a);
}

}  // namespace jet
