// Row deduplication: the candidate-preserving readout of "FastJEV:
// Understanding Redundancy for Compact JEV Inference", section 3.3 (project
// each required predictor node once, normalise over the full vocabulary, and
// gather the token log-probabilities along each candidate path).  With one
// hidden row per scored token, candidates that share a history carry
// bit-identical rows; this pass finds them and compacts the distinct rows so
// the head projects each one once.
//
//   1. hash    one warp per row: 64-bit hash of the row's bytes, fixed order
//   2. insert  open-addressing table hash -> smallest row index with that hash
//   3. resolve rep(r) = that smallest row if its bytes equal row r's (a hash
//              collision between different rows leaves r its own
//              representative: content is never merged)
//   4. scan    one CTA: rank of each representative in row order
//   5. emit    copy representatives to H_unique, row_map[r] = rank(rep(r)),
//              and tok_row_unique[j] = row_map[tok_row[j]]
// The result depends only on the rows' contents: representatives are first
// occurrences, ranks follow row order.
#include <algorithm>
#include <climits>

#include "jet_internal.cuh"

namespace jet {
namespace {

constexpr unsigned long long EMPTY_KEY = 0xFFFFFFFFFFFFFFFFull;

__device__ __forceinline__ unsigned long long mix64(unsigned long long x) {   // splitmix64 finaliser
  x ^= x >> 30;
  x *= 0xBF58476D1CE4E5B9ull;
  x ^= x >> 27;
  x *= 0x94D049BB133111EBull;
  x ^= x >> 31;
  return x;
}

__global__ void dedup_hash_kernel(const uint4* H, int n_rows, int nvec, unsigned long long* hash, int* err) {
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  if (blockIdx.x == 0 && threadIdx.x < ERR_WORDS) err[threadIdx.x] = 0;   // read after the last kernel
  if (r >= n_rows) return;
  const uint4* row = H + (size_t)r * nvec;
  unsigned long long h = 0x9E3779B97F4A7C15ull * (unsigned long long)(lane + 1);
  for (int k = lane; k < nvec; k += 32) {
    const uint4 v = row[k];
    h = mix64(h ^ (((unsigned long long)v.y << 32) | v.x));
    h = mix64(h ^ (((unsigned long long)v.w << 32) | v.z));
  }
  // combine the lanes in lane order
  unsigned long long acc = 0;
  for (int l = 0; l < 32; ++l) acc = mix64(acc ^ __shfl_sync(0xffffffffu, h, l));
  if (acc == EMPTY_KEY) acc ^= 1;    // reserve the empty marker
  if (lane == 0) hash[r] = acc;
}

__global__ void dedup_clear_kernel(unsigned long long* keys, int* vals, int table) {
  pdl_wait();
  pdl_trigger();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < table; i += gridDim.x * blockDim.x) {
    keys[i] = EMPTY_KEY;
    vals[i] = INT_MAX;
  }
}

__global__ void dedup_insert_kernel(const unsigned long long* hash, int n_rows, unsigned long long* keys,
                                    int* vals, int table_mask) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_rows) return;
  const unsigned long long h = hash[r];
  int slot = (int)(h & (unsigned long long)table_mask);
  for (int probe = 0; probe <= table_mask; ++probe) {      // the table has room for every row
    const unsigned long long prev = atomicCAS(&keys[slot], EMPTY_KEY, h);
    if (prev == EMPTY_KEY || prev == h) {
      atomicMin(&vals[slot], r);
      return;
    }
    slot = (slot + 1) & table_mask;
  }
}

__global__ void dedup_resolve_kernel(const uint4* H, int n_rows, int nvec, const unsigned long long* hash,
                                     const unsigned long long* keys, const int* vals, int table_mask, int* rep) {
  pdl_wait();
  pdl_trigger();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= n_rows) return;
  const unsigned long long h = hash[r];
  int slot = (int)(h & (unsigned long long)table_mask);
  int first = r;
  for (int probe = 0; probe <= table_mask; ++probe) {
    if (keys[slot] == h) { first = vals[slot]; break; }
    slot = (slot + 1) & table_mask;
  }
  if (first != r) {                     // same hash: confirm the bytes
    const uint4* a = H + (size_t)r * nvec;
    const uint4* b = H + (size_t)first * nvec;
    bool same = true;
    for (int k = lane; k < nvec; k += 32) {
      const uint4 x = a[k], y = b[k];
      same &= (x.x == y.x) & (x.y == y.y) & (x.z == y.z) & (x.w == y.w);
    }
    if (!__all_sync(0xffffffffu, same)) first = r;
  }
  if (lane == 0) rep[r] = first;
}

// One CTA: rank[r] = number of representatives before r; n_unique at rank[n_rows].
__global__ void __launch_bounds__(1024) dedup_scan_kernel(const int* rep, int n_rows, int* rank) {
  __shared__ int s_warp[32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, nth = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = (n_rows + nth - 1) / nth;
  const int r0 = min(n_rows, tid * chunk), r1 = min(n_rows, r0 + chunk);
  int local = 0;
  for (int r = r0; r < r1; ++r) local += (rep[r] == r);
  int incl = local;
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
    s_warp[lane] = w;
  }
  __syncthreads();
  int run = incl - local + (warp > 0 ? s_warp[warp - 1] : 0);
  for (int r = r0; r < r1; ++r) {
    rank[r] = run;
    run += (rep[r] == r);
  }
  if (tid == nth - 1) rank[n_rows] = s_warp[nth / 32 - 1];
}

__global__ void dedup_emit_kernel(const uint4* H, int n_rows, int nvec, const int* rep, const int* rank,
                                  uint4* H_unique, int32_t* row_map) {
  pdl_wait();
  pdl_trigger();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= n_rows) return;
  const int p = rep[r];
  if (lane == 0 && row_map) row_map[r] = rank[p];
  if (p == r) {
    const uint4* src = H + (size_t)r * nvec;
    uint4* dst = H_unique + (size_t)rank[r] * nvec;
    for (int k = lane; k < nvec; k += 32) dst[k] = src[k];
  }
}

__global__ void dedup_tokens_kernel(const int32_t* tok_row, int n_tok, const int* rep, const int* rank,
                                    int32_t* tok_row_unique, int n_rows, int* err) {
  pdl_wait();
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= n_tok) return;
  const int r = tok_row[j];
  if (r < 0 || r >= n_rows) {
    set_error(err, JET_ERR_TOKEN_RANGE, j);
    return;
  }
  tok_row_unique[j] = rank[rep[r]];
}

}  // namespace

cudaError_t launch_dedup(const DedupArgs& a, cudaStream_t st) {
  const int nvec = a.d / 8;
  const int warps_blocks = (a.n_rows + 7) / 8;   // 8 rows (warps) per 256-thread block
  const int table_mask = a.table - 1;
  dedup_hash_kernel<<<warps_blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(a.H), a.n_rows, nvec, a.hash,
                                                  a.err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_dependent(dedup_clear_kernel, dim3(std::min(1024, (a.table + 255) / 256)), dim3(256), 0, st, a.keys,
                       a.vals, a.table);
  if (e != cudaSuccess) return e;
  e = launch_dependent(dedup_insert_kernel, dim3((a.n_rows + 255) / 256), dim3(256), 0, st,
                       (const unsigned long long*)a.hash, a.n_rows, a.keys, a.vals, table_mask);
  if (e != cudaSuccess) return e;
  e = launch_dependent(dedup_resolve_kernel, dim3(warps_blocks), dim3(256), 0, st,
                       reinterpret_cast<const uint4*>(a.H), a.n_rows, nvec, (const unsigned long long*)a.hash,
                       (const unsigned long long*)a.keys, (const int*)a.vals, table_mask, a.rep);
  if (e != cudaSuccess) return e;
  e = launch_dependent(dedup_scan_kernel, dim3(1), dim3(1024), 0, st, (const int*)a.rep, a.n_rows, a.rank);
  if (e != cudaSuccess) return e;
  e = launch_dependent(dedup_emit_kernel, dim3(warps_blocks), dim3(256), 0, st,
                       reinterpret_cast<const uint4*>(a.H), a.n_rows, nvec, (const int*)a.rep, (const int*)a.rank,
                       reinterpret_cast<uint4*>(a.H_unique), a.row_map);
  if (e != cudaSuccess) return e;
  return launch_dependent(dedup_tokens_kernel, dim3((a.n_tok + 255) / 256), dim3(256), 0, st, a.tok_row, a.n_tok,
                          (const int*)a.rep, (const int*)a.rank, a.tok_row_unique, a.n_rows, a.err);
}

}  // namespace jet
