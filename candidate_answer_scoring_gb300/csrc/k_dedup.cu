// Row deduplication: the candidate-preserving readout of "FastJEV:
// Understanding Redundancy for Compact JEV Inference", section 3.3 (project
// each required predictor node once, normalise over the full vocabulary, and
// gather the token log-probabilities along each candidate path).  With one
// hidden row per scored token, candidates that share a history carry
// bit-identical rows; this pass finds them and compacts the distinct rows so
// the head projects each one once.
//
//   1. hash    one warp per row: 64-bit hash of the row's bytes
//   2. insert  open-addressing table hash -> smallest row index with that hash
//   3. resolve rep(r) = that smallest row if its bytes equal row r's (a hash
//              collision between different rows leaves r its own
//              representative: content is never merged)
//   4. rank    rank of each representative in row order: tiles of 1024 rows,
//              one CTA each, offset by the representatives of earlier tiles
//              (counted per tile by the resolve pass)
//   5. emit    copy representatives to H_unique, row_map[r] = rank(rep(r)),
//              and tok_row_unique[j] = row_map[tok_row[j]]
// (the hash pass also empties the table; five launches in all)
// The result depends only on the rows' contents: representatives are first
// occurrences, ranks follow row order.
#include <algorithm>
#include <climits>

#include "jet_internal.cuh"

namespace jet {
namespace {

constexpr unsigned long long EMPTY_KEY = 0xFFFFFFFFFFFFFFFFull;
constexpr int HASH_BATCH = 8;      // 16-byte loads in flight per lane in the hash pass
constexpr int RANK_TILE = 1024;    // rows per CTA of the rank pass

__device__ __forceinline__ unsigned long long mix64(unsigned long long x) {   // splitmix64 finaliser
  x ^= x >> 30;
  x *= 0xBF58476D1CE4E5B9ull;
  x ^= x >> 27;
  x *= 0x94D049BB133111EBull;
  x ^= x >> 31;
  return x;
}

// Row hash: each lane runs two 32-bit multiply-rotate chains over its words
// (vectors lane, lane + 32, ... in order), finished with splitmix64; the
// lanes' values are seeded by lane index and combined by an xor tree.  Only
// equal rows must hash equal: a collision between different rows costs a byte
// comparison in the resolve pass, never a merge.
__device__ __forceinline__ uint32_t mr32(uint32_t h, uint32_t w, uint32_t mul) {
  const uint32_t x = h ^ w;
  return __funnelshift_l(x, x, 15) * mul;
}

// Also empties the hash table and the tile counts for the passes that follow
// (launched in plain stream order: earlier readers of them have finished).
__global__ void dedup_hash_kernel(const uint4* H, int n_rows, int nvec, unsigned long long* hash, int* err,
                                  unsigned long long* keys, int* vals, int table, int* tile_count, int n_tiles) {
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  if (blockIdx.x == 0 && threadIdx.x < ERR_WORDS) err[threadIdx.x] = 0;   // read after the last kernel
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < table; i += gridDim.x * blockDim.x) {
    keys[i] = EMPTY_KEY;
    vals[i] = INT_MAX;
    if (i < n_tiles) tile_count[i] = 0;
  }
  if (r >= n_rows) return;
  const uint4* row = H + (size_t)r * nvec;
  constexpr uint32_t M1 = 0x9E3779B1u, M2 = 0x85EBCA77u;   // odd multipliers
  uint32_t a = M1 * (uint32_t)(lane + 1), b = M2 * (uint32_t)(lane + 1);
  for (int k0 = lane; k0 < nvec; k0 += 32 * HASH_BATCH) {
    uint4 v[HASH_BATCH];
#pragma unroll
    for (int j = 0; j < HASH_BATCH; ++j)
      if (k0 + 32 * j < nvec) v[j] = __ldg(row + k0 + 32 * j);
#pragma unroll
    for (int j = 0; j < HASH_BATCH; ++j)
      if (k0 + 32 * j < nvec) {
        a = mr32(mr32(a, v[j].x, M1), v[j].z, M1);
        b = mr32(mr32(b, v[j].y, M2), v[j].w, M2);
      }
  }
  unsigned long long h = mix64(((unsigned long long)a << 32) | b);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) h ^= __shfl_xor_sync(0xffffffffu, h, o);
  h = mix64(h);
  if (h == EMPTY_KEY) h ^= 1;    // reserve the empty marker
  if (lane == 0) hash[r] = h;
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

// One row of the resolve pass (one warp): stores its representative; true
// when the row is its own.
__device__ __forceinline__ bool resolve_row(const uint4* H, int r, int lane, int nvec, const unsigned long long* hash,
                                            const unsigned long long* keys, const int* vals, int table_mask,
                                            int* rep) {
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
    bool same = true;   // (few rows get here: a plain loop keeps the probing warps' registers low)
    for (int k = lane; k < nvec; k += 32) {
      const uint4 x = a[k], y = b[k];
      same &= (x.x == y.x) & (x.y == y.y) & (x.z == y.z) & (x.w == y.w);
    }
    if (!__all_sync(0xffffffffu, same)) first = r;
  }
  if (lane == 0) rep[r] = first;
  return first == r;
}

// The block's representatives are counted in shared memory; the last of its
// warps to finish adds them to the rank tile's count (the block's rows lie in
// one tile), so a warp never waits for its block's slower warps.
__global__ void dedup_resolve_kernel(const uint4* H, int n_rows, int nvec, const unsigned long long* hash,
                                     const unsigned long long* keys, const int* vals, int table_mask, int* rep,
                                     int* tile_count) {
  __shared__ int s_reps, s_done;
  if (threadIdx.x == 0) { s_reps = 0; s_done = 0; }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  bool own = false;
  if (r < n_rows) own = resolve_row(H, r, lane, nvec, hash, keys, vals, table_mask, rep);
  if (lane == 0) {
    if (own) atomicAdd(&s_reps, 1);
    __threadfence_block();
    if (atomicAdd(&s_done, 1) == (int)(blockDim.x >> 5) - 1) {
      const int n = atomicAdd(&s_reps, 0);
      if (n > 0) atomicAdd(&tile_count[(blockIdx.x * (blockDim.x >> 5)) / RANK_TILE], n);
    }
  }
}


// rank[r] = number of representatives before row r (n_unique at rank[n_rows]).
// CTA b ranks rows [1024 b, 1024 b + 1024): the representatives of earlier
// tiles (summed from the resolve pass's tile counts) plus a block-wide scan.
__global__ void __launch_bounds__(RANK_TILE) dedup_rank_kernel(const int* rep, int n_rows, const int* tile_count,
                                                             int* rank) {
  __shared__ int s_warp[RANK_TILE / 32];
  __shared__ int s_base;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x * RANK_TILE + tid;
  const int f = (r < n_rows && rep[r] == r) ? 1 : 0;
  if (warp == 0) {   // representatives in the tiles before this one, summed in tile order
    int b = 0;
    for (int t = lane; t < (int)blockIdx.x; t += 32) b += tile_count[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) b += __shfl_xor_sync(0xffffffffu, b, o);
    if (lane == 0) s_base = b;
  }
  int incl = f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    s_warp[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  const int excl = s_base + (warp > 0 ? s_warp[warp - 1] : 0) + incl - f;
  if (r < n_rows) rank[r] = excl;
  if (blockIdx.x == gridDim.x - 1 && tid == RANK_TILE - 1) rank[n_rows] = s_base + s_warp[RANK_TILE / 32 - 1];
}

// Copies each representative to its rank, writes row_map, and maps every
// token's row (tok_row_unique[j] = rank of rep(tok_row[j])), threads striding
// over the tokens.
__global__ void dedup_emit_kernel(const uint4* H, int n_rows, int nvec, const int* rep, const int* rank,
                                  uint4* H_unique, int32_t* row_map, const int32_t* tok_row, int n_tok,
                                  int32_t* tok_row_unique, int* err) {
  pdl_wait();
  pdl_trigger();
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < n_tok; j += gridDim.x * blockDim.x) {
    const int r = tok_row[j];
    if (r < 0 || r >= n_rows) set_error(err, JET_ERR_TOKEN_RANGE, j);
    else tok_row_unique[j] = rank[rep[r]];
  }
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

}  // namespace

cudaError_t launch_dedup(const DedupArgs& a, cudaStream_t st) {
  const int nvec = a.d / 8;
  const int warps_blocks = (a.n_rows + 7) / 8;   // 8 rows (warps) per 256-thread block
  const int table_mask = a.table - 1;
  const int n_tiles = (a.n_rows + RANK_TILE - 1) / RANK_TILE;
  dedup_hash_kernel<<<warps_blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(a.H), a.n_rows, nvec, a.hash,
                                                  a.err, a.keys, a.vals, a.table, a.tile_count, n_tiles);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_dependent(dedup_insert_kernel, dim3((a.n_rows + 255) / 256), dim3(256), 0, st,
                       (const unsigned long long*)a.hash, a.n_rows, a.keys, a.vals, table_mask);
  if (e != cudaSuccess) return e;
  e = launch_dependent(dedup_resolve_kernel, dim3(warps_blocks), dim3(256), 0, st,
                       reinterpret_cast<const uint4*>(a.H), a.n_rows, nvec, (const unsigned long long*)a.hash,
                       (const unsigned long long*)a.keys, (const int*)a.vals, table_mask, a.rep, a.tile_count);
  if (e != cudaSuccess) return e;
  e = launch_dependent(dedup_rank_kernel, dim3(n_tiles), dim3(RANK_TILE), 0, st, (const int*)a.rep, a.n_rows,
                       (const int*)a.tile_count, a.rank);
  if (e != cudaSuccess) return e;
  return launch_dependent(dedup_emit_kernel, dim3(warps_blocks), dim3(256), 0, st,
                          reinterpret_cast<const uint4*>(a.H), a.n_rows, nvec, (const int*)a.rep,
                          (const int*)a.rank, reinterpret_cast<uint4*>(a.H_unique), a.row_map, a.tok_row, a.n_tok,
                          a.tok_row_unique, a.err);
}

}  // namespace jet
