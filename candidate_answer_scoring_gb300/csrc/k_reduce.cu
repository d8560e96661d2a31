// Second half of the path: merge the head's per-split (max, sum-exp) partials
// into each row's log-sum-exp and the per-token log-probabilities, then the
// candidate-set rules.
#include <climits>

#include "jet_internal.cuh"
#include "jet_setrules.cuh"

namespace jet {
namespace {

// ---------------------------------------------------------------------------
// lse[r] = M + log sum_i s_i exp(m_i - M) over the 2*S partials of row r
// ("JET: Justification Evaluation in Transformer", Eq. 2).  One warp per row:
// lane l folds partials l, l+32, ... into a running (max, sum), then the
// lanes take the row's maximum and sum their rescaled sums, both in a fixed
// butterfly, so identical rows give bit-identical results.
// With sets, the row's lse goes to lse_row and the set kernel forms each
// token's logp = z - lse; without (one token per row), logp[r] is written here.
// ---------------------------------------------------------------------------

constexpr int MERGE_LOADS = 8;

__global__ void __launch_bounds__(256) merge_kernel(const MergeArgs a) {
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (r >= a.N) return;
  // the error word is read alongside the partials (every partial slot is in
  // bounds whatever the pre-pass found) and checked before anything is written
  const int err = *(volatile const int*)a.err;
  const Plan& P = a.plan;
  const int rows = plan_tile_rows(P);
  const int m_tile = r / rows, sub = (r - m_tile * rows) / BM, lr = r % BM;
  float m = -INFINITY, s = 0.f;
  const int n_slots = 2 * P.S;                        // (split, column half) pairs
  // rounds of MERGE_LOADS loads per lane, all issued before any is folded
  // (one L2 round trip per round: up to 256 partials per row in one)
  for (int base = 0; base < n_slots; base += 32 * MERGE_LOADS) {
    float2 p[MERGE_LOADS];
#pragma unroll
    for (int i = 0; i < MERGE_LOADS; ++i) {
      const int sl = base + lane + 32 * i;
      p[i] = sl < n_slots ? a.part[part_slot(P, plan_unit_of(P, m_tile, sl >> 1), sub, sl & 1, lr)]
                          : make_float2(-INFINITY, 0.f);
    }
    // the round's maximum first, then its terms scaled to it: independent
    // exponentials instead of a chain of pairwise folds
    float mr = m;
#pragma unroll
    for (int i = 0; i < MERGE_LOADS; ++i) mr = fmaxf(mr, p[i].x);
    if (mr != -INFINITY) {
      float acc = m == -INFINITY ? 0.f : s * expf(m - mr);
#pragma unroll
      for (int i = 0; i < MERGE_LOADS; ++i) acc += p[i].x == -INFINITY ? 0.f : p[i].y * expf(p[i].x - mr);
      s = acc;
      m = mr;
    }
  }
  // the row's maximum over the lanes, then the lanes' sums rescaled to it
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float S = m == -INFINITY ? 0.f : s * expf(m - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  if (err != 0 || lane != 0) return;
  const float lse = M + logf(S);
  if (a.lse) a.lse[r] = lse;
  if (a.lse_row) a.lse_row[r] = lse;
  else a.logp[r] = a.zg[r] - lse;
}

// One warp per set.  The set's index arrays are the caller's inputs, which
// nothing in this call writes and which the pre-pass has already validated
// (it completed before the head did, and the head completed before this grid
// was launched), so they are read while the merge still runs; only the
// gathered logits and row lse wait for it.  Sets of up to 32 single-token
// candidates take the whole chain that way (lane i = candidate i); others
// apply the chain rule after the wait.
__global__ void __launch_bounds__(256) sets_kernel(const SetArgs a) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const bool live = warp < a.n_sets && *(volatile const int*)a.err == 0;
  int c0 = 0, c1 = 0, t0 = 0, row = 0, tok = 0;
  bool single = false;
  if (live) {
    c0 = a.set_offsets[warp];
    c1 = a.set_offsets[warp + 1];
    if (c1 - c0 <= 32 && lane < c1 - c0) {
      t0 = a.cand_offsets[c0 + lane];
      single = a.cand_offsets[c0 + lane + 1] - t0 == 1;
      if (single) {
        row = a.tok_row[t0];
        tok = a.tok_ids[t0];
      }
    }
  }
  pdl_wait();
  pdl_trigger();   // the next call's first kernel may be scheduled; it waits for this grid
  if (!live || *(volatile const int*)a.err != 0) return;
  const int K = c1 - c0;
  if (K > 32) {
    set_rules_warp(a, warp, lane, c0, c1);
    return;
  }
  float sc[1] = {-INFINITY};
  unsigned long long h[1] = {0};
  if (lane < K) {
    if (single) {
      const float l = a.zg[t0] - a.lse_row[row];
      a.logp[t0] = l;
      sc[0] = 0.f + l;   // the chain rule over one token
      h[0] = single_token_hash(tok);
    } else {
      sc[0] = chain_sum(a, c0 + lane, h[0]);
    }
  }
  set_rules_core<1>(a, warp, lane, c0, K, 1.0f / a.T, sc, h);
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  return launch_dependent(merge_kernel, dim3((a.N + 7) / 8), dim3(256), 0, st, a);   // one warp per row
}

cudaError_t launch_sets(const SetArgs& a, cudaStream_t st) {
  if (a.n_sets <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  return launch_dependent(sets_kernel, dim3((a.n_sets + warps_per_block - 1) / warps_per_block),
                          dim3(32 * warps_per_block), 0, st, a);
}

}  // namespace jet
