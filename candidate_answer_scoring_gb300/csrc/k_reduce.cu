// Second half of the path: merge the head's per-split (max, sum-exp) partials
// into each row's log-sum-exp and the per-token log-probabilities, then the
// candidate-set rules.
#include <climits>

#include "jet_internal.cuh"

namespace jet {
namespace {

// ---------------------------------------------------------------------------
// lse[r] = M + log sum_i s_i exp(m_i - M) over the 2*S partials of row r, in a
// fixed order (so identical rows give bit-identical results), then
// logp[j] = z[r, tok_j] - lse[r] for the row's tokens
// ("JET: Justification Evaluation in Transformer", Eq. 2).
// One thread per row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) merge_kernel(const MergeArgs a) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (*(volatile const int*)a.err != 0 || r >= a.N) return;
  const Plan& P = a.plan;
  const int m = r / BM, lr = r - m * BM;
  float M = -INFINITY;
  for (int sp = 0; sp < P.S; ++sp) {
    const size_t u = (size_t)plan_unit_of(P, m, sp);
    for (int h = 0; h < 2; ++h) M = fmaxf(M, a.part[(u * 2 + h) * BM + lr].x);
  }
  float sum = 0.f;
  for (int sp = 0; sp < P.S; ++sp) {
    const size_t u = (size_t)plan_unit_of(P, m, sp);
    for (int h = 0; h < 2; ++h) {
      const float2 p = a.part[(u * 2 + h) * BM + lr];
      if (p.x != -INFINITY) sum += p.y * expf(p.x - M);
    }
  }
  const float lse = M + logf(sum);
  if (a.lse) a.lse[r] = lse;
  for (int e = a.row_ptr[r]; e < a.row_ptr[r + 1]; ++e) {
    const int j = a.row_list[e].y;
    a.logp[j] = a.zg[j] - lse;
  }
}

// ---------------------------------------------------------------------------
// Candidate-set rules, one warp per set, candidates in supplied order:
//   s(c) = sum_t l_{c,t}                                    (JET Eq. 3)
//   q = softmax(s / T) over the set                         (JET Eq. 4; Gemma/MLX
//                                                            "Candidate likelihoods")
//   decision = first index of max s                         (JET Eq. 5)
//   expected = sum_i i q_i;  confidence = 1 - H(q)/ln K     (Gemma/MLX "Output contracts")
//   mass = sum over distinct token sequences of exp(s)      (allowed_token_mass, T = 1)
//   q_equiv(c) = q summed over candidates with c's sequence (labels with identical text)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ bool same_sequence(const int32_t* tok, const int32_t* co, int a, int b) {
  const int la = co[a + 1] - co[a], lb = co[b + 1] - co[b];
  if (la != lb) return false;
  for (int t = 0; t < la; ++t)
    if (tok[co[a] + t] != tok[co[b] + t]) return false;
  return true;
}

__global__ void __launch_bounds__(256) sets_kernel(const SetArgs a) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (*(volatile const int*)a.err != 0 || warp >= a.n_sets) return;
  const int c0 = a.set_offsets[warp], c1 = a.set_offsets[warp + 1], K = c1 - c0;
  const float invT = 1.0f / a.T;

  // pass 1: chain rule, sequence hash, first argmax
  float best = -INFINITY;
  int best_i = INT_MAX;
  for (int c = c0 + lane; c < c1; c += 32) {
    const int t0 = a.cand_offsets[c], t1 = a.cand_offsets[c + 1];
    float acc = 0.f;
    unsigned long long h = 1469598103934665603ull ^ (unsigned long long)(t1 - t0);
    for (int t = t0; t < t1; ++t) {
      acc += a.logp[t];
      h = (h ^ (unsigned long long)(uint32_t)a.tok_ids[t]) * 1099511628211ull;
    }
    a.s[c] = acc;
    a.hash[c] = h;
    if (acc > best || (acc == best && c < best_i)) { best = acc; best_i = c; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
    if (ob > best || (ob == best && oi < best_i)) { best = ob; best_i = oi; }
  }

  // pass 2: softmax denominator over s/T, shifted by the maximum
  float Z = 0.f;
  for (int c = c0 + lane; c < c1; c += 32) Z += expf((a.s[c] - best) * invT);
  Z = warp_sum(Z);

  // pass 3: q, expected index, entropy
  float ex = 0.f, ent = 0.f;
  for (int c = c0 + lane; c < c1; c += 32) {
    const float q = expf((a.s[c] - best) * invT) / Z;
    a.q[c] = q;
    ex += (float)(c - c0) * q;
    if (q > 0.f) ent -= q * logf(q);
  }
  ex = warp_sum(ex);
  ent = warp_sum(ent);
  __syncwarp();

  // pass 4: equivalence classes (identical token sequences)
  float mass = 0.f;
  for (int c = c0 + lane; c < c1; c += 32) {
    const unsigned long long hc = a.hash[c];
    float qe = 0.f;
    bool first = true;
    for (int c2 = c0; c2 < c1; ++c2) {
      if (a.hash[c2] == hc && same_sequence(a.tok_ids, a.cand_offsets, c, c2)) {
        qe += a.q[c2];
        if (c2 < c) first = false;
      }
    }
    a.q_equiv[c] = qe;
    if (first) mass += expf(a.s[c]);
  }
  mass = warp_sum(mass);

  if (lane == 0) {
    a.decision[warp] = best_i - c0;
    a.expected[warp] = ex;
    a.confidence[warp] = (K == 1) ? 1.0f : 1.0f - ent / logf((float)K);
    a.mass[warp] = mass;
  }
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  merge_kernel<<<(a.N + 255) / 256, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sets(const SetArgs& a, cudaStream_t st) {
  if (a.n_sets <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  sets_kernel<<<(a.n_sets + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace jet
