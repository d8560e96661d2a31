// Candidate-set rules for one set, executed by one warp (shared by the set
// kernel of the full-vocabulary path and the fused restricted kernel).
#pragma once

#include <climits>

#include "jet_internal.cuh"

namespace jet {
namespace {

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
  const int a0 = co[a], b0 = co[b], la = co[a + 1] - a0;
  if (la != co[b + 1] - b0) return false;
  bool same = true;
  for (int t = 0; t < la; ++t) same &= (tok[a0 + t] == tok[b0 + t]);   // no early exit: loads overlap
  return same;
}

// Log-probability of scored token t: read as given, or (full-vocabulary path)
// formed from its gathered logit and its row's lse and stored.
__device__ __forceinline__ float token_logp(const SetArgs& a, int t) {
  if (a.zg == nullptr) return a.logp[t];
  const float l = a.zg[t] - a.lse_row[a.tok_row[t]];
  a.logp[t] = l;
  return l;
}

// s(c) and the FNV-1a hash of c's token sequence (length folded in first).
__device__ __forceinline__ float chain_sum(const SetArgs& a, int c, unsigned long long& h) {
  const int t0 = a.cand_offsets[c], t1 = a.cand_offsets[c + 1];
  h = 1469598103934665603ull ^ (unsigned long long)(t1 - t0);
  float acc = 0.f;
  int t = t0;
  for (; t + 4 <= t1; t += 4) {            // four independent loads in flight
    const float l0 = token_logp(a, t), l1 = token_logp(a, t + 1), l2 = token_logp(a, t + 2),
                l3 = token_logp(a, t + 3);
    const int k0 = a.tok_ids[t], k1 = a.tok_ids[t + 1], k2 = a.tok_ids[t + 2], k3 = a.tok_ids[t + 3];
    acc += l0; acc += l1; acc += l2; acc += l3;   // token order
    h = (h ^ (unsigned long long)(uint32_t)k0) * 1099511628211ull;
    h = (h ^ (unsigned long long)(uint32_t)k1) * 1099511628211ull;
    h = (h ^ (unsigned long long)(uint32_t)k2) * 1099511628211ull;
    h = (h ^ (unsigned long long)(uint32_t)k3) * 1099511628211ull;
  }
  for (; t < t1; ++t) {
    acc += token_logp(a, t);
    h = (h ^ (unsigned long long)(uint32_t)a.tok_ids[t]) * 1099511628211ull;
  }
  return acc;
}

// FNV-1a hash of a one-token sequence, as chain_sum forms it.
__device__ __forceinline__ unsigned long long single_token_hash(int tok) {
  return ((1469598103934665603ull ^ 1ull) ^ (unsigned long long)(uint32_t)tok) * 1099511628211ull;
}

// Set rules for K <= 32*CPL candidates held in registers: candidate i of the
// set lives in lane i % 32, slot i / 32, with its score sc and sequence hash h
// (sc = -inf, h = 0 for slots past K).
template <int CPL>
__device__ __forceinline__ void set_rules_core(const SetArgs& a, int set, int lane, int c0, int K, float invT,
                                               float (&sc)[CPL], unsigned long long (&h)[CPL]) {
  float q[CPL];
  float best = -INFINITY;
  int best_i = INT_MAX;
#pragma unroll
  for (int k = 0; k < CPL; ++k) {
    const int i = k * 32 + lane;
    if (i < K) {
      a.s[c0 + i] = sc[k];
      if (sc[k] > best) { best = sc[k]; best_i = i; }      // i grows with k: first maximum kept
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
    if (ob > best || (ob == best && oi < best_i)) { best = ob; best_i = oi; }
  }
  float z = 0.f;
#pragma unroll
  for (int k = 0; k < CPL; ++k) {
    q[k] = (k * 32 + lane < K) ? expf((sc[k] - best) * invT) : 0.f;
    z += q[k];
  }
  const float Z = warp_sum(z);
  float ex = 0.f, ent = 0.f;
#pragma unroll
  for (int k = 0; k < CPL; ++k) {
    q[k] /= Z;
    ex += (float)(k * 32 + lane) * q[k];
    if (q[k] > 0.f) ent -= q[k] * logf(q[k]);
  }
  ex = warp_sum(ex);
  ent = warp_sum(ent);
  float qe[CPL], mass_l = 0.f;
  bool first[CPL];
#pragma unroll
  for (int k = 0; k < CPL; ++k) { qe[k] = 0.f; first[k] = true; }
  for (int j = 0; j < K; ++j) {             // candidate j: lane j % 32, slot j / 32
    const int src = j & 31, slot = j >> 5;
    unsigned long long hj = 0;
    float qj = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      const unsigned long long hk = __shfl_sync(0xffffffffu, h[k], src);
      const float qk = __shfl_sync(0xffffffffu, q[k], src);
      if (k == slot) { hj = hk; qj = qk; }
    }
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      const int i = k * 32 + lane;
      // a candidate is its own class member; others are compared only on a hash match
      if (i < K && hj == h[k] && (j == i || same_sequence(a.tok_ids, a.cand_offsets, c0 + i, c0 + j))) {
        qe[k] += qj;
        if (j < i) first[k] = false;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < CPL; ++k) {
    const int i = k * 32 + lane;
    if (i < K) {
      a.q[c0 + i] = q[k];
      a.q_equiv[c0 + i] = qe[k];
      if (first[k]) mass_l += expf(sc[k]);
    }
  }
  const float mass = warp_sum(mass_l);
  if (lane == 0) {
    a.decision[set] = best_i;
    a.expected[set] = ex;
    a.confidence[set] = (K == 1) ? 1.0f : 1.0f - ent / logf((float)K);
    a.mass[set] = mass;
  }
}

// Set rules with s(c) and the hash formed by the chain rule (chain_sum).
template <int CPL>
__device__ __forceinline__ void set_rules_regs(const SetArgs& a, int set, int lane, int c0, int K, float invT) {
  float sc[CPL];
  unsigned long long h[CPL];
#pragma unroll
  for (int k = 0; k < CPL; ++k) {
    const int i = k * 32 + lane;
    sc[k] = -INFINITY;
    h[k] = 0;
    if (i < K) sc[k] = chain_sum(a, c0 + i, h[k]);
  }
  set_rules_core<CPL>(a, set, lane, c0, K, invT, sc, h);
}

// Set `set` (candidates [c0, c1)) by the calling warp: registers for
// K <= 128, else global passes.
__device__ void set_rules_warp(const SetArgs& a, int set, int lane, int c0, int c1) {
  const int K = c1 - c0;
  const float invT = 1.0f / a.T;
  const int warp = set;   // output index of the set

  if (K <= 32) { set_rules_regs<1>(a, warp, lane, c0, K, invT); return; }
  if (K <= 64) { set_rules_regs<2>(a, warp, lane, c0, K, invT); return; }
  if (K <= 128) { set_rules_regs<4>(a, warp, lane, c0, K, invT); return; }

  // larger sets: the same passes through global memory
  // pass 1: chain rule, sequence hash, first argmax
  float best = -INFINITY;
  int best_i = INT_MAX;
  for (int c = c0 + lane; c < c1; c += 32) {
    unsigned long long h;
    const float acc = chain_sum(a, c, h);
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
      if (a.hash[c2] == hc && (c2 == c || same_sequence(a.tok_ids, a.cand_offsets, c, c2))) {
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
}  // namespace jet
