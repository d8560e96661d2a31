// Temperature fitting on labelled candidate sets (the calibration step of the
// Gemma/MLX architecture page, "Output contracts").  With beta = 1/T:
//
//   loss_k(beta) = LSE_c(beta s_c) - LSE_{c in G_k}(beta s_c)       (-log q(gold class))
//   NLL(beta)    = mean_k loss_k
//   d/dbeta      = E_q[s] - E_{q|G}[s]
//   d2/dbeta2    = Var_q[s] - Var_{q|G}[s]
//
// where G_k holds the candidates of set k whose token sequence equals the gold
// one's (the gold probability is summed over labels with identical text:
// "JET: Justification Evaluation in Transformer", Eq. 5 discussion).  Equal
// texts have equal scores, so Var_{q|G} = 0 and NLL is convex in beta.
//
// One CTA of 1024 threads: each thread evaluates (loss, gradient, curvature)
// of sets t, t+1024, ... in fp32 (fp64 arithmetic is slow on this part, so it
// is kept to the sums over sets), warps combine in a fixed butterfly, thread 0
// combines the warps (warp 0, fixed butterfly) and takes a Newton step on
// beta, kept inside a shrinking bracket [lo, hi] that bisection falls back
// to; iterate until the step or the bracket is below FT_REL_TOL of beta.  The
// per-set terms carry fp32 rounding, so the gradient summed over sets is
// known to about 1e-5 absolute against a curvature summed over the same sets:
// steps below ~1e-8 relative are noise, and a tighter tolerance only walks
// the bracket in by noise-sized steps.  Deterministic.
#include "jet_internal.cuh"

namespace jet {
namespace {

constexpr int FT_THREADS = 1024;
constexpr int FT_WARPS = FT_THREADS / 32;
static_assert(FT_WARPS == 32, "the warp partials are combined by one warp");
constexpr int FT_MAX_IT = 200;
constexpr double FT_REL_TOL = 1e-7;

__device__ __forceinline__ float wmax(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float wsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ bool same_seq(const int32_t* tok, const int32_t* co, int a, int b) {
  const int a0 = co[a], b0 = co[b], la = co[a + 1] - a0;
  if (la != co[b + 1] - b0) return false;
  bool same = true;
  for (int t = 0; t < la; ++t) same &= (tok[a0 + t] == tok[b0 + t]);
  return same;
}

__global__ void __launch_bounds__(FT_THREADS) fit_temperature_kernel(const FitArgs a) {
  __shared__ double s_part[FT_WARPS][3];
  __shared__ double s_beta;
  __shared__ int s_done;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* err = a.err;
  if (tid == 0)
    for (int i = 0; i < ERR_WORDS; ++i) err[i] = 0;
  __syncthreads();

  // validation and the gold class of every set
  if (tid == 0) {
    if (a.set_offsets[0] != 0 || a.set_offsets[a.n_sets] != a.n_cand) set_error(err, JET_ERR_OFFSETS, 0);
    if (a.cand_offsets[0] != 0 || a.cand_offsets[a.n_cand] != a.n_tok) set_error(err, JET_ERR_OFFSETS, 0);
  }
  for (int c = tid; c < a.n_cand; c += FT_THREADS)
    if (a.cand_offsets[c + 1] <= a.cand_offsets[c]) set_error(err, JET_ERR_OFFSETS, c);
  for (int k = tid; k < a.n_sets; k += FT_THREADS) {
    const int K = a.set_offsets[k + 1] - a.set_offsets[k];
    if (K < 1) set_error(err, JET_ERR_OFFSETS, k);
    else if (a.gold[k] < 0 || a.gold[k] >= K) set_error(err, JET_ERR_OFFSETS, k);
  }
  __syncthreads();
  if (*(volatile int*)err != 0) return;
  for (int k = warp; k < a.n_sets; k += FT_WARPS) {
    const int c0 = a.set_offsets[k], c1 = a.set_offsets[k + 1], g = c0 + a.gold[k];
    for (int c = c0 + lane; c < c1; c += 32)
      a.flags[c] = (c == g || same_seq(a.tok_ids, a.cand_offsets, c, g)) ? 1 : 0;
  }
  if (tid == 0) {
    double lo = 1.0 / a.T_max, hi = 1.0 / a.T_min;
    s_beta = fmin(fmax(1.0, lo), hi);   // start from T = 1 (clamped into the interval)
    s_done = 0;
  }
  __syncthreads();

  double lo = 1.0 / a.T_max, hi = 1.0 / a.T_min, loss = 0.0;
  int it = 0;
  for (;; ++it) {
    const double beta = s_beta;
    const float bf = (float)beta;
    // one thread per set: per-set terms in fp32, the sum over sets in fp64
    double L = 0.0, G = 0.0, Hs = 0.0;
    for (int k = tid; k < a.n_sets; k += FT_THREADS) {
      const int c0 = a.set_offsets[k], c1 = a.set_offsets[k + 1];
      float m = -INFINITY, mg = -INFINITY;
      for (int c = c0; c < c1; ++c) {
        const float sv = a.s[c];
        m = fmaxf(m, sv);
        if (a.flags[c]) mg = fmaxf(mg, sv);
      }
      float z = 0.f, s1 = 0.f, s2 = 0.f, zg = 0.f, s1g = 0.f, s2g = 0.f;
      for (int c = c0; c < c1; ++c) {
        const float sv = a.s[c];
        const float x = sv - m;
        const float w = expf(bf * x);
        z += w; s1 += w * x; s2 += w * x * x;
        if (a.flags[c]) {
          const float xg = sv - mg;
          const float wg = expf(bf * xg);
          zg += wg; s1g += wg * xg; s2g += wg * xg * xg;
        }
      }
      const float ea = s1 / z, eg = s1g / zg;       // centred means
      L += (double)(bf * (m - mg) + logf(z) - logf(zg));
      G += (double)((m + ea) - (mg + eg));
      Hs += (double)((s2 / z - ea * ea) - (s2g / zg - eg * eg));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      L += __shfl_xor_sync(0xffffffffu, L, o);
      G += __shfl_xor_sync(0xffffffffu, G, o);
      Hs += __shfl_xor_sync(0xffffffffu, Hs, o);
    }
    if (lane == 0) {
      s_part[warp][0] = L;
      s_part[warp][1] = G;
      s_part[warp][2] = Hs;
    }
    __syncthreads();
    if (warp == 0) {
      double Lt = s_part[lane][0], Gt = s_part[lane][1], Ht = s_part[lane][2];   // FT_WARPS == 32
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        Lt += __shfl_xor_sync(0xffffffffu, Lt, o);
        Gt += __shfl_xor_sync(0xffffffffu, Gt, o);
        Ht += __shfl_xor_sync(0xffffffffu, Ht, o);
      }
      if (lane == 0) {   // thread 0: the bracket and the iterate live here
        loss = Lt;
        if (Gt > 0.0) hi = beta;          // NLL rising in beta: the optimum lies below
        else lo = beta;
        double next = (Ht > 0.0) ? beta - Gt / Ht : 0.5 * (lo + hi);
        if (!(next > lo && next < hi)) next = 0.5 * (lo + hi);
        const bool done = Gt == 0.0 || fabs(next - beta) <= FT_REL_TOL * beta ||
                          (hi - lo) <= FT_REL_TOL * beta || it + 1 >= FT_MAX_IT;
        s_done = done ? 1 : 0;
        if (!done) s_beta = next;
      }
    }
    __syncthreads();
    if (s_done) break;
  }
  if (tid == 0) {
    const double beta = s_beta;
    a.result[0] = 1.0 / beta;
    a.result[1] = loss / a.n_sets;
    a.result[2] = it + 1;
  }
}

}  // namespace

cudaError_t launch_fit_temperature(const FitArgs& a, cudaStream_t st) {
  fit_temperature_kernel<<<1, FT_THREADS, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace jet
