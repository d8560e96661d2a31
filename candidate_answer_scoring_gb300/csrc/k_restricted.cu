// Restricted head: normalise over a gathered union of allowed code tokens
// instead of the full vocabulary ("PARALLEL_SCORING.md", Execution step 5:
// gather only the relevant tied-embedding rows, project the final hidden
// states onto the union of allowed code tokens, and let each field take its
// subset).  For row r and union U:
//   z_u    = H[r] . W[U_u]            (fp32 accumulation of bf16 products)
//   lse_U  = log sum_u exp z_u
//   logp_j = z_{pos(tok_j)} - lse_U   for the row's tokens
// The set rules then run unchanged; within a set sharing one row, lse_U
// cancels and q = softmax(z / T) over the set's codes (step 6).
//
// Work is tiny (|U| is tens of codes) and latency-bound, so the kernel
// spreads it wide: one CTA of 32 warps per hidden row, one code per warp at a
// time.  Lane l multiplies 16-byte bf16 vectors l, l+32, ... of the row and
// of the code's embedding row (the union rows stay L2-resident across CTAs),
// loading up to 4 vector pairs before using them, and a fixed butterfly
// finishes each dot product, so identical rows give bit-identical logits.
// z_U lives in shared memory; the CTA then takes lse_U and writes the
// log-probability of each of the row's tokens.
#include <cuda_bf16.h>

#include "jet_internal.cuh"

namespace jet {
namespace {

constexpr int RT_THREADS = 1024;  // 32 warps
constexpr int RT_WARPS = RT_THREADS / 32;
constexpr int RT_BATCH = 4;       // 16-byte vector pairs in flight per lane (64-register budget)

__device__ __forceinline__ float dot_bf16x8(uint4 h, uint4 w, float acc) {
  const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&h);
  const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 hf = __bfloat1622float2(hp[i]);
    const float2 wf = __bfloat1622float2(wp[i]);
    acc = fmaf(hf.x, wf.x, acc);
    acc = fmaf(hf.y, wf.y, acc);
  }
  return acc;
}

__global__ void __launch_bounds__(RT_THREADS) restricted_kernel(const RestrictedArgs a) {
  __shared__ float sZ[JET_MAX_UNION];
  __shared__ float sRed[2 * RT_WARPS];
  pdl_trigger();
  pdl_wait();
  if (*(volatile const int*)a.err != 0) return;
  const int r = blockIdx.x;
  const int U = a.n_union;
  const int nvec = a.d / 8;                             // 16-byte vectors per row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4* h = reinterpret_cast<const uint4*>(a.H) + (size_t)r * nvec;
  const uint4* Wv = reinterpret_cast<const uint4*>(a.W);

  for (int u = warp; u < U; u += RT_WARPS) {
    const uint4* w = Wv + (size_t)a.union_ids[u] * nvec;
    float acc = 0.f;
    for (int k0 = lane; k0 < nvec; k0 += 32 * RT_BATCH) {
      uint4 hv[RT_BATCH], wv[RT_BATCH];
#pragma unroll
      for (int i = 0; i < RT_BATCH; ++i) {
        const int k = k0 + 32 * i;
        if (k < nvec) { hv[i] = h[k]; wv[i] = w[k]; }
      }
#pragma unroll
      for (int i = 0; i < RT_BATCH; ++i)
        if (k0 + 32 * i < nvec) acc = dot_bf16x8(hv[i], wv[i], acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sZ[u] = acc;
  }
  __syncthreads();

  // lse over the union: block max, then block sum of exp(z - max)
  float M = -INFINITY;
  for (int u = threadIdx.x; u < U; u += RT_THREADS) M = fmaxf(M, sZ[u]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) sRed[warp] = M;
  __syncthreads();
  M = sRed[0];
#pragma unroll
  for (int i = 1; i < RT_WARPS; ++i) M = fmaxf(M, sRed[i]);
  float sum = 0.f;
  for (int u = threadIdx.x; u < U; u += RT_THREADS) sum += expf(sZ[u] - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) sRed[RT_WARPS + warp] = sum;
  __syncthreads();
  sum = 0.f;
#pragma unroll
  for (int i = 0; i < RT_WARPS; ++i) sum += sRed[RT_WARPS + i];
  const float lse = M + logf(sum);
  if (threadIdx.x == 0 && a.lse) a.lse[r] = lse;
  for (int e = a.row_ptr[r] + threadIdx.x; e < a.row_ptr[r + 1]; e += RT_THREADS) {
    const int j = a.row_list[e].y;
    a.logp[j] = sZ[a.upos[j]] - lse;
  }
}

}  // namespace

cudaError_t launch_restricted(const RestrictedArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  return launch_dependent(restricted_kernel, dim3(a.N), dim3(RT_THREADS), 0, st, a);
}

}  // namespace jet
