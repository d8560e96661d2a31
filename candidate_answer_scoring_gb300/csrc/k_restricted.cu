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
// Work is tiny (|U| is tens of codes); the kernel is launch-latency bound.  A
// CTA stages R hidden rows and chunks of the gathered W_U rows in shared
// memory; one warp per row computes the |U| dot products (lane-strided over d
// in 16-byte vectors, fixed-order warp reduction) into shared memory.
#include <cuda_bf16.h>

#include "jet_internal.cuh"

namespace jet {
namespace {

constexpr int RT_THREADS = 256;   // 8 warps
constexpr int RT_MAX_ROWS = 8;

struct RtShape { int R, CH; size_t smem; };

__host__ __device__ inline RtShape rt_shape(int d, int n_union) {
  RtShape s;
  const size_t row_bytes = (size_t)d * 2;
  int R = RT_MAX_ROWS;
  while (R > 1 && (size_t)R * (row_bytes + (size_t)n_union * 4) > 112 * 1024) --R;
  int CH = (int)((64 * 1024) / row_bytes);
  if (CH < 1) CH = 1;
  if (CH > n_union) CH = n_union;
  s.R = R;
  s.CH = CH;
  s.smem = (size_t)R * row_bytes + (size_t)CH * row_bytes + (size_t)R * n_union * 4;
  return s;
}

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

__global__ void __launch_bounds__(RT_THREADS) restricted_kernel(const RestrictedArgs a, const RtShape sh) {
  extern __shared__ __align__(16) uint8_t smem[];
  if (*(volatile const int*)a.err != 0) return;
  const int d = a.d, U = a.n_union;
  const int vec_per_row = d / 8;                       // 16-byte vectors per row
  uint4* sH = reinterpret_cast<uint4*>(smem);                          // [R][d]
  uint4* sW = sH + (size_t)sh.R * vec_per_row;                          // [CH][d]
  float* sZ = reinterpret_cast<float*>(sW + (size_t)sh.CH * vec_per_row);   // [R][U]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * sh.R;
  const int nrows = min(sh.R, a.N - r0);

  const uint4* Hg = reinterpret_cast<const uint4*>(a.H);
  for (int i = threadIdx.x; i < nrows * vec_per_row; i += blockDim.x)
    sH[i] = Hg[(size_t)r0 * vec_per_row + i];

  const uint4* Wg = reinterpret_cast<const uint4*>(a.W);
  for (int u0 = 0; u0 < U; u0 += sh.CH) {
    const int nu = min(sh.CH, U - u0);
    __syncthreads();
    for (int i = threadIdx.x; i < nu * vec_per_row; i += blockDim.x) {
      const int uu = i / vec_per_row, k = i - uu * vec_per_row;
      sW[i] = Wg[(size_t)a.union_ids[u0 + uu] * vec_per_row + k];
    }
    __syncthreads();
    for (int lr = warp; lr < nrows; lr += RT_THREADS / 32) {
      const uint4* h = sH + (size_t)lr * vec_per_row;
      for (int uu = 0; uu < nu; ++uu) {
        const uint4* w = sW + (size_t)uu * vec_per_row;
        float acc = 0.f;
        for (int k = lane; k < vec_per_row; k += 32) acc = dot_bf16x8(h[k], w[k], acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) sZ[(size_t)lr * U + u0 + uu] = acc;
      }
    }
  }
  __syncthreads();

  for (int lr = warp; lr < nrows; lr += RT_THREADS / 32) {
    const float* z = sZ + (size_t)lr * U;
    float M = -INFINITY;
    for (int u = lane; u < U; u += 32) M = fmaxf(M, z[u]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float s = 0.f;
    for (int u = lane; u < U; u += 32) s += expf(z[u] - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float lse = M + logf(s);
    const int r = r0 + lr;
    if (lane == 0 && a.lse) a.lse[r] = lse;
    for (int e = a.row_ptr[r] + lane; e < a.row_ptr[r + 1]; e += 32) {
      const int j = a.row_list[e].y;
      a.logp[j] = z[a.upos[j]] - lse;
    }
  }
}

}  // namespace

cudaError_t launch_restricted(const RestrictedArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  const RtShape sh = rt_shape(a.d, a.n_union);
  static size_t configured = 0;
  if (sh.smem > 48 * 1024 && sh.smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(restricted_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sh.smem);
    if (e != cudaSuccess) return e;
    configured = sh.smem;
  }
  restricted_kernel<<<(a.N + sh.R - 1) / sh.R, RT_THREADS, sh.smem, st>>>(a, sh);
  return cudaGetLastError();
}

}  // namespace jet
