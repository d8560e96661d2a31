// Decision-guided layer sensitivity ("FastJEV: Understanding Redundancy for
// Compact JEV Inference", section 3.4, Eq. 5-6):
//
//   d_l(x) = rms(ctr(z^(-l)(x) - z(x))) / max(eps, rms(ctr(z(x)))),  eps = 1e-8
//   J_l    = mean over calibration inputs x of d_l(x)
//   selected = the k layers of smallest J_l, ties resolved by layer index
//
// with ctr(v) = v - mean(v) and rms(v) = ||v|| / sqrt(m).  Each input's logit
// vector (its candidate logits) is a CSR segment.  Kernel 1: one warp per
// (layer, input), two passes (means, then centred sums of squares) with fixed
// butterfly reductions.  Kernel 2: one CTA; warp per layer sums d in input
// order, then each layer's rank among (J, index) places it in the selection.
#include "jet_internal.cuh"

namespace jet {
namespace {

constexpr float SENS_EPS = 1e-8f;

__device__ __forceinline__ float wsum_s(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void sens_validate_kernel(const SensArgs a) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < ERR_WORDS; ++i) a.err[i] = 0;
  }
  __syncthreads();
  if (tid == 0 && (a.offsets[0] != 0 || a.offsets[a.n_inputs] != a.total)) set_error(a.err, JET_ERR_OFFSETS, 0);
  for (int x = tid; x < a.n_inputs; x += blockDim.x)
    if (a.offsets[x + 1] <= a.offsets[x]) set_error(a.err, JET_ERR_OFFSETS, x);
}

__global__ void sens_d_kernel(const SensArgs a) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (*(volatile const int*)a.err != 0 || wid >= a.L * a.n_inputs) return;
  const int l = wid / a.n_inputs, x = wid - l * a.n_inputs;
  const int b = a.offsets[x], e = a.offsets[x + 1];
  const float inv_m = 1.0f / (float)(e - b);
  const float* z = a.z;
  const float* zs = a.z_skip + (size_t)l * a.total;
  float sz = 0.f, sd = 0.f;
  for (int i = b + lane; i < e; i += 32) {
    sz += z[i];
    sd += zs[i] - z[i];
  }
  const float mz = wsum_s(sz) * inv_m, md = wsum_s(sd) * inv_m;
  float qz = 0.f, qd = 0.f;
  for (int i = b + lane; i < e; i += 32) {
    const float cz = z[i] - mz, cd = (zs[i] - z[i]) - md;
    qz += cz * cz;
    qd += cd * cd;
  }
  const float rz = sqrtf(wsum_s(qz) * inv_m), rd = sqrtf(wsum_s(qd) * inv_m);
  if (lane == 0) a.d[(size_t)l * a.n_inputs + x] = rd / fmaxf(SENS_EPS, rz);
}

__global__ void __launch_bounds__(1024) sens_select_kernel(const SensArgs a) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  if (*(volatile const int*)a.err != 0) return;
  for (int l = warp; l < a.L; l += nw) {
    float acc = 0.f;
    for (int x = lane; x < a.n_inputs; x += 32) acc += a.d[(size_t)l * a.n_inputs + x];
    acc = wsum_s(acc);
    if (lane == 0) a.J[l] = acc / (float)a.n_inputs;
  }
  __syncthreads();
  for (int l = tid; l < a.L; l += blockDim.x) {
    const float jl = a.J[l];
    int rank = 0;
    for (int o = 0; o < a.L; ++o) {
      const float jo = a.J[o];
      rank += (jo < jl) || (jo == jl && o < l);
    }
    if (rank < a.k) a.selected[rank] = l;
  }
}

}  // namespace

cudaError_t launch_sensitivity(const SensArgs& a, cudaStream_t st) {
  sens_validate_kernel<<<1, 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long warps = (long long)a.L * a.n_inputs;
  sens_d_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sens_select_kernel<<<1, 1024, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace jet
