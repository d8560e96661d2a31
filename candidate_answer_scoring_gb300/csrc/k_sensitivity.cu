// Decision-guided layer sensitivity ("FastJEV: Understanding Redundancy for
// Compact JEV Inference", section 3.4, Eq. 5-6):
//
//   d_l(x) = rms(ctr(z^(-l)(x) - z(x))) / max(eps, rms(ctr(z(x)))),  eps = 1e-8
//   J_l    = mean over calibration inputs x of d_l(x)
//   selected = the k layers of smallest J_l, ties resolved by layer index
//
// with ctr(v) = v - mean(v) and rms(v) = ||v|| / sqrt(m).  Each input's logit
// vector (its candidate logits) is a CSR segment.
//   d pass    one warp per (input, group of 32 layers), lanes over the
//             segment's elements (coalesced): the input's logits stay in
//             registers (segments up to 256 logits; longer ones take a
//             two-pass loop over memory), the layers' segments are loaded
//             16 values per lane at a time, the next batch's loads issued
//             before this batch is reduced, and the layers' means and centred
//             sums of squares are reduced together (transpose_reduce, fixed
//             order); rms(ctr(z)) is exactly
//             0 for a flat vector; each warp validates its own segment before
//             reading it;
//   J pass    one CTA per layer sums its d over inputs in a fixed order;
//   select    each layer's rank among (J, index) places it in the selection.
#include <algorithm>

#include "jet_internal.cuh"

namespace jet {
namespace {

constexpr float SENS_EPS = 1e-8f;

__device__ __forceinline__ float wsum_s(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float wmin_s(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float wmax_s(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

constexpr int SENS_LG = 32;  // layers per warp in the d pass

// Sums over the warp of SB values per lane (one per layer), SB a power of two
// <= 32, in 5 + (SB - 1) - log2(SB) shuffles instead of 5 * SB: at each of the
// first log2(SB) butterfly steps a lane keeps the half of its values that its
// partner does not and adds the partner's copy; the remaining steps are a
// plain butterfly.  Afterwards lane l holds the total of value rt_layer<SB>(l).
// Fixed order: identical inputs give identical sums.
template <int SB>
__device__ __forceinline__ float transpose_reduce(float (&v)[SB], int lane) {
#pragma unroll
  for (int half = SB / 2, off = 16; half >= 1; half /= 2, off /= 2) {
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = hi ? v[i] : v[i + half];
      const float recv = __shfl_xor_sync(0xffffffffu, send, off);
      v[i] = (hi ? v[i + half] : v[i]) + recv;
    }
  }
  float t = v[0];
#pragma unroll
  for (int off = 16 / SB; off >= 1; off /= 2) t += __shfl_xor_sync(0xffffffffu, t, off);
  return t;
}

// Which value lane l holds after transpose_reduce<SB>, and a lane holding value u.
template <int SB>
__device__ __forceinline__ int rt_layer(int lane) {
  int u = 0;
#pragma unroll
  for (int half = SB / 2, off = 16; half >= 1; half /= 2, off /= 2)
    if (lane & off) u += half;
  return u;
}
template <int SB>
__device__ __forceinline__ int rt_lane(int u) {
  int l = 0;
#pragma unroll
  for (int half = SB / 2, off = 16; half >= 1; half /= 2, off /= 2)
    if (u & half) l += off;
  return l;
}

// One input's segment (elements b + lane + 32 j of each layer row, VPL per
// lane) in SB consecutive layers from layer l, one load each; layers past the
// last one load the last layer again (never stored).
template <int VPL, int SB>
__device__ __forceinline__ void sens_load_batch(const SensArgs& a, int l, int b, int lane, const bool (&in)[VPL],
                                                float (&dv)[SB][VPL]) {
#pragma unroll
  for (int u = 0; u < SB; ++u) {
    const float* zs = a.z_skip + (size_t)min(l + u, a.L - 1) * a.total;
#pragma unroll
    for (int j = 0; j < VPL; ++j) dv[u][j] = in[j] ? zs[b + lane + 32 * j] : 0.f;
  }
}

// d for layers [l0, l0 + SENS_LG) of input x, its segment [b, e) held as VPL
// values per lane (element b + lane + 32 j); the segments of SB layers are
// loaded together (SB * VPL = 16 loads per lane), and the next SB layers'
// loads are issued before this batch is reduced.
template <int VPL>
__device__ __forceinline__ void sens_d_regs(const SensArgs& a, int x, int l0, int b, int e, int lane) {
  constexpr int SB = 16 / VPL;
  static_assert(SENS_LG % SB == 0, "layer group in whole sub-batches");
  const float fm = (float)(e - b), inv_m = 1.0f / fm;
  float zr[VPL];
  bool in[VPL];
  float sz = 0.f, lo = INFINITY, hi = -INFINITY;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int i = b + lane + 32 * j;
    in[j] = i < e;
    zr[j] = in[j] ? a.z[i] : 0.f;
    sz += zr[j];
    if (in[j]) { lo = fminf(lo, zr[j]); hi = fmaxf(hi, zr[j]); }
  }
  const float mz = __fdiv_rn(wsum_s(sz), fm);   // correctly rounded: no contraction into the centring
  float qz = 0.f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const float c = in[j] ? zr[j] - mz : 0.f;
    qz += c * c;
  }
  // a flat logit vector has rms(ctr(z)) = 0 exactly (fp32 centring would leave ulps)
  const bool flat = wmin_s(lo) == wmax_s(hi);
  const float rz = flat ? SENS_EPS : fmaxf(SENS_EPS, sqrtf(wsum_s(qz) * inv_m));
  float dv[SB][VPL];
  sens_load_batch<VPL, SB>(a, l0, b, lane, in, dv);
#pragma unroll 1
  for (int t0 = 0; t0 < SENS_LG; t0 += SB) {
    float nx[SB][VPL];
    const bool more = t0 + SB < SENS_LG && l0 + t0 + SB < a.L;
    if (more) sens_load_batch<VPL, SB>(a, l0 + t0 + SB, b, lane, in, nx);
    float part[SB];
#pragma unroll
    for (int u = 0; u < SB; ++u) {
      part[u] = 0.f;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        dv[u][j] = in[j] ? dv[u][j] - zr[j] : 0.f;
        part[u] += dv[u][j];
      }
    }
    // lane l now holds the mean of layer rt_layer(l); every lane takes each layer's
    const float mine = __fdiv_rn(transpose_reduce<SB>(part, lane), fm);
#pragma unroll
    for (int u = 0; u < SB; ++u) {
      const float md = __shfl_sync(0xffffffffu, mine, rt_lane<SB>(u));
      part[u] = 0.f;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const float c = in[j] ? dv[u][j] - md : 0.f;
        part[u] += c * c;
      }
    }
    const float rd = sqrtf(transpose_reduce<SB>(part, lane) * inv_m);
    const int l = l0 + t0 + rt_layer<SB>(lane);
    if (lane == rt_lane<SB>(rt_layer<SB>(lane)) && l < a.L) a.d[(size_t)l * a.n_inputs + x] = rd / rz;
    if (!more) break;
#pragma unroll
    for (int u = 0; u < SB; ++u)
#pragma unroll
      for (int j = 0; j < VPL; ++j) dv[u][j] = nx[u][j];
  }
}

// Segments longer than 32 * 8 logits: two passes over memory per layer.
__device__ void sens_d_loop(const SensArgs& a, int x, int l0, int b, int e, int lane) {
  const float fm = (float)(e - b), inv_m = 1.0f / fm;
  float sz = 0.f, lo = INFINITY, hi = -INFINITY;
  for (int i = b + lane; i < e; i += 32) {
    const float v = a.z[i];
    sz += v;
    lo = fminf(lo, v);
    hi = fmaxf(hi, v);
  }
  const bool flat = wmin_s(lo) == wmax_s(hi);
  const float mz = __fdiv_rn(wsum_s(sz), fm);
  float qz = 0.f;
  for (int i = b + lane; i < e; i += 32) {
    const float c = a.z[i] - mz;
    qz += c * c;
  }
  const float rz = flat ? SENS_EPS : fmaxf(SENS_EPS, sqrtf(wsum_s(qz) * inv_m));
  for (int l = l0; l < min(l0 + SENS_LG, a.L); ++l) {
    const float* zs = a.z_skip + (size_t)l * a.total;
    float sd = 0.f;
    for (int i = b + lane; i < e; i += 32) sd += zs[i] - a.z[i];
    const float md = __fdiv_rn(wsum_s(sd), fm);
    float qd = 0.f;
    for (int i = b + lane; i < e; i += 32) {
      const float c = (zs[i] - a.z[i]) - md;
      qd += c * c;
    }
    const float rd = sqrtf(wsum_s(qd) * inv_m);
    if (lane == 0) a.d[(size_t)l * a.n_inputs + x] = rd / rz;
  }
}

__global__ void sens_d_kernel(const SensArgs a) {
  pdl_trigger();   // the J pass waits for this grid before reading d
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int groups = (a.L + SENS_LG - 1) / SENS_LG;
  if (w >= groups * a.n_inputs) return;
  const int x = w / groups, g = w - x * groups;   // neighbouring warps: one input's layer groups
  const int b = a.offsets[x], e = a.offsets[x + 1], m = e - b;
  if (w == 0 && lane == 0 && (a.offsets[0] != 0 || a.offsets[a.n_inputs] != a.total))
    set_error(a.err, JET_ERR_OFFSETS, 0);
  if (!(b >= 0 && b < e && e <= a.total)) {   // empty or out-of-range segment: never read
    if (lane == 0 && g == 0) set_error(a.err, JET_ERR_OFFSETS, x);
    return;
  }
  const int l0 = g * SENS_LG;
  if (m <= 64) sens_d_regs<2>(a, x, l0, b, e, lane);
  else if (m <= 256) sens_d_regs<8>(a, x, l0, b, e, lane);
  else sens_d_loop(a, x, l0, b, e, lane);
}

// J[l] = mean over inputs of d[l][x]: CTA l, thread t sums inputs t, t + 256, ...
__global__ void __launch_bounds__(256) sens_j_kernel(const SensArgs a) {
  __shared__ float s_w[8];
  pdl_wait();
  pdl_trigger();
  if (*(volatile const int*)a.err != 0) return;
  const int l = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* dl = a.d + (size_t)l * a.n_inputs;
  float acc = 0.f;
  for (int x = tid; x < a.n_inputs; x += 256) acc += dl[x];
  acc = wsum_s(acc);
  if (lane == 0) s_w[warp] = acc;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int i = 0; i < 8; ++i) t += s_w[i];
    a.J[l] = t / (float)a.n_inputs;
  }
}

__global__ void __launch_bounds__(1024) sens_select_kernel(const SensArgs a) {
  pdl_wait();
  if (*(volatile const int*)a.err != 0) return;
  for (int l = threadIdx.x; l < a.L; l += blockDim.x) {
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
  cudaError_t e = cudaMemsetAsync(a.err, 0, ERR_WORDS * sizeof(int), st);
  if (e != cudaSuccess) return e;
  const long long warps = (long long)((a.L + SENS_LG - 1) / SENS_LG) * a.n_inputs;
  sens_d_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_dependent(sens_j_kernel, dim3(a.L), dim3(256), 0, st, a);
  if (e != cudaSuccess) return e;
  return launch_dependent(sens_select_kernel, dim3(1), dim3(std::min(1024, ((a.L + 31) / 32) * 32)), 0, st, a);
}

}  // namespace jet
