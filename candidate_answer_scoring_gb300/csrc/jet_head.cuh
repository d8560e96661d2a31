// Internal declarations of libjetscore shared by every kernel, and those of
// the full-vocabulary head (tile shape, schedule, arguments).  Not part of the
// C ABI.  The head's translation unit includes only this header, the bounded
// wait and jetscore.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "jetscore.h"

namespace jet {

// ---- full-vocabulary head tile shape (tcgen05) ------------------------------
// One CTA owns 128 hidden rows (its TMEM lanes) and 256 vocabulary columns of
// a tile.  In the paired variant two CTAs of a cluster run one
// tcgen05.mma.cta_group::2 (M = 256): each stages its own 128 rows of H and
// half (128 rows) of the W tile.
constexpr int BM = 128;             // hidden rows per CTA tile = TMEM lanes
constexpr int BN = 256;             // vocabulary columns per tile = fp32 TMEM columns
constexpr int BK = 64;              // bf16 elements per k-block = one 128-byte swizzle row
constexpr int EPI_WARPS = 8;        // two warpgroups: column halves of a tile
constexpr int HEAD_THREADS = (2 + EPI_WARPS) * 32;
constexpr int TMEM_COLS = 2 * BN;   // two accumulators (double buffer)

// A ring stage holds KPS consecutive k-blocks of H and of W; the MMA thread
// waits once and commits once per stage.  Paired head, schedules of several
// waves of units (tensor-bound batches): stages of two k-blocks (3 stages,
// the same bytes in flight as 6 of one), 1-2% faster there.  One wave (few
// row tiles, W streaming): six stages of one k-block, 3% faster on the
// 256-row batch.  One CTA: four stages of one 48 KB k-block (two of two were
// 4% slower on 128-row batches).
template <bool PAIR, int KPS_ = 1>
struct HeadShape {
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;   // W rows this CTA stages per tile
  static constexpr int KPS = KPS_;                     // k-blocks per ring stage
  static constexpr int A_KB_BYTES = BM * BK * 2;       // one k-block of this CTA's H rows
  static constexpr int B_KB_BYTES = B_ROWS * BK * 2;   // one k-block of this CTA's W rows
  static constexpr int A_BYTES = KPS * A_KB_BYTES;
  static constexpr int B_BYTES = KPS * B_KB_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = !PAIR ? 4 : (KPS == 1 ? 6 : 3);   // shared-memory ring depth
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 512 /*barriers, unit ring*/;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert(A_KB_BYTES % 1024 == 0 && B_KB_BYTES % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
};

// Device-side error word layout: err[0] = first status (0 = ok),
// err[1] = index of the offending element, err[2] = where a wait gave up.
constexpr int ERR_WORDS = 4;
// err[SCHED_WORD]: the head's unit counter when units are handed out
// dynamically; the pre-pass zeroes it together with the error words.
constexpr int SCHED_WORD = ERR_WORDS;

__device__ __forceinline__ void set_error(int* err, int code, int detail) {
  if (atomicCAS(err, 0, code) == 0) err[1] = detail;
}

// Programmatic dependent launch: kernels of one call are launched so that the
// next may be scheduled while the previous is still running.  A kernel calls
// pdl_wait() before it reads anything the previous kernel writes (including
// the error word); pdl_wait() returns at once when there is no dependency.
// pdl_trigger() lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Programmatic dependent launch is on unless the environment variable
// JETSCORE_NO_PDL is set (a diagnostic: launches then serialise normally).
bool pdl_enabled();

// Launch `kernel` on `st` as a programmatic dependent of the preceding kernel.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Vocabulary-split schedule of the head: unit u = (row tile m, split s) covers
// vocabulary tiles [s*n_vt/S, (s+1)*n_vt/S).  A row tile is 128 rows (one CTA)
// or, paired, 256 rows (a CTA pair).  Units are ordered band by band (Gm row
// tiles per band), split-major inside a band, so CTAs running together share
// W tiles through L2 while the band's H tiles stay L2-resident.
struct Plan {
  int n_mt = 0, n_vt = 0, S = 1, Gm = 1, n_full_bands = 0, r_last = 0, units = 0, grid = 0;
  int pair = 0;   // 1: units run on CTA pairs (cta_group::2)
};

__host__ __device__ __forceinline__ int plan_tile_rows(const Plan& p) { return p.pair ? 2 * BM : BM; }

// Slot of the (max, sum-exp) partial of (unit u, CTA sub of the pair, column
// half h, row lr of the CTA's 128).
__host__ __device__ __forceinline__ size_t part_slot(const Plan& p, int u, int sub, int h, int lr) {
  return (((size_t)u * (1 + p.pair) + sub) * 2 + h) * BM + lr;
}

struct HeadArgs {
  int N, V, d;
  Plan plan;
  const int* row_ptr;   // [N+1]   CSR over rows of the scored tokens
  const int2* row_list; // [n_tok] (token id, token index), sorted by id within a row
  float* zg;            // [n_tok] gathered logit of each scored token
  float2* part;         // per (unit, CTA of the pair, column half, row): (max, sum exp(z - max))
  int* err;
  int w_tiled = 0;      // tmW is the 4-D map of a tiled W (jet_tile_weights)
  int* sched = nullptr; // paired head, several waves of units: counter (zeroed by the pre-pass)
                        // from which pairs take units after their first; NULL: static stride
};

// Host: schedule for N rows on G SMs; units * (1 + pair) <= units_cap.
Plan make_plan(int N, int V, int d, int G, int units_cap, bool pair);
bool head_use_dynamic(const Plan& p);

// Host: whether the paired (2-SM) head serves N rows.
bool head_use_pair(int N);

// Decode unit u of the plan into (row tile, first vocab tile, end vocab tile).
__host__ __device__ __forceinline__ void plan_unit(const Plan& p, int u, int& m, int& vt0, int& vt1) {
  const int main_units = p.n_full_bands * p.Gm * p.S;
  int split;
  if (u < main_units) {
    const int per_band = p.Gm * p.S;
    const int band = u / per_band, w = u - band * per_band;
    split = w / p.Gm;
    m = band * p.Gm + (w - split * p.Gm);
  } else {
    const int w = u - main_units;
    split = w / p.r_last;
    m = p.n_full_bands * p.Gm + (w - split * p.r_last);
  }
  vt0 = (int)((int64_t)split * p.n_vt / p.S);
  vt1 = (int)((int64_t)(split + 1) * p.n_vt / p.S);
}

// Unit index of (row tile m, split s): the inverse of plan_unit.
__host__ __device__ __forceinline__ int plan_unit_of(const Plan& p, int m, int split) {
  const int band = m / p.Gm;
  if (band < p.n_full_bands) return band * p.Gm * p.S + split * p.Gm + (m - band * p.Gm);
  return p.n_full_bands * p.Gm * p.S + split * p.r_last + (m - p.n_full_bands * p.Gm);
}

// tmW's box must have HeadShape<a.plan.pair>::B_ROWS rows; tmH's box BM rows.
cudaError_t launch_head(const CUtensorMap& tmH, const CUtensorMap& tmW, const HeadArgs& a,
                        cudaStream_t st);

}  // namespace jet
