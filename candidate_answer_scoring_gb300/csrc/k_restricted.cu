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
// For unions below 192 codes (answer codes A..Z are 26) the work is tiny and
// latency-bound, so the path is two launches with few dependent memory round
// trips each; larger unions are staged by union_rows_kernel (end of this
// file) and projected by the full-vocabulary tcgen05 head instead:
//
//  1. restricted_head_kernel: z = H U^T is a small dense contraction, run on
//     the tensor cores with mma.sync (m16n8k16, bf16 in, fp32 accumulate).
//     A cluster of four CTAs per 16 rows splits d four ways (so the union
//     rows and hidden rows each CTA stages are a quarter, and arrive in one
//     round of loads); each CTA's 16 warps split its quarter further, each
//     accumulating the 16 x 32 tile of a group of 32 codes.  The warps'
//     partials are summed in a fixed order through shared memory, then the
//     first CTA of the cluster adds the other three CTAs' sums (distributed
//     shared memory, rank order) and its warp r folds row r's 32 logits into
//     a running (max, sum) for lse_U.  z goes to an [N, |U|]
//     scratch when that fits the context's workspace, else the second kernel
//     recomputes the few logits it needs (a warp dot product: the same bf16
//     products in fp32, summed in another order).  CTA 0 zeroes the error word
//     and records each union id's position in a token-id map.  This kernel
//     validates nothing and reads only rows < N and union rows whose id lies
//     in [0, V).
//  2. restricted_sets_kernel, one warp per set: checks the set's offsets and
//     kind, that each candidate is one token whose id and row are in range and
//     whose id the map places in the union (the map is trusted only where
//     union_ids agrees, so stale entries from earlier calls are harmless;
//     with at most 32 codes the warp instead finds each token's position in
//     union_ids itself, before the wait),
//     forms logp, then runs the set rules.  Warp 0 of CTA 0 checks the ends of
//     the offset arrays and that the union ids are in range and distinct.
#include <cuda_bf16.h>

#include "jet_internal.cuh"
#include "jet_setrules.cuh"

namespace jet {
namespace {

constexpr int RT_WARPS = 16;                  // warps of the restricted head, splitting d
constexpr int RT_THREADS = RT_WARPS * 32;     // = 16 rows x 32 codes for the reduction
constexpr int RT_CODES = 32;                  // codes per group: four n8 tiles
constexpr int RT_UNROLL = 3;                  // 32-wide k chunks with loads in flight per warp
constexpr int RT_SPLIT = 4;                   // CTAs of a cluster splitting d for one 16-row tile
constexpr int DR_BATCH = 10;                  // 16-byte vectors in flight per lane (warp dot product)
constexpr int RS_WARPS = 8;                   // sets per CTA of the set kernel
constexpr int UR_BATCH = 8;                   // 16-byte loads in flight per lane when staging union rows

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

// Index of 16-byte vector j (elements 8j .. 8j+7) of W's row t, row-major or
// tiled ([ceil(V/128)][d/64][128][64]: vector j of row t lies in k-block j/8
// of tile t/128).  wbase = w_row_base(t).
__device__ __forceinline__ size_t w_row_base(int t, int d, bool tiled) {
  return tiled ? ((size_t)(t >> 7) * (d / 64) * 128 + (t & 127)) * 8 : (size_t)t * (d / 8);
}
__device__ __forceinline__ size_t w_vec(size_t wbase, int j, bool tiled) {
  return tiled ? wbase + (size_t)(j >> 3) * 1024 + (j & 7) : wbase + j;
}

// h . w over nvec 16-byte bf16 vectors by one warp (lane l takes vectors l,
// l+32, ...; a fixed butterfly combines the lanes; every lane gets the sum).
// w is row t of W: vector k at Wv[w_vec(wbase, k, tiled)].
__device__ __forceinline__ float dot_row(const uint4* h, const uint4* Wv, size_t wbase, bool tiled, int nvec,
                                         int lane) {
  float acc = 0.f;
  for (int k0 = lane; k0 < nvec; k0 += 32 * DR_BATCH) {
    uint4 hv[DR_BATCH / 2], wv[DR_BATCH / 2];
    for (int half = 0; half < 2; ++half) {
      const int kb = k0 + 32 * (DR_BATCH / 2) * half;
#pragma unroll
      for (int i = 0; i < DR_BATCH / 2; ++i) {
        const int k = kb + 32 * i;
        if (k < nvec) { hv[i] = h[k]; wv[i] = Wv[w_vec(wbase, k, tiled)]; }
      }
#pragma unroll
      for (int i = 0; i < DR_BATCH / 2; ++i)
        if (kb + 32 * i < nvec) acc = dot_bf16x8(hv[i], wv[i], acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// D += A B for one m16n8k16 tile: A 16x16 bf16 (row-major fragments), B 16x8
// bf16 (column-major fragments), D 16x8 fp32.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Row of H holding problem row r: r itself, or row_index[r] when gathering
// (an index outside [0, n_src) reads row 0; the set kernel reports it).
__device__ __forceinline__ int source_row(const RestrictedArgs& a, int r) {
  if (a.row_index == nullptr) return r;
  const int idx = a.row_index[r];
  return (idx >= 0 && idx < a.n_src) ? idx : 0;
}

__device__ __forceinline__ uint32_t rt_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster: shared-memory writes before it are
// visible to the cluster's reads after it.
__device__ __forceinline__ void rt_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store v at the same shared-memory offset as *p in CTA `rank` of the cluster.
__device__ __forceinline__ void rt_st_cluster(float* p, uint32_t rank, float v) {
  uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p)), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// The union's rows of W are loaded with an L2 evict-last hint: calls that
// score over the same union find them in L2, although the full-vocabulary
// head streams all of W through it (with evict-first) in between (binary
// step: load phase 2.0 -> 1.8 us).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_keep_l2(const uint4* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}

// Fragment mapping.  In an m16n8k16 MMA, lane (g = lane/4, c = lane%4) holds
// A elements (rows g and g+8) and B elements (code g) at k slots {2c, 2c+1,
// 2c+8, 2c+9}.  A dot product does not care which physical k feeds which slot
// as long as A and B agree, so slots {2c, 2c+1} take physical k = 4c, 4c+1 and
// slots {2c+8, 2c+9} take 4c+2, 4c+3: each lane then reads 4 consecutive
// elements per row and step, and one 16-byte load per row serves two steps of
// a 32-wide chunk (words 0-1: step 0, words 2-3: step 1).
__global__ void __launch_bounds__(RT_THREADS, 1) restricted_head_kernel(const RestrictedArgs a) {
  __shared__ float sAcc[RT_WARPS][16][RT_CODES + 1];
  __shared__ float sRecv[RT_SPLIT - 1][16][RT_CODES];   // first CTA: the other CTAs' sums, by rank
  __shared__ float sM[16], sS[16];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int U = a.n_union, d = a.d;
  const uint32_t crank = rt_cluster_rank();
  const int r0 = (int)(blockIdx.x / RT_SPLIT) * 16;
  pdl_wait();      // earlier work on the stream is complete before any access
  pdl_trigger();
  if (blockIdx.x == 0) {
    if (tid < ERR_WORDS) a.err[tid] = 0;
    for (int u = tid; u < U; u += RT_THREADS) {
      const int t = a.union_ids[u];
      if (t >= 0 && t < a.V) a.umap[t] = u;
    }
  }
  if (tid < 16) { sM[tid] = -INFINITY; sS[tid] = 0.f; }

  // this lane's two rows (clamped to the last row: loads stay in bounds, the
  // results of rows past N are never written)
  const int nch = d / 32;                                    // 32-wide k chunks
  const int cs0 = (int)crank * nch / RT_SPLIT, cn = ((int)crank + 1) * nch / RT_SPLIT - cs0;   // this CTA's
  const int ch0 = cs0 + warp * cn / RT_WARPS, ch1 = cs0 + (warp + 1) * cn / RT_WARPS;
  const uint4* hA = reinterpret_cast<const uint4*>(a.H + (size_t)source_row(a, min(r0 + g, a.N - 1)) * d) + c;
  const uint4* hB = reinterpret_cast<const uint4*>(a.H + (size_t)source_row(a, min(r0 + g + 8, a.N - 1)) * d) + c;

  for (int u0 = 0; u0 < U; u0 += RT_CODES) {
    // this lane's code for the reduction below, loaded with the operands
    const int t_lane = u0 + lane < U ? a.union_ids[u0 + lane] : -1;
    const uint4* Wv = reinterpret_cast<const uint4*>(a.W);
    const uint64_t pol_w = l2_evict_last_policy();   // the union's rows stay in L2 for the next call
    const bool tiled = a.w_tiled != 0;
    size_t wb[4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int u = u0 + nt * 8 + g;
      const int t = u < U ? a.union_ids[u] : -1;
      wb[nt] = w_row_base((t >= 0 && t < a.V) ? t : 0, d, tiled);
    }
    float acc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
    for (int ch = ch0; ch < ch1; ch += RT_UNROLL) {
      uint4 A0[RT_UNROLL], A1[RT_UNROLL], B[RT_UNROLL][4];
#pragma unroll
      for (int j = 0; j < RT_UNROLL; ++j) {
        if (ch + j < ch1) {
          const int v = (ch + j) * 4;                         // 16-byte vectors per chunk: 4 per row
          A0[j] = hA[v];
          A1[j] = hB[v];
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) B[j][nt] = ld_keep_l2(Wv + w_vec(wb[nt], v + c, tiled), pol_w);
        }
      }
#pragma unroll
      for (int j = 0; j < RT_UNROLL; ++j) {
        if (ch + j < ch1) {
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            mma_bf16_16816(acc[nt], A0[j].x, A1[j].x, A0[j].y, A1[j].y, B[j][nt].x, B[j][nt].y);
            mma_bf16_16816(acc[nt], A0[j].z, A1[j].z, A0[j].w, A1[j].w, B[j][nt].z, B[j][nt].w);
          }
        }
      }
    }
    // partial tiles to shared memory: (row g | g+8, code nt*8 + 2c | +1)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      sAcc[warp][g][nt * 8 + 2 * c] = acc[nt][0];
      sAcc[warp][g][nt * 8 + 2 * c + 1] = acc[nt][1];
      sAcc[warp][g + 8][nt * 8 + 2 * c] = acc[nt][2];
      sAcc[warp][g + 8][nt * 8 + 2 * c + 1] = acc[nt][3];
    }
    __syncthreads();
    // warp w now owns row w of the tile, lane = code: sum the warps' partials
    // in order; the first CTA adds the others' sums in rank order, stores z
    // and folds the group into the row's running (max, sum)
    float zp = 0.f;
#pragma unroll
    for (int w = 0; w < RT_WARPS; ++w) zp += sAcc[w][warp][lane];
    if (crank != 0) rt_st_cluster(&sRecv[crank - 1][warp][lane], 0, zp);
    rt_cluster_sync();   // the stores above are visible in the first CTA
    if (crank == 0) {
      const int row = warp, u = u0 + lane, r = r0 + row;
      float z = zp;
#pragma unroll
      for (int k = 0; k < RT_SPLIT - 1; ++k) z += sRecv[k][row][lane];
      bool valid = u < U;
      if (valid) {
        if (!(t_lane >= 0 && t_lane < a.V)) z = __int_as_float(0x7fc00000);   // reported by the set kernel
        if (a.zu && r < a.N) a.zu[(size_t)r * U + u] = z;
      }
      float m = valid ? z : -INFINITY;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const float M = fmaxf(sM[row], m);
      float e = valid ? expf(z - M) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
      if (lane == 0) {
        sS[row] = (sM[row] == -INFINITY ? 0.f : sS[row] * expf(sM[row] - M)) + e;
        sM[row] = M;
      }
    }
    // another group reuses sAcc and sRecv: the first CTA has read this one's first
    if (u0 + RT_CODES < U) rt_cluster_sync();
    else __syncthreads();
  }
  if (crank == 0 && lane == 0 && r0 + warp < a.N) {
    const float lse = sM[warp] + logf(sS[warp]);
    a.lse_row[r0 + warp] = lse;
    if (a.lse) a.lse[r0 + warp] = lse;
  }
}

// Candidate c of a restricted set: one token, id and row in range, id in the
// union.  Returns false (after recording the error) otherwise; with the
// union-logit scratch, also forms and stores the token's logp.
__device__ __forceinline__ bool restricted_candidate(const RestrictedSetArgs& a, int c, int& tok, float& lp) {
  const SetArgs& sa = a.s;
  const RestrictedArgs& ra = a.r;
  int* err = ra.err;
  const int t0 = sa.cand_offsets[c], t1 = sa.cand_offsets[c + 1];
  if (!(t0 >= 0 && t0 < t1 && t1 <= a.n_tok)) { set_error(err, JET_ERR_OFFSETS, c); return false; }
  if (t1 - t0 != 1) { set_error(err, JET_ERR_MODE, c); return false; }
  const int t = sa.tok_ids[t0], r = a.tok_row[t0];
  if (t < 0 || t >= ra.V || r < 0 || r >= ra.N) { set_error(err, JET_ERR_TOKEN_RANGE, t0); return false; }
  const int pos = ra.umap[t];
  const float lse = ra.lse_row[r];
  if (pos < 0 || pos >= ra.n_union) { set_error(err, JET_ERR_NOT_IN_UNION, t0); return false; }
  const int uid = ra.union_ids[pos];
  const float z = ra.zu ? ra.zu[(size_t)r * ra.n_union + pos] : 0.f;
  if (uid != t) { set_error(err, JET_ERR_NOT_IN_UNION, t0); return false; }   // a stale map entry
  tok = t;
  lp = z - lse;
  if (ra.zu) sa.logp[t0] = lp;
  return true;
}

// Sets of K <= 32*CPL candidates with the scratch: scores straight from the
// candidates' logp (s(c) = logp of its one token), rules in registers.
template <int CPL>
__device__ __forceinline__ void restricted_set_regs(const RestrictedSetArgs& a, int set, int lane, int c0, int K) {
  float sc[CPL];
  unsigned long long h[CPL];
  bool bad = false;
#pragma unroll
  for (int k = 0; k < CPL; ++k) {
    const int i = k * 32 + lane;
    sc[k] = -INFINITY;
    h[k] = 0;
    if (i < K) {
      int tok;
      float lp;
      if (restricted_candidate(a, c0 + i, tok, lp)) {
        sc[k] = 0.f + lp;                 // the chain rule over one token
        h[k] = single_token_hash(tok);
      } else {
        bad = true;
      }
    }
  }
  if (__any_sync(0xffffffffu, bad)) return;
  set_rules_core<CPL>(a.s, set, lane, c0, K, 1.0f / a.s.T, sc, h);
}

__global__ void __launch_bounds__(32 * RS_WARPS) restricted_sets_kernel(const RestrictedSetArgs a) {
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = blockIdx.x * RS_WARPS + wib;
  const SetArgs& sa = a.s;
  const RestrictedArgs& ra = a.r;
  int* err = ra.err;
  const int U = ra.n_union;

  // Before the restricted head finishes: the caller's index arrays (nothing in
  // this call writes them, and the head started only after everything earlier
  // on the stream had finished), checked as they are followed.  Errors are
  // held in registers and recorded after the wait (the head zeroes the error
  // word first).
  const bool live = k < sa.n_sets;
  int c0 = 0, c1 = 0, kd = 0, set_code = 0;
  int cand_code = 0, cand_at = 0, t0 = 0, tok = 0, row = 0;
  if (live) {
    c0 = sa.set_offsets[k];
    c1 = sa.set_offsets[k + 1];
    kd = a.kind[k];
    const int K = c1 - c0;
    if (!(c0 >= 0 && c0 < c1 && c1 <= a.n_cand)) set_code = JET_ERR_OFFSETS;
    else if (kd > JET_KIND_ORDINAL) set_code = JET_ERR_ARG;
    else if ((kd == JET_KIND_BINARY && K != 2) || (kd == JET_KIND_ORDINAL && K < 2)) set_code = JET_ERR_OFFSETS;
    if (set_code == 0 && ra.zu && K <= 32 && lane < K) {
      const int c = c0 + lane;
      t0 = sa.cand_offsets[c];
      const int t1 = sa.cand_offsets[c + 1];
      if (!(t0 >= 0 && t0 < t1 && t1 <= a.n_tok)) { cand_code = JET_ERR_OFFSETS; cand_at = c; }
      else if (t1 - t0 != 1) { cand_code = JET_ERR_MODE; cand_at = c; }
      else {
        tok = sa.tok_ids[t0];
        row = a.tok_row[t0];
        if (tok < 0 || tok >= ra.V || row < 0 || row >= ra.N) { cand_code = JET_ERR_TOKEN_RANGE; cand_at = t0; }
      }
    }
  }
  // unions of up to 32 codes: each candidate's union position from union_ids
  // itself (a caller input), so only the logit load waits for the head
  const bool pos_early = live && set_code == 0 && ra.zu && c1 - c0 <= 32 && U <= 32;
  int pos_pre = -1;
  if (pos_early) {
    const int u_lane = lane < U ? ra.union_ids[lane] : -1;
    const bool mine = lane < c1 - c0 && cand_code == 0;
    for (int j = 0; j < U; ++j) {
      const int uj = __shfl_sync(0xffffffffu, u_lane, j);
      if (mine && pos_pre < 0 && uj == tok) pos_pre = j;   // first position (a repeat is reported below)
    }
  }
  pdl_wait();
  pdl_trigger();
  if (ra.row_index)   // gathered rows: every index within the source array
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < ra.N; r += gridDim.x * blockDim.x) {
      const int idx = ra.row_index[r];
      if (idx < 0 || idx >= ra.n_src) set_error(err, JET_ERR_TOKEN_RANGE, r);
    }
  if (blockIdx.x == 0 && wib == 0) {
    if (lane == 0) {
      if (sa.set_offsets[0] != 0 || sa.set_offsets[sa.n_sets] != a.n_cand) set_error(err, JET_ERR_OFFSETS, 0);
      if (sa.cand_offsets[0] != 0 || sa.cand_offsets[a.n_cand] != a.n_tok) set_error(err, JET_ERR_OFFSETS, 0);
    }
    for (int u = lane; u < U; u += 32) {
      const int t = ra.union_ids[u];
      if (t < 0 || t >= ra.V) set_error(err, JET_ERR_TOKEN_RANGE, u);
      else if (ra.umap[t] != u) set_error(err, JET_ERR_NOT_IN_UNION, u);   // a repeated id keeps one position
    }
  }
  if (!live) return;
  // the set's own offsets and kind (consecutive sets share a boundary, so
  // with both ends checked above the sets tile [0, n_cand) exactly)
  if (set_code != 0) {
    if (lane == 0) set_error(err, set_code, k);
    return;
  }
  const int K = c1 - c0;
  if (ra.zu && K <= 32) {   // candidates followed before the wait: the union lookup remains
    float sc[1] = {-INFINITY};
    unsigned long long h[1] = {0};
    bool bad = false;
    if (lane < K) {
      if (cand_code != 0) {
        set_error(err, cand_code, cand_at);
        bad = true;
      } else {
        const int pos = pos_early ? pos_pre : ra.umap[tok];
        const float lse = ra.lse_row[row];
        if (pos < 0 || pos >= U) {
          set_error(err, JET_ERR_NOT_IN_UNION, t0);
          bad = true;
        } else {
          const int uid = pos_early ? tok : ra.union_ids[pos];   // found by id: no stale entry
          const float z = ra.zu[(size_t)row * U + pos];
          if (uid != tok) {   // a stale map entry
            set_error(err, JET_ERR_NOT_IN_UNION, t0);
            bad = true;
          } else {
            const float lp = z - lse;
            sa.logp[t0] = lp;
            sc[0] = 0.f + lp;   // the chain rule over one token
            h[0] = single_token_hash(tok);
          }
        }
      }
    }
    if (__any_sync(0xffffffffu, bad)) return;
    set_rules_core<1>(sa, k, lane, c0, K, 1.0f / sa.T, sc, h);
    return;
  }
  if (ra.zu && K <= 128) {
    if (K <= 64) restricted_set_regs<2>(a, k, lane, c0, K);
    else restricted_set_regs<4>(a, k, lane, c0, K);
    return;
  }

  // large sets, or no scratch: logp through global memory, then the general rules
  bool bad = false;
  for (int c = c0 + lane; c < c1; c += 32) {
    int tok;
    float lp;
    if (!restricted_candidate(a, c, tok, lp)) bad = true;
  }
  if (__any_sync(0xffffffffu, bad)) return;
  if (!ra.zu) {   // no scratch: the warp recomputes each candidate's logit
    const int nvec = ra.d / 8;
    for (int c = c0; c < c1; ++c) {
      const int t0 = sa.cand_offsets[c];
      const int t = sa.tok_ids[t0], r = a.tok_row[t0];
      const float z = dot_row(reinterpret_cast<const uint4*>(ra.H) + (size_t)source_row(ra, r) * nvec,
                              reinterpret_cast<const uint4*>(ra.W), w_row_base(t, ra.d, ra.w_tiled != 0),
                              ra.w_tiled != 0, nvec, lane);
      if (lane == 0) sa.logp[t0] = z - ra.lse_row[r];
    }
  }
  __syncwarp();    // logp written by any lane is visible to the whole warp
  set_rules_warp(sa, k, lane, c0, c1);
}

// Larger unions run on the full-vocabulary tensor-core head with the union as
// its vocabulary: this kernel stages the union's rows of W contiguously (the
// head's TMA loads read a row-major [n_union, d] operand) and records each
// id's position for the pre-pass.  One warp per union row, 16-byte copies.
__global__ void __launch_bounds__(256) union_rows_kernel(const uint4* W, int V, int d, int w_tiled,
                                                         const int32_t* union_ids, int n_union, uint4* wU,
                                                         int* umap) {
  pdl_wait();      // earlier work on the stream (readers of wU and umap) is complete
  pdl_trigger();   // the pre-pass may start; it waits for this grid before anything reads wU
  const int lane = threadIdx.x & 31, nvec = d / 8;
  const bool tiled = w_tiled != 0;
  for (int u = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < n_union; u += (gridDim.x * blockDim.x) >> 5) {
    const int t = union_ids[u];
    uint4* o = wU + (size_t)u * nvec;
    if (t < 0 || t >= V) {   // reported by the pre-pass; the row is never used
      for (int k = lane; k < nvec; k += 32) o[k] = make_uint4(0, 0, 0, 0);
      continue;
    }
    if (lane == 0) umap[t] = u;
    const size_t wb = w_row_base(t, d, tiled);
    for (int k0 = lane; k0 < nvec; k0 += 32 * UR_BATCH) {   // UR_BATCH loads in flight per lane
      uint4 v[UR_BATCH];
#pragma unroll
      for (int j = 0; j < UR_BATCH; ++j)
        if (k0 + 32 * j < nvec) v[j] = W[w_vec(wb, k0 + 32 * j, tiled)];
#pragma unroll
      for (int j = 0; j < UR_BATCH; ++j)
        if (k0 + 32 * j < nvec) o[k0 + 32 * j] = v[j];
    }
  }
}

}  // namespace

cudaError_t launch_union_rows(const uint16_t* W, int V, int d, int w_tiled, const int32_t* union_ids, int n_union,
                              uint16_t* wU, int* umap, cudaStream_t st) {
  if (n_union <= 0) return cudaSuccess;
  const int blocks = (n_union + 7) / 8 < 1184 ? (n_union + 7) / 8 : 1184;   // 8 rows per block
  return launch_dependent(union_rows_kernel, dim3(blocks), dim3(256), 0, st, reinterpret_cast<const uint4*>(W), V,
                          d, w_tiled, union_ids, n_union, reinterpret_cast<uint4*>(wU), umap);
}

cudaError_t launch_restricted(const RestrictedArgs& a, cudaStream_t st) {
  if (a.N <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(RT_SPLIT * ((a.N + 15) / 16));
  cfg.blockDim = dim3(RT_THREADS);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = RT_SPLIT;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, restricted_head_kernel, a);
}

cudaError_t launch_restricted_sets(const RestrictedSetArgs& a, cudaStream_t st) {
  if (a.s.n_sets <= 0) return cudaSuccess;
  return launch_dependent(restricted_sets_kernel, dim3((a.s.n_sets + RS_WARPS - 1) / RS_WARPS),
                          dim3(32 * RS_WARPS), 0, st, a);
}

}  // namespace jet
