// Full-vocabulary scoring head on the 5th-generation tensor cores.
//
// For hidden rows H[N, d] and the output embedding W[V, d] (both bf16,
// K-major) it computes, per row r and per vocabulary split of the schedule,
//   m = max_v z[r, v],  s = sum_v exp(z[r, v] - m),     z = H W^T   (fp32)
// and writes the logit z[r, tok] of every scored token whose id falls in the
// split ("JET: Justification Evaluation in Transformer", Eq. 1-2: the
// denominator runs over the full vocabulary; GPU scoring computes it but
// transfers only the candidate log-probabilities).  The [N, V] logit matrix
// lives only in tensor memory, one 128 x 256 fp32 tile per CTA at a time.
//
// Structure (persistent CTAs, 320 threads each):
//   warp 0      TMA producer: H and W k-blocks (64 bf16 = 128 B, 128B swizzle)
//               into a shared-memory ring (stages of two k-blocks for a
//               paired head with several waves of units, else one),
//               completion on mbarriers;
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators) and
//               issues tcgen05.mma (K=16 per instruction) from one thread;
//   warps 2-9   epilogue: each thread owns one row (its TMEM lane) and half of
//               the tile's columns, reads them with tcgen05.ld, folds them into
//               a running (max, sum-exp) and picks out the logits of its row's
//               tokens while walking the row's sorted token list.
// The two accumulators let the epilogue of tile j overlap the MMAs of tile
// j+1.
//
// Paired variant (PAIR = true, clusters of two CTAs on two SMs): one
// tcgen05.mma.cta_group::2 computes a 256 x 256 tile; each CTA stages its own
// 128 rows of H and 128 of the tile's 256 W rows, so its ring (6 k-blocks)
// holds twice the W bytes of the single-CTA ring.  This is what lets few rows
// (N ~ 256, where two row tiles would otherwise share each W tile and halve
// each CTA's DRAM bytes in flight) stream W at full bandwidth.  Both CTAs'
// TMA copies complete on the issuing CTA's barrier, which expects the bytes of
// both halves, and the MMA commits are multicast back to both CTAs.
//
// Every mbarrier wait is bounded: on timeout the kernel records
// JET_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include <atomic>
#include <climits>

#include "jet_head.cuh"
#include "jet_wait.cuh"

namespace jet {
namespace {

constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;        // 2 s per wait
constexpr unsigned long long EXIT_LIMIT_NS = 3 * WAIT_LIMIT_NS;    // pair exit handshake

// ---- TMA ----------------------------------------------------------------------
// Every load carries an L2 eviction policy (createpolicy): W tiles that no
// other CTA reads are marked evict-first so that the stream of W does not push
// the row tiles, the partials and the small per-call arrays out of L2; W tiles
// that sibling row tiles of the band re-read, and the band's H tiles, are
// marked evict-last (measured on the 20k-row workload with units in counter
// order: 2% faster than evict-normal W or H, level with evict-first W).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// Paired form: the copy lands in this CTA's shared memory and completes on
// the barrier at cluster address `bar` (the issuing CTA's barrier).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// Tiled W (4-D map over [tiles][k-blocks][128 rows][64]): the box at
// (0, 0, kb, tile) is the same 128- or 256-row slice as the 2-D box at
// (64 kb, 128 tile) of row-major W, one contiguous 16 KB read per 128 rows.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int kb, int tile, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(0), "r"(kb), "r"(tile), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(void* dst, const CUtensorMap* map, int kb, int tile, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(kb), "r"(tile), "l"(policy)
      : "memory");
}

// ---- cluster ------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Cluster address of the object at the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  return remote;
}

// Arrive on the mbarrier at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint64_t* bar_local, uint32_t rank) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr(bar_local, rank))
               : "memory");
}

// Spin on %globaltimer for about `ns` nanoseconds.
__device__ __forceinline__ void settle_ns(unsigned long long ns) {
  const unsigned long long t0 = globaltimer();
  while (globaltimer() - t0 < ns) {
  }
}

// ---- unit ring (paired head, dynamic schedule) ------------------------------------
// With several waves of units, the pairs take units in order from a global
// counter instead of a fixed stride, so that the units running at any moment
// stay neighbours in the schedule (the same band of row tiles, adjacent
// vocabulary splits) however unevenly the pairs progress; their shared H and W
// tiles are then still in L2.  The issuing CTA's producer takes each unit id
// and publishes it in a small ring held by both CTAs; its MMA thread and the
// epilogue warps, and the second CTA's producer and epilogue warps, read it
// from there and free the slot on the issuing CTA's barrier.
constexpr int UR = 4;                           // ring slots
constexpr int UR_CONSUMERS = 2 * (1 + EPI_WARPS);   // per slot: see above

__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait with cluster-scope acquire: data stored by the other CTA before its
// release-arrive is visible afterwards.  Bounded like mbar_wait.
__device__ __noinline__ bool mbar_wait_acq_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                   int* err, int where, unsigned long long limit_ns) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_acq_cluster(a, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        if (err != nullptr && atomicCAS(err, 0, JET_ERR_TIMEOUT) == 0) err[2] = where;
        return false;
      }
    }
  }
}

// Issuing CTA's producer: publish unit u at ring position ui in both CTAs,
// once every consumer has read the slot's previous id.
__device__ __forceinline__ bool ring_publish(volatile int* uring, uint64_t* ufull, uint64_t* uempty, uint32_t ui,
                                             int u, volatile int* abort_flag, int* err, unsigned long long limit) {
  const uint32_t slot = ui % UR, ph = (ui / UR) & 1u;
  if (!mbar_wait_acq_cluster(&uempty[slot], ph ^ 1u, abort_flag, err, 8, limit)) return false;
  uring[slot] = u;
  mbar_arrive(&ufull[slot]);   // release (CTA scope): this CTA's consumers see the id
  const uint32_t remote = cluster_addr(const_cast<int*>(&uring[slot]), 1);
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(u) : "memory");
  mbar_arrive_cluster(&ufull[slot], 1);   // release (cluster scope): orders the store above
  return true;
}

// Consumer (one thread): the unit id at ring position ui; frees the slot on
// the issuing CTA's barrier.  INT_MAX (and ok = false) when the wait fails.
__device__ __forceinline__ int ring_take(volatile int* uring, uint64_t* ufull, uint64_t* uempty, uint32_t ui,
                                         bool in_issuer, volatile int* abort_flag, int* err, bool& ok,
                                         unsigned long long limit) {
  const uint32_t slot = ui % UR, ph = (ui / UR) & 1u;
  if (!mbar_wait_acq_cluster(&ufull[slot], ph, abort_flag, err, 9, limit)) {
    ok = false;
    return INT_MAX;
  }
  const int u = uring[slot];
  if (in_issuer) mbar_arrive(&uempty[slot]);
  else mbar_arrive_cluster(&uempty[slot], 0);
  return u;
}

// ring_take for a whole warp: lane 0 takes the id, every lane returns it.
__device__ __forceinline__ int ring_take_warp(volatile int* uring, uint64_t* ufull, uint64_t* uempty, uint32_t ui,
                                              bool in_issuer, volatile int* abort_flag, int* err, bool& ok,
                                              unsigned long long limit) {
  int u = 0, good = 1;
  if ((threadIdx.x & 31) == 0) {
    bool o = true;
    u = ring_take(uring, ufull, uempty, ui, in_issuer, abort_flag, err, o, limit);
    good = o ? 1 : 0;
  }
  u = __shfl_sync(0xffffffffu, u, 0);
  if (!__shfl_sync(0xffffffffu, good, 0)) ok = false;
  return u;
}

// ---- tcgen05 ------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  if constexpr (PAIR) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
}

template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  if constexpr (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row swizzle atoms 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);     // bits  0-13: start address >> 4
  d |= (uint64_t)(16u >> 4) << 16;               // bits 16-29: leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;             // bits 32-45: stride byte offset >> 4
  d |= (uint64_t)1 << 46;                        // bits 46-48: descriptor version 1
  d |= (uint64_t)2 << 61;                        // bits 61-63: 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// N = BN, M = 128 (one CTA) or 256 (CTA pair).
template <bool PAIR>
__host__ __device__ constexpr uint32_t idesc() {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | ((uint32_t)(BN >> 3) << 17)               // N >> 3
         | ((uint32_t)((PAIR ? 2 * BM : BM) >> 4) << 24);   // M >> 4
}

template <bool PAIR>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accum) {
  if constexpr (PAIR)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc<true>()), "r"(accum)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc<false>()), "r"(accum)
        : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed:
// in the paired variant on the barrier at that offset in both CTAs.
template <bool PAIR>
__device__ __forceinline__ void tc_commit_all(uint64_t* bar) {
  if constexpr (PAIR) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
  } else {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
  }
}

// As tc_commit_all, but only on this CTA's barrier.
template <bool PAIR>
__device__ __forceinline__ void tc_commit_local(uint64_t* bar) {
  if constexpr (PAIR)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Load 32 consecutive fp32 columns of this thread's TMEM lane, then wait for
// the load.  The wait names the destination registers as operands so that no
// use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
        "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
        "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {   // hardware 2^x (MUFU), flushes subnormals
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float LOG2E = 1.4426950408889634f;

template <bool PAIR, int KPS>
__global__ void __launch_bounds__(HEAD_THREADS, 1)
    head_lse_gather_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmW,
                           const HeadArgs a) {
  using SH = HeadShape<PAIR, KPS>;
  constexpr int NST = SH::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // 128B-swizzled operand tiles must start on 1024-byte boundaries
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + NST * SH::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + NST * SH::B_BYTES);
  uint64_t* full = bars;                  // [NST] TMA -> MMA (paired: used in the issuing CTA)
  uint64_t* empty = bars + NST;           // [NST] MMA -> TMA
  uint64_t* tfull = bars + 2 * NST;       // [2] MMA -> epilogue
  uint64_t* tempty = tfull + 2;           // [2] epilogue(s) -> MMA
  uint64_t* drain = tempty + 2;           // [1] MMA drain on abort
  uint64_t* exitb = drain + 1;            // [1] paired exit handshake
  uint64_t* ufull = exitb + 1;            // [UR] unit ring: id published
  uint64_t* uempty = ufull + UR;          // [UR] unit ring: id read by every consumer (issuing CTA's)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(uempty + UR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* uring = abort_flag + 1;   // [UR] unit ids

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_rank() : 0u;   // CTA within the pair; 0 issues the MMAs
  const bool issuer = rank == 0;
  const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int unit_step = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const bool dyn = PAIR && a.sched != nullptr;   // units after the first come from the ring
  // No early launch_dependents here: the merge kernel is launched when this
  // grid completes.  Launched early, its CTAs pile onto the SMs the head
  // leaves free and run there several times slower than when spread over all
  // SMs after the head (measured on GB300).

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);   // the issuer's arrive.expect_tx (+ both CTAs' bytes when paired)
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], EPI_WARPS * (PAIR ? 2 : 1));
    }
    mbar_init(drain, 1);
    mbar_init(exitb, 1);
    for (int i = 0; i < UR; ++i) {
      mbar_init(&ufull[i], 1);
      mbar_init(&uempty[i], UR_CONSUMERS);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if constexpr (PAIR) cluster_sync_all();   // peer barriers exist before any remote arrival
  if (warp == 1) {
    tmem_alloc<PAIR>(tmem_slot, TMEM_COLS);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const Plan& P = a.plan;
  const int kblocks = a.d / BK;
  const int tile_rows = plan_tile_rows(P);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;   // per stage: has a load, parity of its phase
      // one row tile: each W tile is read by this CTA (pair) alone; several:
      // sibling row tiles of the band read it too, so it is kept in L2
      const uint64_t pol_w = P.n_mt == 1 ? l2_policy_evict_first() : l2_policy_evict_last();
      const uint64_t pol_h = l2_policy_evict_last();
      bool ok = true;
      uint32_t ui = 0;   // unit ring position
      int u = unit0;
      if (dyn) {
        if (issuer) ok = ring_publish(uring, ufull, uempty, ui, u, abort_flag, a.err, WAIT_LIMIT_NS);
        else u = ring_take(uring, ufull, uempty, ui, false, abort_flag, a.err, ok, WAIT_LIMIT_NS);
        ++ui;
      }
      while (ok && u < P.units) {
        int m, vt0, vt1;
        plan_unit(P, u, m, vt0, vt1);
        const int a_row = m * tile_rows + (int)rank * BM;
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          if (*abort_flag) { ok = false; break; }
          const int b_row = vt * BN + (int)rank * SH::B_ROWS;
          for (int kb = 0; kb < kblocks; kb += SH::KPS) {
            const int nk = min(SH::KPS, kblocks - kb);   // k-blocks in this stage (the last may be short)
            const uint32_t bytes = (uint32_t)nk * (SH::A_KB_BYTES + SH::B_KB_BYTES);
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.err, 1, WAIT_LIMIT_NS)) { ok = false; break; }
            uint8_t* dA = sA + stage * SH::A_BYTES;
            uint8_t* dB = sB + stage * SH::B_BYTES;
            if constexpr (PAIR) {
              if (issuer) mbar_arrive_expect_tx(&full[stage], 2 * bytes);   // both CTAs' halves
              const uint32_t bar = cluster_addr(&full[stage], 0);
              for (int j = 0; j < nk; ++j) {
                tma_load_2d_pair(dA + j * SH::A_KB_BYTES, &tmH, (kb + j) * BK, a_row, bar, pol_h);
                if (a.w_tiled) tma_load_4d_pair(dB + j * SH::B_KB_BYTES, &tmW, kb + j, b_row >> 7, bar, pol_w);
                else tma_load_2d_pair(dB + j * SH::B_KB_BYTES, &tmW, (kb + j) * BK, b_row, bar, pol_w);
              }
            } else {
              mbar_arrive_expect_tx(&full[stage], bytes);
              for (int j = 0; j < nk; ++j) {
                tma_load_2d(dA + j * SH::A_KB_BYTES, &tmH, (kb + j) * BK, a_row, &full[stage], pol_h);
                if (a.w_tiled) tma_load_4d(dB + j * SH::B_KB_BYTES, &tmW, kb + j, b_row >> 7, &full[stage], pol_w);
                else tma_load_2d(dB + j * SH::B_KB_BYTES, &tmW, (kb + j) * BK, b_row, &full[stage], pol_w);
              }
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == NST) { stage = 0; phase ^= 1u; }
          }
        }
        if (!ok) break;
        if (!dyn) {
          u += unit_step;
        } else if (issuer) {
          if (ui == 1) pdl_wait();   // the pre-pass zeroes the counter
          u = unit_step + atomicAdd(a.sched, 1);
          ok = ring_publish(uring, ufull, uempty, ui, u, abort_flag, a.err, WAIT_LIMIT_NS);
          ++ui;
        } else {
          u = ring_take(uring, ufull, uempty, ui, false, abort_flag, a.err, ok, WAIT_LIMIT_NS);
          ++ui;
        }
      }
      if (ok) {
        // tail: wait until the MMA has released every stage, so that no
        // barrier arrival is still pending when the CTA exits
        for (int i = 0; i < NST; ++i) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.err, 5, WAIT_LIMIT_NS)) break;
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
      } else if (!PAIR || issuer) {
        // abort: let copies already in flight land before the CTA exits
        volatile int never = 0;
        for (int s = 0; s < NST; ++s)
          if (issued_mask & (1u << s))
            mbar_wait(&full[s], (issued_parity >> s) & 1u, &never, nullptr, 0, WAIT_LIMIT_NS);
      } else {
        // abort in the second CTA: its copies complete on the issuer's barrier,
        // which it cannot observe; give them ample time (a TMA round trip is
        // microseconds) before the exit handshake lets the pair leave
        settle_ns(200000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && issuer) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, any = false;
      uint32_t ui = 0;
      int u = dyn ? ring_take(uring, ufull, uempty, ui++, true, abort_flag, a.err, ok, WAIT_LIMIT_NS) : unit0;
      while (ok && u < P.units) {
        int m, vt0, vt1;
        plan_unit(P, u, m, vt0, vt1);
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, a.err, 2, WAIT_LIMIT_NS)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
          for (int kb = 0; kb < kblocks; kb += SH::KPS) {
            const int nk = min(SH::KPS, kblocks - kb);
            if (!mbar_wait(&full[stage], phase, abort_flag, a.err, 3, WAIT_LIMIT_NS)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < SH::KPS; ++j) {
              if (j < nk) {
                const uint32_t a0 = smem_u32(sA + stage * SH::A_BYTES + j * SH::A_KB_BYTES);
                const uint32_t b0 = smem_u32(sB + stage * SH::B_BYTES + j * SH::B_KB_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)   // 16 bf16 = 32 bytes along K per MMA
                  tc_mma<PAIR>(d_tmem, sdesc_k128(a0 + 32 * k), sdesc_k128(b0 + 32 * k), (kb | j | k) != 0);
              }
            }
            tc_commit_all<PAIR>(&empty[stage]);
            any = true;
            if (++stage == NST) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          tc_commit_all<PAIR>(&tfull[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok) break;
        u = dyn ? ring_take(uring, ufull, uempty, ui++, true, abort_flag, a.err, ok, WAIT_LIMIT_NS) : u + unit_step;
      }
      if (!ok && any) {   // wait until every MMA issued so far has completed
        volatile int never = 0;
        tc_commit_local<PAIR>(drain);
        mbar_wait(drain, 0, &never, nullptr, 0, WAIT_LIMIT_NS);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;              // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;          // column half of each tile
    const int row_in_tile = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    pdl_wait();   // row lists and the error word come from the pre-pass
    bool ok = *(volatile const int*)a.err == 0;
    if (!ok) *abort_flag = 1;   // pre-pass rejected the batch: every role stops
    uint32_t ui = 0;
    int u = unit0;
    if (dyn && ok) u = ring_take_warp(uring, ufull, uempty, ui++, issuer, abort_flag, a.err, ok, WAIT_LIMIT_NS);
    while (ok && u < P.units) {
      int m, vt0, vt1;
      plan_unit(P, u, m, vt0, vt1);
      const int row = m * tile_rows + (int)rank * BM + row_in_tile;
      const bool valid = row < a.N;
      int e = 0, e_end = 0, t_next = INT_MAX;
      if (valid) {
        e = a.row_ptr[row];
        e_end = a.row_ptr[row + 1];
        const int col_begin = vt0 * BN;
        while (e < e_end && a.row_list[e].x < col_begin) ++e;
        if (e < e_end) t_next = a.row_list[e].x;
      }
      float m_run = -INFINITY, s_run = 0.f;
      for (int vt = vt0; vt < vt1; ++vt) {
        if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, a.err, 4, WAIT_LIMIT_NS)) { ok = false; break; }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + half * 128);
        const int col0 = vt * BN + half * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          __syncwarp();                            // .sync.aligned: whole warp, converged
          tmem_ld32_wait(taddr + 32 * c, r);
          float x[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
          const int cb = col0 + 32 * c;
          if (cb + 32 > a.V) {                    // vocabulary tail: columns >= V do not exist
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cb + i >= a.V) x[i] = -INFINITY;
          }
          while (t_next < cb + 32) {               // this row's tokens in this chunk
            if (t_next >= cb) {
              const int kk = t_next - cb;
              float g = 0.f;
#pragma unroll
              for (int i = 0; i < 32; ++i) g = (i == kk) ? x[i] : g;
              a.zg[a.row_list[e].y] = g;
            }
            ++e;
            t_next = (e < e_end) ? a.row_list[e].x : INT_MAX;
          }
          float cmax = x[0];
#pragma unroll
          for (int i = 1; i < 32; ++i) cmax = fmaxf(cmax, x[i]);
          const float m_new = fmaxf(m_run, cmax);
          if (m_new != -INFINITY) {
            const float mb = m_new * LOG2E;
            float cs = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) cs += ex2(fmaf(x[i], LOG2E, -mb));
            s_run = s_run * ex2((m_run - m_new) * LOG2E) + cs;
            m_run = m_new;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR && !issuer) mbar_arrive_cluster(&tempty[acc], 0);
          else mbar_arrive(&tempty[acc]);
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (ok && valid) a.part[part_slot(P, u, (int)rank, half, row_in_tile)] = make_float2(m_run, s_run);
      if (!ok) break;
      u = dyn ? ring_take_warp(uring, ufull, uempty, ui++, issuer, abort_flag, a.err, ok, WAIT_LIMIT_NS)
              : u + unit_step;
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // neither CTA of the pair leaves while the other may still signal it or
    // read its shared memory through the MMA
    if (threadIdx.x == 0) {
      mbar_arrive_cluster(exitb, rank ^ 1u);
      volatile int never = 0;
      mbar_wait(exitb, 0, &never, a.err, 7, EXIT_LIMIT_NS);
    }
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<PAIR>(tmem_base, TMEM_COLS);
  }
}

template <bool PAIR, int KPS>
cudaError_t launch_variant(const CUtensorMap& tmH, const CUtensorMap& tmW, const HeadArgs& a, cudaStream_t st) {
  // the shared-memory attribute belongs to the function on each device
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit == 0 || (configured.load() & bit) == 0) {
    e = cudaFuncSetAttribute(head_lse_gather_kernel<PAIR, KPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             HeadShape<PAIR, KPS>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.plan.grid);
  cfg.blockDim = dim3(HEAD_THREADS);
  cfg.dynamicSmemBytes = HeadShape<PAIR, KPS>::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (PAIR) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, head_lse_gather_kernel<PAIR, KPS>, tmH, tmW, a);
}

}  // namespace

cudaError_t launch_head(const CUtensorMap& tmH, const CUtensorMap& tmW, const HeadArgs& a, cudaStream_t st) {
  if (!a.plan.pair) return launch_variant<false, 1>(tmH, tmW, a, st);
  // several waves of units (more units than pairs): stages of two k-blocks
  return a.plan.units > a.plan.grid / 2 ? launch_variant<true, 2>(tmH, tmW, a, st)
                                        : launch_variant<true, 1>(tmH, tmW, a, st);
}

}  // namespace jet
