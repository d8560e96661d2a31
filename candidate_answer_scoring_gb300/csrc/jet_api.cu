// C ABI of libjetscore: context and workspace, host-side argument checks, the
// vocabulary-split schedule, TMA tensor maps, and the launch sequences
//   full vocabulary:  [row gather ->] pre-pass -> head -> merge -> set rules
//   restricted union: restricted head -> validation + set rules
// (each launch a programmatic dependent of the previous one).
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <new>
#include <vector>

#include "jet_internal.cuh"

using namespace jet;

namespace jet {

// Choose the number of vocabulary splits S per row tile: every unit is one row
// tile over n_vt/S vocabulary tiles, G_u units run at a time (G SMs, or G/2
// CTA pairs), so the busiest CTA processes ceil(n_mt*S/G_u) * ceil(n_vt/S)
// tiles; take the smallest such count (ties: fewer splits).  Bands of Gm row
// tiles keep Gm H tiles (rows*d*2 bytes each) within ~48 MB of L2 while the
// band's units stream W.
Plan make_plan(int N, int V, int d, int G, int units_cap, bool pair) {
  Plan p;
  p.pair = pair ? 1 : 0;
  const int rows = plan_tile_rows(p);
  const int per_unit = 1 + p.pair;                 // CTAs per unit
  const int G_u = std::max(1, G / per_unit);
  p.n_mt = (N + rows - 1) / rows;
  p.n_vt = (V + BN - 1) / BN;
  const int S_max = std::max(1, std::min(p.n_vt, units_cap / (per_unit * std::max(1, p.n_mt))));
  long long best = -1;
  for (int S = 1; S <= S_max; ++S) {
    const long long waves = ((long long)p.n_mt * S + G_u - 1) / G_u;
    const long long t = waves * ((p.n_vt + S - 1) / S);
    if (best < 0 || t < best) { best = t; p.S = S; }
  }
  const long long a_tile = (long long)rows * d * 2;
  const int gm_max = (int)std::max(1LL, (48LL << 20) / a_tile);
  p.Gm = std::max(1, std::min(p.n_mt, gm_max));
  p.n_full_bands = p.n_mt / p.Gm;
  p.r_last = p.n_mt - p.n_full_bands * p.Gm;
  p.units = p.n_mt * p.S;
  p.grid = per_unit * std::min(p.units, G_u);
  return p;
}

// Diagnostic switches are read once per process; the function-local statics
// that hold them are initialised thread-safely.  Unset: -1.
static int env_switch(const char* name) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : -1;
}

// The paired head serves every batch of more than one 128-row tile: it halves
// each CTA's share of the W tile, which keeps twice the W bytes in flight per
// SM.  JETSCORE_HEAD_PAIR=0/1 forces a variant (diagnostics).
bool head_use_pair(int N) {
  static const int env = env_switch("JETSCORE_HEAD_PAIR");
  if (env >= 0) return env != 0;
  return N > BM;
}

// Dynamic unit order for the paired head when the schedule has more than one
// wave of units (JETSCORE_HEAD_DYN=0: fixed stride, diagnostics).
bool head_use_dynamic(const Plan& p) {
  static const int env = env_switch("JETSCORE_HEAD_DYN");
  if (env == 0) return false;
  return p.pair && p.units > p.grid / 2;
}

// Restricted mode on the tensor-core head (the union gathered into a staging
// copy and used as the vocabulary) for unions of at least this many codes;
// smaller unions take the two-launch mma.sync path.  JETSCORE_RESTRICTED_TC=0/1
// forces a path (diagnostics; 1 applies wherever the staging copy fits).
constexpr int RESTRICTED_TC_MIN_UNION = 192;

bool restricted_use_tc(int n_union, int staging_rows) {
  static const int env = env_switch("JETSCORE_RESTRICTED_TC");
  if (n_union > staging_rows || env == 0) return false;
  return env > 0 || n_union >= RESTRICTED_TC_MIN_UNION;
}

bool pdl_enabled() {
  static const bool on = std::getenv("JETSCORE_NO_PDL") == nullptr;
  return on;
}

}  // namespace jet

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int UNITS_PER_SM_CAP = 64;   // bound on schedule units (partials workspace)
// Restricted path: logits over the union are kept in an [N, |U|] scratch of
// max(max_rows * 128, 2^20) floats; larger products recompute the scored
// logits in the set kernel instead.
constexpr size_t ZU_FLOATS_PER_ROW = 128;
constexpr size_t ZU_FLOATS_MIN = size_t(1) << 20;
constexpr size_t IO_HEAD = 64;   // bytes of the error words at the front of the output block
constexpr int STATUS_RING = 4096;   // per-call status words of jet_score_sets_host_async between waits

template <class T>
cudaError_t dalloc(T** p, size_t n) {
  return cudaMalloc(reinterpret_cast<void**>(p), (n ? n : 1) * sizeof(T));
}

}  // namespace

struct jet_ctx {
  int device = 0, d = 0, V = 0, max_rows = 0, max_tokens = 0, num_sms = 0, units_cap = 0;
  int w_layout = JET_W_ROWMAJOR;   // how calls read their W argument
  EncodeTiledFn encode = nullptr;
  // device workspace
  int* err = nullptr;        // error words: the head of io_dev (below)
  int* row_ptr = nullptr;
  int* row_cur = nullptr;
  int2* row_list = nullptr;
  int* iscratch = nullptr;   // [max_tokens] ints (temperature fit flags)
  float* lse_row = nullptr;  // [max_rows] per-row lse handed from merge / restricted head to the set kernel
  int* umap = nullptr;       // [V] token id -> union position (restricted path)
  float* zu = nullptr;       // [zu_cap] logits over the union (restricted path)
  size_t zu_cap = 0;
  float* zg = nullptr;
  float2* part = nullptr;
  unsigned long long* hash = nullptr;
  // scratch for outputs the caller did not ask for
  float *lse = nullptr, *logp = nullptr, *s = nullptr, *q = nullptr, *qe = nullptr;
  int32_t* dec = nullptr;
  float *expd = nullptr, *conf = nullptr, *mass = nullptr;
  // [max_rows, d] staging copy of H: host inputs (jet_score_sets_host) and
  // gathered rows (jet_score_sets_gather)
  uint16_t* stH = nullptr;
  // [wU_rows, d] staging copy of the union's rows of W (restricted mode on the
  // tensor-core head); wU_rows = min(V, JET_MAX_UNION)
  uint16_t* wU = nullptr;
  int wU_rows = 0;
  // jet_score_sets_host packs the small inputs into one pinned block (one
  // copy in) and lays the requested outputs out behind the error word in one
  // device block (one copy out, status included)
  uint8_t *h_in = nullptr, *d_in = nullptr;     // pinned host / device, in_cap bytes
  uint8_t *io_dev = nullptr, *h_out = nullptr;  // device / pinned host: [IO_HEAD error words][outputs]
  size_t in_cap = 0, out_cap = 0;
  int* h_err = nullptr;   // pinned
  // jet_score_sets_host_async: the second staging slot (slot 0 is stH/d_in),
  // the copy stream, per-slot events, and the per-call status words (pinned)
  uint16_t* stH2 = nullptr;
  uint8_t* d_in2 = nullptr;
  cudaStream_t copy_st = nullptr;
  cudaEvent_t ev_copied[2] = {nullptr, nullptr};   // slot's inputs are on the device
  cudaEvent_t ev_free[2] = {nullptr, nullptr};     // the kernels reading the slot are done
  int* h_status = nullptr;                         // [STATUS_RING]
  int n_async = 0;                                 // calls since the last jet_host_wait
  int async_err = 0;                               // first status seen by an implicit wait
  unsigned long long async_calls = 0;              // slot of the next call = its parity
  // row deduplication workspace
  unsigned long long *dd_hash = nullptr, *dd_keys = nullptr;
  int *dd_vals = nullptr, *dd_rep = nullptr, *dd_rank = nullptr, *dd_tiles = nullptr;
  int dd_table = 0;
  // temperature fitting
  double *fit_res = nullptr, *h_fit = nullptr;   // device [3], pinned host [3]
  // schedule cache
  int plan_rows = -1, plan_V = -1;
  Plan plan;
  // kernel timing (jet_profile_enable)
  bool prof = false;
  std::vector<cudaEvent_t> ev[5];   // pairs: start, stop
  size_t ev_used[5] = {0, 0, 0, 0, 0};
  double launches[5] = {0, 0, 0, 0, 0};
  double untimed = 0;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = (cudaSetDevice(dev) == cudaSuccess);
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

int cuda_status(cudaError_t e) { return e == cudaSuccess ? JET_OK : JET_ERR_CUDA; }

enum { K_PREP = 0, K_HEAD = 1, K_MERGE = 2, K_RESTRICTED = 3, K_SETS = 4 };
constexpr size_t PROF_PAIRS = 65536;

// Event pair around one launch when timing is on; returns the pair's slot or -1.
long prof_begin(jet_ctx* c, int kind, cudaStream_t st) {
  if (!c->prof) return -1;
  c->launches[kind] += 1;
  std::vector<cudaEvent_t>& v = c->ev[kind];
  if (c->ev_used[kind] + 2 > 2 * PROF_PAIRS) { c->untimed += 1; return -1; }
  while (v.size() < c->ev_used[kind] + 2) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) { c->untimed += 1; return -1; }
    v.push_back(e);
  }
  const long slot = (long)c->ev_used[kind];
  c->ev_used[kind] += 2;
  cudaEventRecord(v[slot], st);
  return slot;
}

void prof_end(jet_ctx* c, int kind, long slot, cudaStream_t st) {
  if (slot >= 0) cudaEventRecord(c->ev[kind][slot + 1], st);
}

struct ProfScope {
  jet_ctx* c; int kind; long slot; cudaStream_t st;
  ProfScope(jet_ctx* c_, int k, cudaStream_t s) : c(c_), kind(k), slot(prof_begin(c_, k, s)), st(s) {}
  ~ProfScope() { prof_end(c, kind, slot, st); }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tiled W (jetscore.h, "Tiled weights"): dims (64, 128 rows, d/64 k-blocks,
// ceil(V/128) tiles), one box = box_rows rows of one k-block (box_rows/128 tiles).
int encode_tiled_w(jet_ctx* c, CUtensorMap* map, const void* base, int box_rows) {
  const cuuint64_t dims[4] = {64, 128, (cuuint64_t)c->d / 64, (cuuint64_t)(c->V + 127) / 128};
  const cuuint64_t strides[3] = {128, 128 * 128, (cuuint64_t)c->d / 64 * 128 * 128};
  const cuuint32_t box[4] = {64, 128, 1, (cuuint32_t)box_rows / 128};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = c->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? JET_OK : JET_ERR_CUDA;
}

int encode_kmajor(jet_ctx* c, CUtensorMap* map, const void* base, int rows, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)c->d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)c->d * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = c->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? JET_OK : JET_ERR_CUDA;
}

const Plan& plan_for(jet_ctx* c, int n_rows, int V) {
  if (c->plan_rows != n_rows || c->plan_V != V) {
    c->plan = make_plan(n_rows, V, c->d, c->num_sms, c->units_cap, head_use_pair(n_rows));
    c->plan_rows = n_rows;
    c->plan_V = V;
  }
  return c->plan;
}

// Tensor-core head and merge for the rows/tokens the pre-pass listed, over
// the V rows of W (the full vocabulary in the caller's layout, or the staged
// union, row-major).  lse_row NULL: one token per row, logp[r] written by the
// merge; else the merge leaves each row's lse in lse_row for the set kernel.
int run_full_head(jet_ctx* c, const void* H, const void* W, int V, bool w_tiled, int n_rows, float* logp,
                  float* lse, float* lse_row, cudaStream_t st) {
  const Plan& plan = plan_for(c, n_rows, V);
  CUtensorMap tmH, tmW;
  int rc = encode_kmajor(c, &tmH, H, n_rows, BM);
  if (rc != JET_OK) return rc;
  const int w_box = plan.pair ? HeadShape<true>::B_ROWS : HeadShape<false>::B_ROWS;
  rc = w_tiled ? encode_tiled_w(c, &tmW, W, w_box) : encode_kmajor(c, &tmW, W, V, w_box);
  if (rc != JET_OK) return rc;
  HeadArgs ha;
  ha.N = n_rows;
  ha.V = V;
  ha.d = c->d;
  ha.plan = plan;
  ha.row_ptr = c->row_ptr;
  ha.row_list = c->row_list;
  ha.zg = c->zg;
  ha.part = c->part;
  ha.err = c->err;
  ha.w_tiled = w_tiled ? 1 : 0;
  ha.sched = head_use_dynamic(plan) ? c->err + SCHED_WORD : nullptr;
  cudaError_t e;
  {
    ProfScope ps(c, K_HEAD, st);
    e = launch_head(tmH, tmW, ha, st);
  }
  if (e != cudaSuccess) return JET_ERR_CUDA;
  MergeArgs ma;
  ma.N = n_rows;
  ma.plan = ha.plan;
  ma.part = c->part;
  ma.zg = c->zg;
  ma.lse = lse;
  ma.lse_row = lse_row;
  ma.logp = logp;
  ma.err = c->err;
  ProfScope ps(c, K_MERGE, st);
  return cuda_status(launch_merge(ma, st));
}

int check_sets_args(jet_ctx* c, const void* H, const void* W, int n_rows, const int32_t* tok_row,
                    const int32_t* tok_ids, int n_tok, const int32_t* cand_offsets, int n_cand,
                    const int32_t* set_offsets, const uint8_t* kind, int n_sets, float T, int mode,
                    const int32_t* union_ids, int n_union) {
  if (!c) return JET_ERR_ARG;
  if (n_rows < 0 || n_tok < 0 || n_cand < 0 || n_sets < 0) return JET_ERR_ARG;
  if (!(T > 0.f) || !std::isfinite(T)) return JET_ERR_ARG;
  if (mode != JET_MODE_FULL && mode != JET_MODE_RESTRICTED) return JET_ERR_MODE;
  if (n_tok == 0) return (n_cand == 0 && n_sets == 0) ? JET_OK : JET_ERR_OFFSETS;
  if (n_cand < 1 || n_sets < 1 || n_cand > n_tok || n_sets > n_cand) return JET_ERR_OFFSETS;
  if (n_rows < 1) return JET_ERR_ARG;
  if (n_rows > c->max_rows || n_tok > c->max_tokens) return JET_ERR_WORKSPACE;
  if (!H || !W || !tok_row || !tok_ids || !cand_offsets || !set_offsets || !kind) return JET_ERR_ARG;
  if (!aligned16(H) || !aligned16(W)) return JET_ERR_ARG;
  if (mode == JET_MODE_RESTRICTED && (!union_ids || n_union < 1 || n_union > JET_MAX_UNION)) return JET_ERR_ARG;
  return JET_OK;
}

int score_sets_enqueue(jet_ctx* c, const void* H, const void* W, int n_rows, const int32_t* tok_row,
                       const int32_t* tok_ids, int n_tok, const int32_t* cand_offsets, int n_cand,
                       const int32_t* set_offsets, const uint8_t* kind, int n_sets, float T, int mode,
                       const int32_t* union_ids, int n_union, const jet_set_out* out, cudaStream_t st,
                       const int32_t* row_index = nullptr, int n_src = 0) {
  jet_set_out o;
  std::memset(&o, 0, sizeof o);
  if (out) o = *out;

  SetArgs sa;
  sa.n_sets = n_sets;
  sa.logp = o.logp ? o.logp : c->logp;
  sa.tok_ids = tok_ids;
  sa.cand_offsets = cand_offsets;
  sa.set_offsets = set_offsets;
  sa.T = T;
  sa.s = o.s ? o.s : c->s;
  sa.q = o.q ? o.q : c->q;
  sa.q_equiv = o.q_equiv ? o.q_equiv : c->qe;
  sa.decision = o.decision ? o.decision : c->dec;
  sa.expected = o.expected ? o.expected : c->expd;
  sa.confidence = o.confidence ? o.confidence : c->conf;
  sa.mass = o.mass ? o.mass : c->mass;
  sa.hash = c->hash;
  sa.zg = nullptr;
  sa.lse_row = nullptr;
  sa.tok_row = nullptr;
  sa.err = c->err;

  // restricted mode over a large union: the union's rows of W are staged and
  // the tensor-core head runs with the union as its vocabulary
  const bool union_tc = mode == JET_MODE_RESTRICTED && restricted_use_tc(n_union, c->wU_rows);
  if (mode == JET_MODE_RESTRICTED && !union_tc) {
    // restricted head (zeroes the error word), then validation + set rules
    RestrictedSetArgs rs;
    RestrictedArgs& ra = rs.r;
    ra.N = n_rows;
    ra.d = c->d;
    ra.V = c->V;
    ra.n_union = n_union;
    ra.num_sms = c->num_sms;
    ra.H = static_cast<const uint16_t*>(H);
    ra.W = static_cast<const uint16_t*>(W);
    ra.union_ids = union_ids;
    ra.row_index = row_index;
    ra.n_src = n_src;
    ra.w_tiled = c->w_layout == JET_W_TILED ? 1 : 0;
    ra.zu = (size_t)n_rows * (size_t)n_union <= c->zu_cap ? c->zu : nullptr;
    ra.lse_row = c->lse_row;
    ra.lse = o.lse;
    ra.umap = c->umap;
    ra.err = c->err;
    rs.s = sa;
    rs.n_cand = n_cand;
    rs.n_tok = n_tok;
    rs.tok_row = tok_row;
    rs.kind = kind;
    {
      ProfScope ps(c, K_RESTRICTED, st);
      if (launch_restricted(ra, st) != cudaSuccess) return JET_ERR_CUDA;
    }
    ProfScope ps(c, K_SETS, st);
    return cuda_status(launch_restricted_sets(rs, st));
  }

  if (row_index) {
    // gathered rows: compact copy for the head's tiled loads (staging buffer)
    ProfScope ps(c, K_PREP, st);
    if (launch_gather_rows(static_cast<const uint16_t*>(H), n_src, row_index, n_rows, c->d, c->stH, st) !=
        cudaSuccess)
      return JET_ERR_CUDA;
  }
  if (union_tc) {
    ProfScope ps(c, K_PREP, st);
    if (launch_union_rows(static_cast<const uint16_t*>(W), c->V, c->d, c->w_layout == JET_W_TILED ? 1 : 0,
                          union_ids, n_union, c->wU, c->umap, st) != cudaSuccess)
      return JET_ERR_CUDA;
  }
  PrepArgs pa;
  pa.n_rows = n_rows;
  pa.n_tok = n_tok;
  pa.V = c->V;
  pa.row_index = row_index;
  pa.n_src = n_src;
  pa.tok_row = tok_row;
  pa.tok_ids = tok_ids;
  pa.cand_offsets = cand_offsets;
  pa.n_cand = n_cand;
  pa.set_offsets = set_offsets;
  pa.kind = kind;
  pa.n_sets = n_sets;
  pa.row_ptr = c->row_ptr;
  pa.row_cur = c->row_cur;
  pa.row_list = c->row_list;
  pa.err = c->err;
  if (union_tc) {
    pa.union_ids = union_ids;
    pa.n_union = n_union;
    pa.umap = c->umap;
  }
  {
    ProfScope ps(c, K_PREP, st);
    if (launch_prep(pa, st) != cudaSuccess) return JET_ERR_CUDA;
  }
  const void* Hs = row_index ? static_cast<const void*>(c->stH) : H;
  const int rc = union_tc ? run_full_head(c, Hs, c->wU, n_union, false, n_rows, sa.logp, o.lse, c->lse_row, st)
                          : run_full_head(c, Hs, W, c->V, c->w_layout == JET_W_TILED, n_rows, sa.logp, o.lse,
                                          c->lse_row, st);
  if (rc != JET_OK) return rc;
  sa.zg = c->zg;            // logp = z - lse(row), formed by the set kernel
  sa.lse_row = c->lse_row;
  sa.tok_row = tok_row;
  ProfScope ps(c, K_SETS, st);
  return cuda_status(launch_sets(sa, st));
}

// Host-buffer entries: the caller's requested outputs (*out_host, host
// pointers; NULL members not wanted) get device places behind the error words
// in the context's output block, 16-byte aligned; *h receives the host
// pointers, *dev the device ones.  Returns the bytes of the block in use.
size_t place_host_outputs(jet_ctx* c, const jet_set_out* out_host, int n_rows, int n_tok, int n_cand, int n_sets,
                          jet_set_out* h, jet_set_out* dev) {
  std::memset(h, 0, sizeof *h);
  if (out_host) *h = *out_host;
  std::memset(dev, 0, sizeof *dev);
  size_t off = IO_HEAD;
  auto place = [&](void* host_ptr, size_t bytes) -> uint8_t* {
    if (!host_ptr) return nullptr;
    uint8_t* p = c->io_dev + off;
    off += (bytes + 15) & ~size_t(15);
    return p;
  };
  dev->logp = reinterpret_cast<float*>(place(h->logp, (size_t)n_tok * 4));
  dev->lse = reinterpret_cast<float*>(place(h->lse, (size_t)n_rows * 4));
  dev->s = reinterpret_cast<float*>(place(h->s, (size_t)n_cand * 4));
  dev->q = reinterpret_cast<float*>(place(h->q, (size_t)n_cand * 4));
  dev->q_equiv = reinterpret_cast<float*>(place(h->q_equiv, (size_t)n_cand * 4));
  dev->decision = reinterpret_cast<int32_t*>(place(h->decision, (size_t)n_sets * 4));
  dev->expected = reinterpret_cast<float*>(place(h->expected, (size_t)n_sets * 4));
  dev->confidence = reinterpret_cast<float*>(place(h->confidence, (size_t)n_sets * 4));
  dev->mass = reinterpret_cast<float*>(place(h->mass, (size_t)n_sets * 4));
  return off;
}

int read_status(jet_ctx* c, cudaStream_t st) {
  if (cudaMemcpyAsync(c->h_err, c->err, ERR_WORDS * sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return JET_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return JET_ERR_CUDA;
  return c->h_err[0];
}

}  // namespace

extern "C" {

const char* jet_status_string(int status) {
  switch (status) {
    case JET_OK: return "ok";
    case JET_ERR_ARG: return "invalid argument";
    case JET_ERR_TOKEN_RANGE: return "token id or row index out of range";
    case JET_ERR_OFFSETS: return "invalid candidate or set offsets";
    case JET_ERR_MODE: return "invalid mode, or multi-token candidate in restricted mode";
    case JET_ERR_NOT_IN_UNION: return "candidate token not in the union, or repeated union id";
    case JET_ERR_WORKSPACE: return "batch larger than the context workspace";
    case JET_ERR_UNSUPPORTED: return "device is not a GB300 (sm_103)";
    case JET_ERR_CUDA: return "CUDA runtime error";
    case JET_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int jet_create(jet_ctx** out, int d, int V, int max_rows, int max_tokens, int device) {
  if (!out) return JET_ERR_ARG;
  *out = nullptr;
  if (d < 64 || d > 16384 || d % 64 != 0 || V < 1 || max_rows < 1 || max_tokens < 1) return JET_ERR_ARG;
  DeviceGuard g(device);
  if (!g.ok) return JET_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return JET_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return JET_ERR_UNSUPPORTED;

  jet_ctx* c = new (std::nothrow) jet_ctx;
  if (!c) return JET_ERR_CUDA;
  c->device = device;
  c->d = d;
  c->V = V;
  c->max_rows = max_rows;
  c->max_tokens = max_tokens;
  c->num_sms = prop.multiProcessorCount;
  c->units_cap = std::max(UNITS_PER_SM_CAP * c->num_sms, (max_rows + BM - 1) / BM);

  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    delete c;
    return JET_ERR_CUDA;
  }
  c->encode = reinterpret_cast<EncodeTiledFn>(fn);

  const size_t R = (size_t)max_rows, Tk = (size_t)max_tokens;
  cudaError_t e = cudaSuccess;
  auto A = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
  c->out_cap = IO_HEAD + (8 * Tk + R) * 4 + 9 * 16;   // the nine outputs, each 16-byte aligned
  c->in_cap = (4 * Tk + 2 + JET_MAX_UNION) * 4 + Tk + 6 * 16;   // rows, ids, two offset arrays, union, kind
  A(dalloc(&c->io_dev, c->out_cap));
  c->err = reinterpret_cast<int*>(c->io_dev);   // the error words head the output block
  A(dalloc(&c->row_ptr, R + 1));
  A(dalloc(&c->row_cur, R + 1));
  A(dalloc(&c->row_list, Tk));
  A(dalloc(&c->iscratch, Tk));
  A(dalloc(&c->lse_row, R));
  A(dalloc(&c->umap, (size_t)V));
  c->zu_cap = std::max(R * ZU_FLOATS_PER_ROW, ZU_FLOATS_MIN);
  A(dalloc(&c->zu, c->zu_cap));
  A(dalloc(&c->zg, Tk));
  A(dalloc(&c->part, (size_t)c->units_cap * 2 * BM));
  A(dalloc(&c->hash, Tk));
  A(dalloc(&c->lse, R));
  A(dalloc(&c->logp, Tk));
  A(dalloc(&c->s, Tk));
  A(dalloc(&c->q, Tk));
  A(dalloc(&c->qe, Tk));
  A(dalloc(&c->dec, Tk));
  A(dalloc(&c->expd, Tk));
  A(dalloc(&c->conf, Tk));
  A(dalloc(&c->mass, Tk));
  A(dalloc(&c->stH, R * (size_t)d));
  c->wU_rows = std::min(V, JET_MAX_UNION);
  A(dalloc(&c->wU, (size_t)c->wU_rows * d));
  A(dalloc(&c->d_in, c->in_cap));
  A(cudaMallocHost(reinterpret_cast<void**>(&c->h_in), c->in_cap));
  A(cudaMallocHost(reinterpret_cast<void**>(&c->h_out), c->out_cap));
  c->dd_table = 1;
  while (c->dd_table < 2 * max_rows) c->dd_table <<= 1;
  A(dalloc(&c->dd_hash, R));
  A(dalloc(&c->dd_keys, (size_t)c->dd_table));
  A(dalloc(&c->dd_vals, (size_t)c->dd_table));
  A(dalloc(&c->dd_rep, R));
  A(dalloc(&c->dd_rank, R + 1));
  A(dalloc(&c->dd_tiles, R / 1024 + 1));
  A(dalloc(&c->fit_res, 3));
  A(cudaMallocHost(reinterpret_cast<void**>(&c->h_fit), 3 * sizeof(double)));
  A(cudaMallocHost(reinterpret_cast<void**>(&c->h_err), 2 * ERR_WORDS * sizeof(int)));   // + result words
  A(cudaMemset(c->err, 0, (SCHED_WORD + 1) * sizeof(int)));
  if (e != cudaSuccess) {
    jet_destroy(c);
    return JET_ERR_CUDA;
  }
  *out = c;
  return JET_OK;
}

void jet_destroy(jet_ctx* c) {
  if (!c) return;
  DeviceGuard g(c->device);
  cudaDeviceSynchronize();
  void* ptrs[] = {c->io_dev, c->row_ptr, c->row_cur, c->row_list, c->iscratch, c->lse_row, c->umap, c->zu, c->zg, c->part, c->hash,
                  c->lse, c->logp, c->s, c->q, c->qe, c->dec, c->expd, c->conf, c->mass, c->stH, c->wU,
                  c->d_in,
                  c->dd_hash, c->dd_keys, c->dd_vals, c->dd_rep, c->dd_rank, c->dd_tiles};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  for (auto& v : c->ev)
    for (cudaEvent_t e : v) cudaEventDestroy(e);
  for (int i = 0; i < 2; ++i) {
    if (c->ev_copied[i]) cudaEventDestroy(c->ev_copied[i]);
    if (c->ev_free[i]) cudaEventDestroy(c->ev_free[i]);
  }
  if (c->copy_st) cudaStreamDestroy(c->copy_st);
  if (c->stH2) cudaFree(c->stH2);
  if (c->d_in2) cudaFree(c->d_in2);
  if (c->h_status) cudaFreeHost(c->h_status);
  if (c->h_err) cudaFreeHost(c->h_err);
  if (c->h_in) cudaFreeHost(c->h_in);
  if (c->h_out) cudaFreeHost(c->h_out);
  if (c->h_fit) cudaFreeHost(c->h_fit);
  if (c->fit_res) cudaFree(c->fit_res);
  delete c;
}

int jet_dedup_rows(jet_ctx* c, const void* H, int n_rows, const int32_t* tok_row, int n_tok, void* H_unique,
                   int32_t* tok_row_unique, int32_t* row_map, int* n_unique, void* stream) {
  if (!c || !n_unique || n_rows < 1 || n_tok < 0) return JET_ERR_ARG;
  if (n_rows > c->max_rows || n_tok > c->max_tokens) return JET_ERR_WORKSPACE;
  if (!H || !H_unique || (n_tok > 0 && (!tok_row || !tok_row_unique))) return JET_ERR_ARG;
  if (!aligned16(H) || !aligned16(H_unique)) return JET_ERR_ARG;
  const size_t bytes = (size_t)n_rows * c->d * 2;
  const uintptr_t h0 = reinterpret_cast<uintptr_t>(H), u0 = reinterpret_cast<uintptr_t>(H_unique);
  if (h0 < u0 + bytes && u0 < h0 + bytes) return JET_ERR_ARG;   // must not overlap
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int table = 1;
  while (table < 2 * n_rows) table <<= 1;
  DedupArgs a;
  a.n_rows = n_rows;
  a.d = c->d;
  a.n_tok = n_tok;
  a.H = static_cast<const uint16_t*>(H);
  a.tok_row = tok_row;
  a.H_unique = static_cast<uint16_t*>(H_unique);
  a.tok_row_unique = tok_row_unique;
  a.row_map = row_map;
  a.hash = c->dd_hash;
  a.keys = c->dd_keys;
  a.vals = c->dd_vals;
  a.table = table;
  a.rep = c->dd_rep;
  a.rank = c->dd_rank;
  a.tile_count = c->dd_tiles;
  a.err = c->err;
  if (launch_dedup(a, st) != cudaSuccess) {
    cudaStreamSynchronize(st);
    return JET_ERR_CUDA;
  }
  int* h_count = c->h_err + ERR_WORDS;   // pinned word after the error block
  if (cudaMemcpyAsync(h_count, c->dd_rank + n_rows, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return JET_ERR_CUDA;
  const int rc = read_status(c, st);
  if (rc == JET_OK) *n_unique = *h_count;
  return rc;
}

int jet_fit_temperature(jet_ctx* c, const float* s, const int32_t* tok_ids, int n_tok, const int32_t* cand_offsets,
                        int n_cand, const int32_t* set_offsets, int n_sets, const int32_t* gold, double T_min,
                        double T_max, double* T_out, double* nll_out, void* stream) {
  if (!c || !s || !tok_ids || !cand_offsets || !set_offsets || !gold || !T_out) return JET_ERR_ARG;
  if (n_sets < 1 || n_cand < n_sets || n_tok < n_cand) return JET_ERR_OFFSETS;
  if (n_tok > c->max_tokens) return JET_ERR_WORKSPACE;
  if (!(T_min > 0.0) || !(T_max > T_min) || !std::isfinite(T_max)) return JET_ERR_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  FitArgs a;
  a.n_sets = n_sets;
  a.n_cand = n_cand;
  a.n_tok = n_tok;
  a.s = s;
  a.tok_ids = tok_ids;
  a.cand_offsets = cand_offsets;
  a.set_offsets = set_offsets;
  a.gold = gold;
  a.T_min = T_min;
  a.T_max = T_max;
  a.flags = reinterpret_cast<uint8_t*>(c->iscratch);   // [max_tokens] ints of scratch, n_cand bytes used
  a.result = c->fit_res;
  a.err = c->err;
  if (launch_fit_temperature(a, st) != cudaSuccess) {
    cudaStreamSynchronize(st);
    return JET_ERR_CUDA;
  }
  if (cudaMemcpyAsync(c->h_fit, c->fit_res, 3 * sizeof(double), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return JET_ERR_CUDA;
  const int rc = read_status(c, st);
  if (rc == JET_OK) {
    *T_out = c->h_fit[0];
    if (nll_out) *nll_out = c->h_fit[1];
  }
  return rc;
}

int jet_layer_sensitivity(jet_ctx* c, const float* z, const float* z_skip, const int32_t* offsets, int n_inputs,
                          int total, int L, int k, float* d, float* J, int32_t* selected, void* stream) {
  if (!c || !z || !z_skip || !offsets || !d || !J || n_inputs < 1 || total < n_inputs || L < 1 || k < 0 || k > L)
    return JET_ERR_ARG;
  if (k > 0 && !selected) return JET_ERR_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SensArgs a;
  a.n_inputs = n_inputs;
  a.L = L;
  a.total = total;
  a.k = k;
  a.z = z;
  a.z_skip = z_skip;
  a.offsets = offsets;
  a.d = d;
  a.J = J;
  a.selected = selected;
  a.err = c->err;
  if (launch_sensitivity(a, st) != cudaSuccess) {
    cudaStreamSynchronize(st);
    return JET_ERR_CUDA;
  }
  return read_status(c, st);
}

int jet_profile_enable(jet_ctx* c, int enable) {
  if (!c) return JET_ERR_ARG;
  c->prof = enable != 0;
  return JET_OK;
}

int jet_profile_read(jet_ctx* c, double* out, int n_out) {
  if (!c || !out || n_out < 10) return JET_ERR_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  int rc = JET_OK;
  for (int k = 0; k < 5; ++k) {
    double ms_total = 0;
    for (size_t i = 0; i + 1 < c->ev_used[k]; i += 2) {
      float ms = 0.f;
      if (cudaEventSynchronize(c->ev[k][i + 1]) != cudaSuccess ||
          cudaEventElapsedTime(&ms, c->ev[k][i], c->ev[k][i + 1]) != cudaSuccess) {
        rc = JET_ERR_CUDA;
        continue;
      }
      ms_total += ms;
    }
    out[2 * k] = c->launches[k];
    out[2 * k + 1] = ms_total;
    c->ev_used[k] = 0;
    c->launches[k] = 0;
  }
  if (n_out > 10) out[10] = c->untimed;
  c->untimed = 0;
  return rc;
}

int jet_selftest_wait_timeout(jet_ctx* c, int limit_us, void* stream) {
  if (!c || limit_us < 1 || limit_us > 2000000) return JET_ERR_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_wait_selftest(c->err, 1000ull * (unsigned long long)limit_us, st) != cudaSuccess) return JET_ERR_CUDA;
  if (cudaMemcpyAsync(c->h_err, c->err, ERR_WORDS * sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return JET_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return JET_ERR_CUDA;
  return (c->h_err[0] == JET_ERR_TIMEOUT && c->h_err[2] == 99) ? JET_ERR_TIMEOUT : JET_ERR_CUDA;
}

int jet_plan_info(jet_ctx* c, int n_rows, int* info) {
  if (!c || !info || n_rows < 1 || n_rows > c->max_rows) return JET_ERR_ARG;
  const Plan& p = plan_for(c, n_rows, c->V);
  const int v[8] = {p.n_mt, p.n_vt, p.S, p.Gm, p.units, p.grid, plan_tile_rows(p), BN};
  std::memcpy(info, v, sizeof v);
  return JET_OK;
}

int jet_score_sets_async(jet_ctx* c, const void* H, const void* W, int n_rows, const int32_t* tok_row,
                         const int32_t* tok_ids, int n_tok, const int32_t* cand_offsets, int n_cand,
                         const int32_t* set_offsets, const uint8_t* kind, int n_sets, float T, int mode,
                         const int32_t* union_ids, int n_union, const jet_set_out* out, void* stream) {
  int rc = check_sets_args(c, H, W, n_rows, tok_row, tok_ids, n_tok, cand_offsets, n_cand, set_offsets, kind,
                           n_sets, T, mode, union_ids, n_union);
  if (rc != JET_OK || n_tok == 0) return rc;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  return score_sets_enqueue(c, H, W, n_rows, tok_row, tok_ids, n_tok, cand_offsets, n_cand, set_offsets, kind,
                            n_sets, T, mode, union_ids, n_union, out, static_cast<cudaStream_t>(stream));
}

int jet_sync_status(jet_ctx* c, void* stream) {
  if (!c) return JET_ERR_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  return read_status(c, static_cast<cudaStream_t>(stream));
}

size_t jet_tiled_weights_bytes(const jet_ctx* c) {
  if (!c) return 0;
  return (size_t)((c->V + 127) / 128) * 128 * (size_t)c->d * 2;
}

int jet_tile_weights(jet_ctx* c, const void* W, void* W_tiled, void* stream) {
  if (!c || !W || !W_tiled || !aligned16(W) || !aligned16(W_tiled)) return JET_ERR_ARG;
  const uintptr_t w0 = reinterpret_cast<uintptr_t>(W), t0 = reinterpret_cast<uintptr_t>(W_tiled);
  const uintptr_t w1 = w0 + (size_t)c->V * c->d * 2, t1 = t0 + jet_tiled_weights_bytes(c);
  if (w0 < t1 && t0 < w1) return JET_ERR_ARG;   // overlap
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  return cuda_status(launch_tile_weights(static_cast<const uint16_t*>(W), c->V, c->d,
                                         static_cast<uint16_t*>(W_tiled), static_cast<cudaStream_t>(stream)));
}

int jet_set_weights_layout(jet_ctx* c, int layout) {
  if (!c || (layout != JET_W_ROWMAJOR && layout != JET_W_TILED)) return JET_ERR_ARG;
  c->w_layout = layout;
  return JET_OK;
}

int jet_score_sets_gather_async(jet_ctx* c, const void* H_src, int n_src_rows, const int32_t* row_index,
                                int n_rows, const void* W, const int32_t* tok_row, const int32_t* tok_ids,
                                int n_tok, const int32_t* cand_offsets, int n_cand, const int32_t* set_offsets,
                                const uint8_t* kind, int n_sets, float T, int mode, const int32_t* union_ids,
                                int n_union, const jet_set_out* out, void* stream) {
  const int rc = check_sets_args(c, H_src, W, n_rows, tok_row, tok_ids, n_tok, cand_offsets, n_cand, set_offsets,
                                 kind, n_sets, T, mode, union_ids, n_union);
  if (rc != JET_OK || n_tok == 0) return rc;
  if (!row_index || n_src_rows < 1 || (reinterpret_cast<uintptr_t>(row_index) & 3u) != 0) return JET_ERR_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  return score_sets_enqueue(c, H_src, W, n_rows, tok_row, tok_ids, n_tok, cand_offsets, n_cand, set_offsets, kind,
                            n_sets, T, mode, union_ids, n_union, out, static_cast<cudaStream_t>(stream), row_index,
                            n_src_rows);
}

int jet_score_sets_gather(jet_ctx* c, const void* H_src, int n_src_rows, const int32_t* row_index, int n_rows,
                          const void* W, const int32_t* tok_row, const int32_t* tok_ids, int n_tok,
                          const int32_t* cand_offsets, int n_cand, const int32_t* set_offsets, const uint8_t* kind,
                          int n_sets, float T, int mode, const int32_t* union_ids, int n_union,
                          const jet_set_out* out, void* stream) {
  const int rc = jet_score_sets_gather_async(c, H_src, n_src_rows, row_index, n_rows, W, tok_row, tok_ids, n_tok,
                                             cand_offsets, n_cand, set_offsets, kind, n_sets, T, mode, union_ids,
                                             n_union, out, stream);
  if (rc != JET_OK || n_tok == 0) {
    if (rc == JET_ERR_CUDA && c) cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    return rc;
  }
  return read_status(c, static_cast<cudaStream_t>(stream));
}

int jet_score_sets(jet_ctx* c, const void* H, const void* W, int n_rows, const int32_t* tok_row,
                   const int32_t* tok_ids, int n_tok, const int32_t* cand_offsets, int n_cand,
                   const int32_t* set_offsets, const uint8_t* kind, int n_sets, float T, int mode,
                   const int32_t* union_ids, int n_union, const jet_set_out* out, void* stream) {
  int rc = check_sets_args(c, H, W, n_rows, tok_row, tok_ids, n_tok, cand_offsets, n_cand, set_offsets, kind,
                           n_sets, T, mode, union_ids, n_union);
  if (rc != JET_OK || n_tok == 0) return rc;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = score_sets_enqueue(c, H, W, n_rows, tok_row, tok_ids, n_tok, cand_offsets, n_cand, set_offsets, kind,
                          n_sets, T, mode, union_ids, n_union, out, st);
  if (rc != JET_OK) {
    cudaStreamSynchronize(st);
    return rc;
  }
  return read_status(c, st);
}

int jet_score_tokens(jet_ctx* c, const void* H, const void* W, const int32_t* tok_ids, int n_pos, float* logp,
                     float* lse, void* stream) {
  if (!c || n_pos < 0) return JET_ERR_ARG;
  if (n_pos == 0) return JET_OK;
  if (!H || !W || !tok_ids || !logp || !aligned16(H) || !aligned16(W)) return JET_ERR_ARG;
  if (n_pos > c->max_rows || n_pos > c->max_tokens) return JET_ERR_WORKSPACE;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PrepArgs pa;
  std::memset(&pa, 0, sizeof pa);
  pa.n_rows = n_pos;
  pa.n_tok = n_pos;
  pa.V = c->V;
  pa.tok_row = nullptr;   // token i is predicted by row i
  pa.tok_ids = tok_ids;
  pa.row_ptr = c->row_ptr;
  pa.row_cur = c->row_cur;
  pa.row_list = c->row_list;
  pa.err = c->err;
  {
    ProfScope ps(c, K_PREP, st);
    if (launch_prep(pa, st) != cudaSuccess) return JET_ERR_CUDA;
  }
  int rc = run_full_head(c, H, W, c->V, c->w_layout == JET_W_TILED, n_pos, logp, lse, nullptr, st);
  if (rc != JET_OK) {
    cudaStreamSynchronize(st);
    return rc;
  }
  return read_status(c, st);
}

int jet_score_sets_host(jet_ctx* c, const void* H, const void* W, int n_rows, const int32_t* tok_row,
                        const int32_t* tok_ids, int n_tok, const int32_t* cand_offsets, int n_cand,
                        const int32_t* set_offsets, const uint8_t* kind, int n_sets, float T, int mode,
                        const int32_t* union_ids, int n_union, const jet_set_out* out_host, void* stream) {
  int rc = check_sets_args(c, H, W, n_rows, tok_row, tok_ids, n_tok, cand_offsets, n_cand, set_offsets, kind,
                           n_sets, T, mode, union_ids, n_union);
  if (rc != JET_OK || n_tok == 0) return rc;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // inputs: H straight from the caller, the index arrays packed into one
  // pinned block (16-byte aligned pieces) and copied in once
  size_t in_off = 0;
  auto pack = [&](const void* src, size_t bytes) -> const void* {
    uint8_t* dst = c->d_in + in_off;
    std::memcpy(c->h_in + in_off, src, bytes);
    in_off += (bytes + 15) & ~size_t(15);
    return dst;
  };
  const int32_t* d_row = static_cast<const int32_t*>(pack(tok_row, (size_t)n_tok * 4));
  const int32_t* d_tok = static_cast<const int32_t*>(pack(tok_ids, (size_t)n_tok * 4));
  const int32_t* d_co = static_cast<const int32_t*>(pack(cand_offsets, (size_t)(n_cand + 1) * 4));
  const int32_t* d_so = static_cast<const int32_t*>(pack(set_offsets, (size_t)(n_sets + 1) * 4));
  const uint8_t* d_kind = static_cast<const uint8_t*>(pack(kind, (size_t)n_sets));
  const int32_t* d_union =
      mode == JET_MODE_RESTRICTED ? static_cast<const int32_t*>(pack(union_ids, (size_t)n_union * 4)) : nullptr;
  if (cudaMemcpyAsync(c->stH, H, (size_t)n_rows * c->d * 2, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(c->d_in, c->h_in, in_off, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return JET_ERR_CUDA;

  // outputs: the requested ones behind the error words, in one device block
  jet_set_out h, dev;
  const size_t out_off = place_host_outputs(c, out_host, n_rows, n_tok, n_cand, n_sets, &h, &dev);
  rc = score_sets_enqueue(c, c->stH, W, n_rows, d_row, d_tok, n_tok, d_co, n_cand, d_so, d_kind, n_sets, T, mode,
                          d_union, n_union, &dev, st);
  if (rc != JET_OK) {
    cudaStreamSynchronize(st);
    return rc;
  }
  // one copy back: error words and every requested output
  if (cudaMemcpyAsync(c->h_out, c->io_dev, out_off, cudaMemcpyDeviceToHost, st) != cudaSuccess) {
    cudaStreamSynchronize(st);
    return JET_ERR_CUDA;
  }
  if (cudaStreamSynchronize(st) != cudaSuccess) return JET_ERR_CUDA;
  const int status = reinterpret_cast<const int*>(c->h_out)[0];
  auto unpack = [&](void* host_ptr, const void* dev_ptr, size_t bytes) {
    if (host_ptr) std::memcpy(host_ptr, c->h_out + (static_cast<const uint8_t*>(dev_ptr) - c->io_dev), bytes);
  };
  unpack(h.logp, dev.logp, (size_t)n_tok * 4);
  unpack(h.lse, dev.lse, (size_t)n_rows * 4);
  unpack(h.s, dev.s, (size_t)n_cand * 4);
  unpack(h.q, dev.q, (size_t)n_cand * 4);
  unpack(h.q_equiv, dev.q_equiv, (size_t)n_cand * 4);
  unpack(h.decision, dev.decision, (size_t)n_sets * 4);
  unpack(h.expected, dev.expected, (size_t)n_sets * 4);
  unpack(h.confidence, dev.confidence, (size_t)n_sets * 4);
  unpack(h.mass, dev.mass, (size_t)n_sets * 4);
  return status;
}

}  // extern "C"

namespace {

// Second staging slot, copy stream and events of jet_score_sets_host_async,
// made on the first call (each piece once, so a failed set-up can be retried).
int host_async_setup(jet_ctx* c) {
  if (c->copy_st) return JET_OK;
  cudaError_t e = cudaSuccess;
  auto A = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
  if (!c->stH2) A(dalloc(&c->stH2, (size_t)c->max_rows * c->d));
  if (!c->d_in2) A(dalloc(&c->d_in2, c->in_cap));
  if (!c->h_status) A(cudaMallocHost(reinterpret_cast<void**>(&c->h_status), STATUS_RING * sizeof(int)));
  for (int i = 0; i < 2; ++i) {
    if (!c->ev_copied[i]) A(cudaEventCreateWithFlags(&c->ev_copied[i], cudaEventDisableTiming));
    if (!c->ev_free[i]) A(cudaEventCreateWithFlags(&c->ev_free[i], cudaEventDisableTiming));
  }
  if (e == cudaSuccess) A(cudaStreamCreateWithFlags(&c->copy_st, cudaStreamNonBlocking));
  return e == cudaSuccess ? JET_OK : JET_ERR_CUDA;
}

// Waits for `st` and folds the statuses of the calls since the last wait into
// async_err (first non-zero wins).
int host_async_drain(jet_ctx* c, cudaStream_t st) {
  if (cudaStreamSynchronize(st) != cudaSuccess) return JET_ERR_CUDA;
  for (int i = 0; i < c->n_async && c->async_err == 0; ++i) c->async_err = c->h_status[i];
  c->n_async = 0;
  return JET_OK;
}

}  // namespace

extern "C" {

int jet_score_sets_host_async(jet_ctx* c, const void* H, const void* W, int n_rows, const int32_t* tok_row,
                              const int32_t* tok_ids, int n_tok, const int32_t* cand_offsets, int n_cand,
                              const int32_t* set_offsets, const uint8_t* kind, int n_sets, float T, int mode,
                              const int32_t* union_ids, int n_union, const jet_set_out* out_host, void* stream) {
  int rc = check_sets_args(c, H, W, n_rows, tok_row, tok_ids, n_tok, cand_offsets, n_cand, set_offsets, kind,
                           n_sets, T, mode, union_ids, n_union);
  if (rc != JET_OK || n_tok == 0) return rc;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = host_async_setup(c);
  if (rc != JET_OK) return rc;
  if (c->n_async == STATUS_RING && host_async_drain(c, st) != JET_OK) return JET_ERR_CUDA;

  // inputs into this call's slot, on the copy stream, once the kernels that
  // last read the slot (two calls back) are done
  const int slot = (int)(c->async_calls & 1);
  uint16_t* stH = slot ? c->stH2 : c->stH;
  uint8_t* din = slot ? c->d_in2 : c->d_in;
  cudaStream_t cs = c->copy_st;
  bool ok = cudaStreamWaitEvent(cs, c->ev_free[slot], 0) == cudaSuccess;
  size_t off = 0;
  auto put = [&](const void* src, size_t bytes) -> const void* {
    uint8_t* dst = din + off;
    off += (bytes + 15) & ~size_t(15);
    ok = ok && cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, cs) == cudaSuccess;
    return dst;
  };
  const int32_t* d_row = static_cast<const int32_t*>(put(tok_row, (size_t)n_tok * 4));
  const int32_t* d_tok = static_cast<const int32_t*>(put(tok_ids, (size_t)n_tok * 4));
  const int32_t* d_co = static_cast<const int32_t*>(put(cand_offsets, (size_t)(n_cand + 1) * 4));
  const int32_t* d_so = static_cast<const int32_t*>(put(set_offsets, (size_t)(n_sets + 1) * 4));
  const uint8_t* d_kind = static_cast<const uint8_t*>(put(kind, (size_t)n_sets));
  const int32_t* d_union =
      mode == JET_MODE_RESTRICTED ? static_cast<const int32_t*>(put(union_ids, (size_t)n_union * 4)) : nullptr;
  ok = ok && cudaMemcpyAsync(stH, H, (size_t)n_rows * c->d * 2, cudaMemcpyHostToDevice, cs) == cudaSuccess;
  ok = ok && cudaEventRecord(c->ev_copied[slot], cs) == cudaSuccess;
  ok = ok && cudaStreamWaitEvent(st, c->ev_copied[slot], 0) == cudaSuccess;
  if (!ok) return JET_ERR_CUDA;
  c->async_calls += 1;

  // outputs: written by the kernels into the output block (in stream order,
  // so the next call's kernels come after these copies), copied to the caller
  jet_set_out h, dev;
  place_host_outputs(c, out_host, n_rows, n_tok, n_cand, n_sets, &h, &dev);
  rc = score_sets_enqueue(c, stH, W, n_rows, d_row, d_tok, n_tok, d_co, n_cand, d_so, d_kind, n_sets, T, mode,
                          d_union, n_union, &dev, st);
  if (rc != JET_OK) {
    cudaStreamSynchronize(st);
    return rc;
  }
  ok = cudaEventRecord(c->ev_free[slot], st) == cudaSuccess;
  auto get = [&](void* host_ptr, const void* dev_ptr, size_t bytes) {
    if (host_ptr) ok = ok && cudaMemcpyAsync(host_ptr, dev_ptr, bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  };
  get(h.logp, dev.logp, (size_t)n_tok * 4);
  get(h.lse, dev.lse, (size_t)n_rows * 4);
  get(h.s, dev.s, (size_t)n_cand * 4);
  get(h.q, dev.q, (size_t)n_cand * 4);
  get(h.q_equiv, dev.q_equiv, (size_t)n_cand * 4);
  get(h.decision, dev.decision, (size_t)n_sets * 4);
  get(h.expected, dev.expected, (size_t)n_sets * 4);
  get(h.confidence, dev.confidence, (size_t)n_sets * 4);
  get(h.mass, dev.mass, (size_t)n_sets * 4);
  get(c->h_status + c->n_async, c->err, sizeof(int));
  c->n_async += 1;
  if (!ok) {
    cudaStreamSynchronize(st);
    return JET_ERR_CUDA;
  }
  return JET_OK;
}

int jet_host_wait(jet_ctx* c, void* stream) {
  if (!c) return JET_ERR_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return JET_ERR_CUDA;
  if (host_async_drain(c, static_cast<cudaStream_t>(stream)) != JET_OK) return JET_ERR_CUDA;
  const int status = c->async_err;
  c->async_err = 0;
  return status;
}

}  // extern "C"
