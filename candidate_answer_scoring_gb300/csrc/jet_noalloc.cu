// jet_score_tokens_noalloc: per-position log-probabilities without any device
// allocation and without a context.
//
// Who needs it: code that runs inside a host process whose device memory is
// owned by someone else's pool allocator (an inference server or framework
// plugin that reserves all memory up front), where a cudaMalloc would either
// fail or stall every stream with its implicit device synchronisation in the
// middle of a request.  Such callers pass only their own inputs and outputs.
//
// Where the scratch lives: the pre-pass row lists, the gathered logits, the
// per-split (max, sum-exp) partials and the error word sit in one file-scope
// __device__ array, g_noalloc_scratch, that every GPU loading this library
// holds until the process exits.  Its size is fixed: at most
// JET_NOALLOC_MAX_POS positions and JET_NOALLOC_MAX_UNITS schedule units
// (about 2.2 MB).  Every call shares it and it keeps the last call's contents;
// the pre-pass clears what must start at zero (the error word and the per-row
// counters) and everything else is written before it is read.  Calls whose
// work overlaps on the GPU (different streams, or different host threads) race
// on the array.
//
// Set-up: in host code the array's name is only a host-side stand-in; its
// device address is taken with cudaGetSymbolAddress on the first call made in
// each CUDA context on a device (with that device current) and cached, keyed
// on the context's unique id, so a context created after cudaDeviceReset, or
// a caller's own driver-API context, never receives an address from another
// context.  Make that first call before any stream capture.
#include <mutex>

#include "jet_internal.cuh"

namespace {

using namespace jet;

constexpr int NA_MAX_POS = JET_NOALLOC_MAX_POS;
constexpr int NA_MAX_UNITS = JET_NOALLOC_MAX_UNITS;
constexpr int NA_MAX_DEVICES = 64;

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t OFF_ERR = 0;
// the error words and, after them, the head's unit counter err[SCHED_WORD]
constexpr size_t ERR_BLOCK_BYTES = sizeof(int) * (SCHED_WORD + 1);
constexpr size_t OFF_ROW_PTR = align256(OFF_ERR + ERR_BLOCK_BYTES);
static_assert(OFF_ROW_PTR >= OFF_ERR + ERR_BLOCK_BYTES, "row offsets overlap the error block");
static_assert(SCHED_WORD >= ERR_WORDS, "the unit counter follows the error words");
constexpr size_t OFF_ROW_CUR = align256(OFF_ROW_PTR + sizeof(int) * (NA_MAX_POS + 1));
constexpr size_t OFF_ROW_LIST = align256(OFF_ROW_CUR + sizeof(int) * (NA_MAX_POS + 1));
constexpr size_t OFF_ZG = align256(OFF_ROW_LIST + sizeof(int2) * NA_MAX_POS);
constexpr size_t OFF_PART = align256(OFF_ZG + sizeof(float) * NA_MAX_POS);
constexpr size_t NA_SCRATCH_BYTES = align256(OFF_PART + sizeof(float2) * 2 * BM * (size_t)NA_MAX_UNITS);

static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_SCRATCH_BYTES];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_mu;
struct ScratchSlot {
  unsigned long long ctx_id;   // unique id of the context the address belongs to
  unsigned char* addr;         // device address of g_noalloc_scratch in that context (NULL: not looked up)
};
ScratchSlot g_slot[NA_MAX_DEVICES] = {};
EncodeTiledFn g_encode = nullptr;
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

template <typename Fn>
bool driver_entry(const char* name, Fn* out) {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  *out = reinterpret_cast<Fn>(fn);
  return true;
}

// Device address of the scratch array in the current context of `dev`
// (which must be current).
int scratch_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= NA_MAX_DEVICES) return JET_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode && !driver_entry("cuTensorMapEncodeTiled", &g_encode)) return JET_ERR_CUDA;
  if (!g_ctx_current && !driver_entry("cuCtxGetCurrent", &g_ctx_current)) return JET_ERR_CUDA;
  if (!g_ctx_id && !driver_entry("cuCtxGetId", &g_ctx_id)) return JET_ERR_CUDA;
  // The kernels run in the thread's current context.  When none is current
  // yet, the runtime's first context-bound call (the symbol lookup) makes the
  // device's primary context current, so look up first and read the id after.
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return JET_ERR_CUDA;
  ScratchSlot& slot = g_slot[dev];
  unsigned long long id = 0;
  if (ctx && g_ctx_id(ctx, &id) != CUDA_SUCCESS) return JET_ERR_CUDA;
  if (!ctx || !slot.addr || slot.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return JET_ERR_CUDA;
    if (!ctx && (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx || g_ctx_id(ctx, &id) != CUDA_SUCCESS))
      return JET_ERR_CUDA;
    slot.addr = static_cast<unsigned char*>(p);
    slot.ctx_id = id;
  }
  *out = slot.addr;
  return JET_OK;
}

int encode(CUtensorMap* map, const void* base, int d, int rows, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? JET_OK
             : JET_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int jet_score_tokens_noalloc(const void* H, const void* W, int d, int V, const int32_t* tok_ids,
                                        int n_pos, float* logp, float* lse, void* stream) {
  if (d < 64 || d > 16384 || d % 64 != 0 || V < 1 || n_pos < 0) return JET_ERR_ARG;
  if (n_pos == 0) return JET_OK;
  if (!H || !W || !tok_ids || !logp || !aligned16(H) || !aligned16(W)) return JET_ERR_ARG;
  if (n_pos > NA_MAX_POS) return JET_ERR_WORKSPACE;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return JET_ERR_CUDA;
  if (major != 10 || minor != 3) return JET_ERR_UNSUPPORTED;
  unsigned char* base = nullptr;
  int rc = scratch_address(dev, &base);
  if (rc != JET_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  int* err = reinterpret_cast<int*>(base + OFF_ERR);
  int* row_ptr = reinterpret_cast<int*>(base + OFF_ROW_PTR);
  int* row_cur = reinterpret_cast<int*>(base + OFF_ROW_CUR);
  int2* row_list = reinterpret_cast<int2*>(base + OFF_ROW_LIST);
  float* zg = reinterpret_cast<float*>(base + OFF_ZG);
  float2* part = reinterpret_cast<float2*>(base + OFF_PART);

  PrepArgs pa = {};
  pa.n_rows = n_pos;
  pa.n_tok = n_pos;
  pa.V = V;
  pa.tok_row = nullptr;   // token i is predicted by row i
  pa.tok_ids = tok_ids;
  pa.row_ptr = row_ptr;
  pa.row_cur = row_cur;
  pa.row_list = row_list;
  pa.err = err;
  if (launch_prep(pa, st) != cudaSuccess) return JET_ERR_CUDA;

  const Plan plan = make_plan(n_pos, V, d, sms, NA_MAX_UNITS, head_use_pair(n_pos));
  CUtensorMap tmH, tmW;
  if (encode(&tmH, H, d, n_pos, BM) != JET_OK ||
      encode(&tmW, W, d, V, plan.pair ? HeadShape<true>::B_ROWS : HeadShape<false>::B_ROWS) != JET_OK) {
    cudaStreamSynchronize(st);
    return JET_ERR_CUDA;
  }
  HeadArgs ha;
  ha.N = n_pos;
  ha.V = V;
  ha.d = d;
  ha.plan = plan;
  ha.row_ptr = row_ptr;
  ha.row_list = row_list;
  ha.zg = zg;
  ha.part = part;
  ha.err = err;
  ha.sched = head_use_dynamic(plan) ? err + SCHED_WORD : nullptr;
  if (launch_head(tmH, tmW, ha, st) != cudaSuccess) {
    cudaStreamSynchronize(st);
    return JET_ERR_CUDA;
  }
  MergeArgs ma;
  ma.N = n_pos;
  ma.plan = ha.plan;
  ma.part = part;
  ma.zg = zg;
  ma.lse = lse;
  ma.logp = logp;
  ma.err = err;
  if (launch_merge(ma, st) != cudaSuccess) {
    cudaStreamSynchronize(st);
    return JET_ERR_CUDA;
  }
  int status = 0;
  if (cudaMemcpyAsync(&status, err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return JET_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return JET_ERR_CUDA;
  return status;
}
