// The C ABI of libdspark.so: argument checks, the cached device capacity query, the
// launch plan (cooperative grid, shared-memory-resident W2 rows) and the launches.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "lmhead.cuh"
#include "walk_params.cuh"

namespace dspark {

const void* walk_cc_kernel_ptr(bool int8, bool prob, bool logits);
const void* walk_tc_kernel_ptr(bool int8, bool prob, bool logits, int nq, bool rows);
const void* topk_walk_kernel_ptr(bool int8, bool prob, bool logits);
int32_t verify_launch(const uint16_t* target, const uint16_t* draft, const int32_t* dtok,
                      const uint64_t* seeds, int64_t V, int32_t bs, int32_t K, float temperature,
                      int32_t* accepted, int32_t* out_tokens, float* norms, cudaStream_t stream);
size_t topk_walk_smem(int bs);
cudaError_t launch_topk_select(const uint16_t* base, int64_t V, int k, int rows, int32_t* cand,
                               float* cand_base, uint16_t* logits, cudaStream_t stream);
cudaError_t launch_quantize_w2(const uint16_t* w2, int64_t V, int8_t* q, float* scales,
                               int32_t* status_dev, cudaStream_t stream);
cudaError_t launch_gumbel_noise(const uint64_t* seeds, int bs, int K, int64_t V, uint32_t* words,
                                float* gumbel, cudaStream_t stream);
cudaError_t launch_lmhead(LmParams& p, int sms, int pivot_rank, cudaStream_t stream);
cudaError_t launch_fill_neg_inf(uint16_t* x, size_t n, cudaStream_t stream);

// Checks of a walk's arguments other than its workspace, made before any CUDA call.
int32_t check_walk_inputs(const dspark_walk_args* a) {
  if (!a) return DSPARK_ERR_INVALID_ARG;
  // candidates given by the caller: both arrays, a top-k walk; base_logits not read then
  const bool given = a->topk_cand != nullptr || a->topk_base != nullptr;
  if (given && (!a->topk_cand || !a->topk_base || a->top_k < 1)) return DSPARK_ERR_INVALID_ARG;
  if ((!a->base_logits && !given) || !a->w1 || !a->prev_tokens || !a->draft_tokens) return DSPARK_ERR_INVALID_ARG;
  if (a->rank != DSPARK_RANK) return DSPARK_ERR_INVALID_ARG;
  if (a->V <= 0 || a->V > DSPARK_MAX_V) return DSPARK_ERR_INVALID_ARG;
  if (a->bs < 1 || a->bs > DSPARK_MAX_BS || a->K < 1 || a->K > DSPARK_MAX_K) return DSPARK_ERR_INVALID_ARG;
  if (a->mode != DSPARK_GREEDY && a->mode != DSPARK_PROBABILISTIC) return DSPARK_ERR_INVALID_ARG;
  // with per-row modes any row may be sampled; per-row temperatures are checked on the
  // device (a bad one invalidates its row only)
  if (a->mode == DSPARK_PROBABILISTIC || a->row_modes) {
    if (!a->seeds) return DSPARK_ERR_INVALID_ARG;
    if (!a->temperatures && (!(a->temperature > 0.f) || !(a->temperature < 3.4e38f)))
      return DSPARK_ERR_INVALID_ARG;
  }
  const bool have_bf16 = a->w2 != nullptr;
  const bool have_int8 = a->w2q != nullptr;
  if (have_bf16 == have_int8) return DSPARK_ERR_INVALID_ARG;
  if (have_int8 && !a->w2_scales) return DSPARK_ERR_INVALID_ARG;
  if (a->top_k < 0 || a->top_k > a->V) return DSPARK_ERR_INVALID_ARG;
  // 16-byte vector loads of W1 / W2 rows
  if ((reinterpret_cast<uintptr_t>(a->w1) | reinterpret_cast<uintptr_t>(a->w2) |
       reinterpret_cast<uintptr_t>(a->w2q)) & 15u)
    return DSPARK_ERR_INVALID_ARG;
  return DSPARK_OK;
}

namespace {
thread_local char g_last_error[256] = "";
}  // namespace

// Records the failing call for dspark_last_cuda_error and returns DSPARK_ERR_CUDA.
int32_t cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s: %s", where, cudaGetErrorString(e));
  return DSPARK_ERR_CUDA;
}

namespace {

struct DeviceCaps {
  bool valid = false;
  int sms = 0;
  int smem_optin = 0;
  int smem_per_sm = 0;
  int coop = 0;
};

constexpr int kMaxDevices = 64;
DeviceCaps g_caps[kMaxDevices];
std::mutex g_caps_mu;

int32_t get_caps(int device, DeviceCaps* out) {
  if (device < 0 || device >= kMaxDevices) return DSPARK_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_caps_mu);
  DeviceCaps& c = g_caps[device];
  if (!c.valid) {
    cudaError_t e;
    if ((e = cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    if ((e = cudaDeviceGetAttribute(&c.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(smem opt-in)");
    if ((e = cudaDeviceGetAttribute(&c.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(smem per SM)");
    if ((e = cudaDeviceGetAttribute(&c.coop, cudaDevAttrCooperativeLaunch, device)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(cooperative launch)");
    c.valid = true;
  }
  *out = c;
  return DSPARK_OK;
}

int32_t current_caps(DeviceCaps* caps) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  return get_caps(dev, caps);
}

struct Plan {
  int grid;
  int resident_rows;  // per CTA
  int slice_cap;      // rows of the largest vocabulary slice, rounded up to 32
  size_t smem;
};

// One CTA per SM; the shared memory left after the fixed working set holds W2 rows.
Plan plan_dense(const DeviceCaps& caps, int64_t V, bool int8, int bs, int cap_rows) {
  Plan pl{};
  pl.grid = caps.sms;
  const int row_bytes = int8 ? kRank : 2 * kRank;
  const int64_t per_cta = (V + pl.grid - 1) / pl.grid;
  pl.slice_cap = static_cast<int>((per_cta + 31) & ~31LL);
  const size_t fixed = walk_cc_fixed_smem(bs, int8, pl.slice_cap);
  int64_t rows = caps.smem_optin > static_cast<int>(fixed)
                     ? (static_cast<int64_t>(caps.smem_optin) - static_cast<int64_t>(fixed)) / row_bytes
                     : 0;
  rows = rows & ~31LL;
  const int64_t need = (per_cta + 31) & ~31LL;
  if (rows > need) rows = need;
  if (cap_rows >= 0 && rows > cap_rows) rows = cap_rows & ~31;
  pl.resident_rows = static_cast<int>(rows);
  pl.smem = fixed + static_cast<size_t>(rows) * row_bytes;
  return pl;
}

// Smallest batch that takes the tensor-core contraction by default.
constexpr int kTcMinBs = 3;

struct TcPlan {
  int grid;
  int resident_rows;  // per CTA
  int slice_cap;
  int nq;             // padded request rows / 4
  size_t smem;
};

// Tensor-core walk: B operand (N x 512 bytes), the slice's scales, bookkeeping, and as
// many resident W2 rows (whole 32-row blocks) as the remaining shared memory holds.
TcPlan plan_tc(const DeviceCaps& caps, int64_t V, bool int8, bool prob, int bs, int cap_rows, bool base_tma) {
  (void)prob;
  TcPlan pl{};
  pl.grid = caps.sms;
  const int N = bs <= 16 ? 16 : bs <= 32 ? 32 : 64;
  pl.nq = N / 4;
  const int64_t per_cta = (V + pl.grid - 1) / pl.grid + 32;
  pl.slice_cap = static_cast<int>((per_cta + 31) & ~31LL);
  const int row_bytes = int8 ? kRank : 2 * kRank;
  const size_t fixed = 1024 + static_cast<size_t>(N) * 512 + (base_tma ? tc_stage_ring_bytes(N) : 0) +
                       (int8 ? static_cast<size_t>(pl.slice_cap) * 4 : 0) + walk_tc_misc_smem();
  int64_t rows = caps.smem_optin > static_cast<int>(fixed)
                     ? (static_cast<int64_t>(caps.smem_optin) - static_cast<int64_t>(fixed)) / row_bytes
                     : 0;
  rows &= ~31LL;
  if (rows > pl.slice_cap) rows = pl.slice_cap;
  if (cap_rows >= 0 && rows > cap_rows) rows = cap_rows & ~31;
  pl.resident_rows = static_cast<int>(rows);
  pl.smem = fixed + static_cast<size_t>(rows) * row_bytes;
  return pl;
}

// The tensor-core walk handles vocabulary slices of up to kTcMaxTiles tiles.
bool tc_fits(const DeviceCaps& caps, int64_t V) {
  const int64_t per_cta = (V + caps.sms - 1) / caps.sms + 32;
  return (per_cta + 127) / 128 <= kTcMaxTiles;
}

int32_t check_common(const dspark_walk_args* a) {
  const int32_t st = check_walk_inputs(a);
  if (st != DSPARK_OK) return st;
  if (!a->workspace) return DSPARK_ERR_WORKSPACE;
  if (a->workspace_bytes < ws_total(a->K, a->bs, a->top_k)) return DSPARK_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return DSPARK_ERR_WORKSPACE;
  return DSPARK_OK;
}

StepSync make_sync(const dspark_walk_args* a, int grid) {
  StepSync s{};
  char* ws = static_cast<char*>(a->workspace);
  s.hdr = reinterpret_cast<WsHeader*>(ws);
  s.counters = reinterpret_cast<uint32_t*>(ws + ws_counters_off());
  s.slots = reinterpret_cast<uint64_t*>(ws + ws_slots_off(a->K));
  s.status_dev = a->status_dev;
  s.grid = static_cast<uint32_t>(grid);
  s.timeout_ns = 1000ull * (a->timeout_us ? a->timeout_us : 1000000u);
  s.flags = a->flags;
  return s;
}

WalkParams make_params(const dspark_walk_args* a, int grid, int resident_rows, int slice_cap) {
  WalkParams p{};
  p.base = a->base_logits;
  p.w1 = a->w1;
  p.w2 = a->w2;
  p.w2q = a->w2q;
  p.scales = a->w2_scales;
  p.prev = a->prev_tokens;
  p.seeds = a->seeds;
  p.tokens = a->draft_tokens;
  p.logits = a->draft_logits;
  p.cand = reinterpret_cast<const int32_t*>(static_cast<char*>(a->workspace) + ws_cand_off(a->K, a->bs));
  p.V = a->V;
  p.bs = a->bs;
  p.K = a->K;
  p.top_k = a->top_k;
  p.temperature = a->temperature;
  p.temp_is_one = a->temperature == 1.0f ? 1 : 0;
  p.inv_temperature = static_cast<float>(1.0 / static_cast<double>(a->temperature));
  p.temps = a->temperatures;
  p.modes = a->row_modes;
  p.resident_rows = resident_rows;
  p.slice_cap = slice_cap;
  p.sync = make_sync(a, grid);
  return p;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// Tensor map over the W2 rows for the tensor-core walk's resident copies: [V][256] int8
// or bf16, box of 32 rows x 128 bytes, 128-byte swizzle. False when the driver entry
// point is missing (the walk then keeps no rows resident).
bool make_w2_map(const dspark_walk_args* a, CUtensorMap* m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const bool int8 = a->w2q != nullptr;
  void* ptr = int8 ? const_cast<int8_t*>(a->w2q) : static_cast<void*>(const_cast<uint16_t*>(a->w2));
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRank), static_cast<cuuint64_t>(a->V)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRank) * (int8 ? 1 : 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(int8 ? 128 : 64), 32};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = enc(m, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr,
                         dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The tensor-core walk's warpgroups rebalance their registers with setmaxnreg on the
// assumption that the kernel was compiled for kTcLaunchRegs registers per thread; with
// any other count a request for more registers could wait forever, so the walk is not
// launched. Checked once per kernel instance.
int32_t check_tc_registers(const void* fn) {
  constexpr int kSlots = 64;
  static const void* checked[kSlots] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  for (int k = 0; k < kSlots && checked[k]; ++k)
    if (checked[k] == fn) return DSPARK_OK;
  cudaFuncAttributes attr{};
  const cudaError_t e = cudaFuncGetAttributes(&attr, fn);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(walk_tc_kernel)");
  if (attr.numRegs != kTcLaunchRegs) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "walk_tc_kernel compiled for %d registers per thread, its register split assumes %d",
                  attr.numRegs, kTcLaunchRegs);
    return DSPARK_ERR_UNSUPPORTED;
  }
  for (int k = 0; k < kSlots; ++k)
    if (!checked[k]) { checked[k] = fn; break; }
  return DSPARK_OK;
}

// Tensor map over the base logits [bs][K][V] bf16 for the tensor-core walk's stages:
// box of 128 vocabulary rows x 1 position x N requests. False (the walk then loads the
// base logits per thread) when the layout cannot be described: V not a multiple of 8
// (row strides must be multiples of 16 bytes) or a pointer not 16-byte aligned.
bool make_base_map(const dspark_walk_args* a, int N, CUtensorMap* m) {
  if ((a->V & 7) != 0 || (reinterpret_cast<uintptr_t>(a->base_logits) & 15u) != 0) return false;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a->V), static_cast<cuuint64_t>(a->K),
                              static_cast<cuuint64_t>(a->bs)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a->V) * 2,
                                 static_cast<cuuint64_t>(a->V) * 2 * static_cast<cuuint64_t>(a->K)};
  const cuuint32_t box[3] = {128, 1, static_cast<cuuint32_t>(N)};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a->base_logits),
                         dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Dynamic shared memory that keeps a kernel at one CTA per SM: more than half of the
// SM's shared memory (capped at the per-block opt-in). Kernels that allocate all 512
// tensor-memory columns need this: a second CTA on the same SM would wait in
// tcgen05.alloc until the first one exits, which a grid-wide barrier never allows.
size_t exclusive_smem(size_t smem, int smem_per_sm, int smem_optin) {
  const size_t half = static_cast<size_t>(smem_per_sm) / 2 + 1024;
  if (smem >= half) return smem;
  return half < static_cast<size_t>(smem_optin) ? half : static_cast<size_t>(smem_optin);
}

// Cooperative launch of a persistent walk kernel. tmem_exclusive: the kernel takes all
// of tensor memory, so exactly one CTA may be resident per SM.
int32_t launch_coop(const void* fn, int grid, int threads, size_t smem, WalkParams& p, cudaStream_t stream,
                    const DeviceCaps& caps, bool tmem_exclusive) {
  for (int attempt = 0; attempt < 2; ++attempt) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (per_sm < 1) return DSPARK_ERR_COOP_TOO_LARGE;
    if (!tmem_exclusive || per_sm == 1) break;
    const size_t more = exclusive_smem(smem, caps.smem_per_sm, caps.smem_optin);
    if (attempt == 1 || more == smem) return DSPARK_ERR_COOP_TOO_LARGE;
    smem = more;
  }
  void* args[] = {&p};
  cudaError_t e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(threads), args, smem, stream);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return DSPARK_ERR_COOP_TOO_LARGE;
  }
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchCooperativeKernel");
  return DSPARK_OK;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" {

const char* dspark_status_string(int32_t status) {
  switch (status) {
    case DSPARK_OK: return "ok";
    case DSPARK_ERR_INVALID_ARG: return "invalid argument";
    case DSPARK_ERR_UNSUPPORTED: return "unsupported combination";
    case DSPARK_ERR_CUDA: return "CUDA runtime error";
    case DSPARK_ERR_COOP_TOO_LARGE: return "cooperative grid cannot be co-resident";
    case DSPARK_ERR_TIMEOUT: return "device wait timed out";
    case DSPARK_ERR_BAD_TOKEN: return "previous token outside [0, V)";
    case DSPARK_ERR_NONFINITE_W2: return "non-finite W2 entry";
    case DSPARK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

const char* dspark_last_cuda_error(void) { return g_last_error; }

size_t dspark_walk_workspace_size(int64_t V, int32_t bs, int32_t K, int32_t top_k) {
  (void)V;
  if (bs < 1 || K < 1 || top_k < 0) return 0;
  return ws_total(K, bs, top_k);
}

int32_t dspark_query_capacity(int32_t device, int64_t V, int32_t w2_is_int8, int32_t bs,
                              int32_t* grid_ctas, int64_t* resident_rows) {
  if (V <= 0 || V > DSPARK_MAX_V || bs < 1 || bs > DSPARK_MAX_BS) return DSPARK_ERR_INVALID_ARG;
  DeviceCaps caps;
  int32_t st = get_caps(device, &caps);
  if (st != DSPARK_OK) return st;
  // The plan dspark_walk takes by default for this batch size.
  const bool tc = bs >= kTcMinBs && tc_fits(caps, V);
  int grid, per_cta;
  if (tc) {
    const TcPlan pl = plan_tc(caps, V, w2_is_int8 != 0, false, bs, -1, V % 8 == 0);
    grid = pl.grid;
    per_cta = pl.resident_rows;
  } else {
    const Plan pl = plan_dense(caps, V, w2_is_int8 != 0, bs, -1);
    grid = pl.grid;
    per_cta = pl.resident_rows;
  }
  if (grid_ctas) *grid_ctas = grid;
  if (resident_rows) {
    int64_t tot = 0;
    for (int c = 0; c < grid; ++c) {
      const int64_t n = slice_start(c + 1, grid, V) - slice_start(c, grid, V);
      const int64_t cap = tc ? n : (n & ~31LL);
      tot += cap < per_cta ? cap : per_cta;
    }
    *resident_rows = tot;
  }
  return DSPARK_OK;
}

int32_t dspark_quantize_w2(const uint16_t* w2, int64_t V, int32_t rank, int8_t* w2q, float* scales,
                           int32_t* status_dev, dspark_stream_t stream) {
  if (!w2 || !w2q || !scales || V <= 0 || rank != DSPARK_RANK) return DSPARK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w2) & 15u) || (reinterpret_cast<uintptr_t>(w2q) & 7u))
    return DSPARK_ERR_INVALID_ARG;
  const int64_t blocks = (V + 7) / 8;
  if (blocks > 0x7FFFFFFF) return DSPARK_ERR_INVALID_ARG;
  cudaError_t e = launch_quantize_w2(w2, V, w2q, scales, status_dev, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSPARK_OK : cuda_fail(e, "quantize_w2_kernel launch");
}

int32_t dspark_walk_topk(const dspark_walk_args* a, dspark_stream_t stream) {
  int32_t st = check_common(a);
  if (st != DSPARK_OK) return st;
  if (a->top_k < 1) return DSPARK_ERR_INVALID_ARG;
  DeviceCaps caps;
  if ((st = current_caps(&caps)) != DSPARK_OK) return st;
  if (!caps.coop) return DSPARK_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int rows = a->bs * a->K;
  WalkParams p = make_params(a, caps.sms, 0, 0);
  if (a->topk_cand) {  // candidates and their base logits from the caller
    p.cand = a->topk_cand;
    p.cand_base = a->topk_base;
    if (a->draft_logits) {
      const cudaError_t e = launch_fill_neg_inf(a->draft_logits, static_cast<size_t>(rows) * a->V, s);
      if (e != cudaSuccess) return cuda_fail(e, "fill_neg_inf_kernel launch");
    }
  } else {
    float* cand_base = reinterpret_cast<float*>(static_cast<char*>(a->workspace) +
                                                ws_cand_base_off(a->K, a->bs, a->top_k));
    p.cand_base = cand_base;
    const cudaError_t e = launch_topk_select(a->base_logits, a->V, a->top_k, rows,
                                             const_cast<int32_t*>(p.cand), cand_base, a->draft_logits, s);
    if (e != cudaSuccess) return cuda_fail(e, "topk_select_kernel launch");
  }
  const size_t smem = topk_walk_smem(a->bs);
  const bool prob = a->mode == DSPARK_PROBABILISTIC || a->row_modes, lg = a->draft_logits != nullptr;
  const void* fn = topk_walk_kernel_ptr(a->w2q != nullptr, prob, lg);
  return launch_coop(fn, caps.sms, kWalkThreads, smem, p, s, caps, false);
}

int32_t dspark_walk(const dspark_walk_args* a, dspark_stream_t stream) {
  int32_t st = check_common(a);
  if (st != DSPARK_OK) return st;
  if (a->top_k > 0) return dspark_walk_topk(a, stream);
  DeviceCaps caps;
  if ((st = current_caps(&caps)) != DSPARK_OK) return st;
  if (!caps.coop) return DSPARK_ERR_UNSUPPORTED;
  const bool int8 = a->w2q != nullptr;
  const bool lg = a->draft_logits != nullptr;
  const bool prob = a->mode == DSPARK_PROBABILISTIC || a->row_modes;  // any sampled row
  const bool use_tc = !(a->flags & DSPARK_FLAG_FORCE_CUDA_CORES) &&
                      (a->bs >= kTcMinBs || (a->flags & DSPARK_FLAG_FORCE_TENSOR_CORES)) &&
                      tc_fits(caps, a->V);
  if (use_tc) {
    CUtensorMap base_map;
    const int N = a->bs <= 16 ? 16 : a->bs <= 32 ? 32 : 64;
    const bool base_tma = make_base_map(a, N, &base_map);
    const TcPlan pl = plan_tc(caps, a->V, int8, prob, a->bs, a->resident_rows_cap, base_tma);
    int resident = pl.resident_rows;
    size_t smem = pl.smem;
    WalkParams p = make_params(a, pl.grid, resident, pl.slice_cap);
    p.base_tma = base_tma ? 1 : 0;
    if (base_tma) p.base_map = base_map;
    p.w2_tma = make_w2_map(a, &p.w2_map) ? 1 : 0;
    if (!p.w2_tma) {  // no tensor map: every row streamed
      smem -= static_cast<size_t>(resident) * (int8 ? kRank : 2 * kRank);
      p.resident_rows = 0;
    }
    const bool rows = prob && (a->temperatures || a->row_modes);  // per-row settings
    const void* fn = walk_tc_kernel_ptr(int8, prob, lg, pl.nq, rows);
    if ((st = check_tc_registers(fn)) != DSPARK_OK) return st;
    return launch_coop(fn, pl.grid, kTcThreads, smem, p, reinterpret_cast<cudaStream_t>(stream), caps, true);
  }
  const Plan pl = plan_dense(caps, a->V, int8, a->bs, a->resident_rows_cap);
  WalkParams p = make_params(a, pl.grid, pl.resident_rows, pl.slice_cap);
  const void* fn = walk_cc_kernel_ptr(int8, prob, lg);
  return launch_coop(fn, pl.grid, kWalkThreads, pl.smem, p, reinterpret_cast<cudaStream_t>(stream), caps, true);
}

size_t dspark_lmhead_workspace_size(int32_t M, int64_t V, int32_t top_k) {
  if (M < 1 || V < 1 || top_k < 1) return 0;
  return lm_ws_total(M, V, top_k);
}

int32_t dspark_lmhead_topk(const dspark_lmhead_args* a, dspark_stream_t stream) {
  if (!a || !a->hidden || !a->lm_head || !a->cand || !a->cand_base) return DSPARK_ERR_INVALID_ARG;
  if (a->M < 1 || a->V < 1 || a->V > DSPARK_MAX_V || a->d < 64 || a->d > 16384 || (a->d % 64) != 0)
    return DSPARK_ERR_INVALID_ARG;
  if (a->top_k < 1 || a->top_k > a->V || a->top_k > 8192) return DSPARK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a->hidden) | reinterpret_cast<uintptr_t>(a->lm_head)) & 15u)
    return DSPARK_ERR_INVALID_ARG;
  if (!a->workspace || (reinterpret_cast<uintptr_t>(a->workspace) & 255u) ||
      a->workspace_bytes < lm_ws_total(a->M, a->V, a->top_k))
    return DSPARK_ERR_WORKSPACE;
  DeviceCaps caps;
  int32_t st;
  if ((st = current_caps(&caps)) != DSPARK_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return DSPARK_ERR_UNSUPPORTED;
  // The GEMM passes take all 512 tensor-memory columns of their SM: their shared memory
  // must fit the device and keep a second CTA off the SM (more than half of it).
  const size_t gemm_smem = static_cast<size_t>(lm_gemm_smem(a->M));
  if (gemm_smem > static_cast<size_t>(caps.smem_optin) || 2 * gemm_smem <= static_cast<size_t>(caps.smem_per_sm))
    return DSPARK_ERR_UNSUPPORTED;
  LmParams p{};
  p.hidden = a->hidden;
  p.lm_head = a->lm_head;
  p.V = a->V;
  p.M = a->M;
  p.d = a->d;
  p.k = a->top_k;
  p.S = lm_samples(a->V);
  p.cap = lm_cap(a->top_k);
  char* ws = static_cast<char*>(a->workspace);
  p.sample = reinterpret_cast<float*>(ws);
  p.pivot = reinterpret_cast<uint32_t*>(ws + lm_ws_sample(a->M, a->V));
  p.cnt = reinterpret_cast<uint32_t*>(ws + lm_ws_sample(a->M, a->V) + lm_align(4ull * a->M));
  p.list = reinterpret_cast<uint64_t*>(ws + lm_ws_sample(a->M, a->V) + lm_align(4ull * a->M) + lm_ws_cnt(a->M));
  p.cand = a->cand;
  p.cand_base = a->cand_base;
  p.stats = a->stats_dev;
  p.status_dev = a->status_dev;
  p.flags = (a->flags & DSPARK_LMHEAD_FLAG_EXACT) ? kLmForceExact : 0;
  p.timeout_ns = 1000ull * (a->timeout_us ? a->timeout_us : 1000000u);
  auto map2d = [&](CUtensorMap* m, const void* ptr, cuuint64_t inner, cuuint64_t rows, cuuint64_t stride_bytes,
                   cuuint32_t box_rows) {
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const cuuint64_t d = static_cast<cuuint64_t>(a->d);
  if (!map2d(&p.w_map, a->lm_head, d, static_cast<cuuint64_t>(a->V), 2 * d, 128) ||
      !map2d(&p.ws_map, a->lm_head, d, static_cast<cuuint64_t>(p.S), 2 * d * kLmSampleStride, 128) ||
      !map2d(&p.h_map0, a->hidden, d, static_cast<cuuint64_t>(a->M), 2 * d, static_cast<cuuint32_t>(lm_box0(a->M))) ||
      (lm_box1(a->M) > 0 &&
       !map2d(&p.h_map1, a->hidden, d, static_cast<cuuint64_t>(a->M), 2 * d, static_cast<cuuint32_t>(lm_box1(a->M)))))
    return DSPARK_ERR_UNSUPPORTED;
  // pivot rank: the sampled keys that stand for about 1.5 k + 512 of the V logits. The
  // list's size then has a relative spread of about 1/sqrt(rank) (rank >= 32 at every
  // k), which puts k at least 5.3 standard deviations below it and the capacity
  // 3 k + 1024 far above: a row that needs the exact path (a short list) is a rare event.
  const double frac = static_cast<double>(p.S) / static_cast<double>(a->V);
  int rank = static_cast<int>((1.5 * a->top_k + 512.0) * frac + 0.5);
  if (rank < 1) rank = 1;
  if (rank > p.S) rank = p.S;
  const cudaError_t e = launch_lmhead(p, caps.sms, rank, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSPARK_OK : cuda_fail(e, "lmhead kernels launch");
}

int32_t dspark_verify(const dspark_verify_args* a, dspark_stream_t stream) {
  if (!a || !a->target_logits || !a->draft_logits || !a->draft_tokens || !a->seeds || !a->accepted ||
      !a->out_tokens)
    return DSPARK_ERR_INVALID_ARG;
  if (a->V <= 0 || a->V > DSPARK_MAX_V || a->bs < 1 || a->bs > DSPARK_MAX_BS || a->K < 1 || a->K > DSPARK_MAX_K)
    return DSPARK_ERR_INVALID_ARG;
  if (!(a->temperature > 0.f) || !(a->temperature < 3.4e38f)) return DSPARK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(a->norms) & 15u) return DSPARK_ERR_INVALID_ARG;
  const int32_t e = verify_launch(a->target_logits, a->draft_logits, a->draft_tokens, a->seeds, a->V,
                                  a->bs, a->K, a->temperature, a->accepted, a->out_tokens, a->norms,
                                  reinterpret_cast<cudaStream_t>(stream));
  return e == 0 ? DSPARK_OK : cuda_fail(static_cast<cudaError_t>(e), "verify kernels launch");
}

int32_t dspark_walk_from_host(const dspark_walk_args* a, const uint16_t* base_host,
                              const int32_t* prev_host, const uint64_t* seeds_host,
                              int32_t* tokens_host, uint16_t* logits_host, dspark_stream_t stream) {
  int32_t st = check_common(a);
  if (st != DSPARK_OK) return st;
  if (!base_host || !prev_host || !tokens_host) return DSPARK_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t nb = static_cast<size_t>(a->bs) * a->K * static_cast<size_t>(a->V) * 2;
  cudaError_t e;
  if ((e = cudaMemcpyAsync(const_cast<uint16_t*>(a->base_logits), base_host, nb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "copy base_logits to device");
  if ((e = cudaMemcpyAsync(const_cast<int32_t*>(a->prev_tokens), prev_host, 4ull * a->bs, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "copy prev_tokens to device");
  if (seeds_host && a->seeds &&
      (e = cudaMemcpyAsync(const_cast<uint64_t*>(a->seeds), seeds_host, 8ull * a->bs, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "copy seeds to device");
  if ((st = dspark_walk(a, stream)) != DSPARK_OK) return st;
  if ((e = cudaMemcpyAsync(tokens_host, a->draft_tokens, 4ull * a->bs * a->K, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "copy draft_tokens to host");
  if (logits_host && a->draft_logits &&
      (e = cudaMemcpyAsync(logits_host, a->draft_logits, nb, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "copy draft_logits to host");
  return DSPARK_OK;
}

int32_t dspark_gumbel_noise(const uint64_t* seeds, int32_t bs, int32_t K, int64_t V, uint32_t* words,
                            float* gumbel, dspark_stream_t stream) {
  if (!seeds || bs < 1 || K < 1 || V <= 0 || (!words && !gumbel)) return DSPARK_ERR_INVALID_ARG;
  cudaError_t e = launch_gumbel_noise(seeds, bs, K, V, words, gumbel, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSPARK_OK : cuda_fail(e, "gumbel_noise_kernel launch");
}

}  // extern "C"
