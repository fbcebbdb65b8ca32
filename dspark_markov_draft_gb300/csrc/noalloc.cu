// dspark_walk_noalloc: the full-vocabulary walk for callers that cannot allocate device
// memory at all -- for example a plugin whose enqueue hook may not call cudaMalloc, or
// a serving process whose device memory is handed in full to a caching allocator at
// start-up, where a cudaMalloc on the decode path would fail or would synchronise the
// device. Such a caller passes only the walk's inputs and outputs; the walk's scratch
// (argmax words, barrier counters, status header) lives in one file-scope device array
// of fixed size that every GPU loading this library holds until the process exits.
#include <cstdint>
#include <mutex>

#include "common.cuh"

namespace dspark {

int32_t check_walk_inputs(const dspark_walk_args* a);
int32_t cuda_fail(cudaError_t e, const char* where);

namespace {

// Stated maximum of the static scratch: enough for every walk the dense entry point
// accepts (bs <= 64, K <= 32 need 256 + 128 K + 8 K bs <= 20,736 bytes).
constexpr size_t kStaticScratchBytes = 24576;

static __device__ __align__(256) unsigned char g_walk_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace
}  // namespace dspark

extern "C" int32_t dspark_walk_noalloc(const dspark_walk_args* a, dspark_stream_t stream) {
  using namespace dspark;
  // every argument check before the first CUDA call, as in the other entry points
  const int32_t st = check_walk_inputs(a);
  if (st != DSPARK_OK) return st;
  if (a->top_k != 0) return DSPARK_ERR_UNSUPPORTED;  // the top-k lists do not fit
  const size_t need = ws_total(a->K, a->bs, 0);
  if (need > kStaticScratchBytes) return DSPARK_ERR_WORKSPACE;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "dspark_walk_noalloc device index");
  void* scratch = nullptr;
  {
    // Once per device, with that device current: the array's device address. In host
    // code the array's name is only a host-side stand-in and must not reach a kernel.
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_walk_scratch);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static walk scratch)");
      if (!p) return cuda_fail(cudaErrorInvalidSymbol, "cudaGetSymbolAddress(static walk scratch)");
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents (a timed-out call leaves it dirty):
  // clear the part this walk uses. Calls that overlap on the GPU race on the array.
  e = cudaMemsetAsync(scratch, 0, need, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static walk scratch)");
  dspark_walk_args b = *a;
  b.workspace = scratch;
  b.workspace_bytes = kStaticScratchBytes;
  return dspark_walk(&b, stream);
}
