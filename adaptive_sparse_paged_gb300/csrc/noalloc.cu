// noalloc.cu - asp_coverage_select_noalloc: coverage selection for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: an
// engine that owns all device memory through its own pool and gives plugins
// only their input and output buffers, or a loop that must not allocate once
// it is running. This entry point runs the same score and select kernels as
// asp_coverage_select, but the per-page scores they exchange live in a
// file-scope device array of fixed size instead of a caller workspace.
//
// The array is a static __device__ object: every GPU that loads libasp.so
// holds it (ASP_NOALLOC_MAX_SCORES floats + 256 bytes) until the process exits.
// Its name is only a host-side stand-in in host code, so the first call on
// each device looks its device address up with cudaGetSymbolAddress (with
// that device current) and caches it; make that first call before any stream
// capture. All calls share the one array and it keeps the last call's
// contents: nothing in it has to start at zero (every score the select kernel
// reads is written by the same call, and the spare error word is cleared by
// each call), but calls that overlap on the GPU (two streams, or two host
// threads) race on it and must be serialised by the caller.
#include <mutex>

#include "asp_internal.cuh"

namespace asp {
namespace {

constexpr size_t kHeaderWords = 64;  // 256 bytes: word 0 is a spare device error word
static __device__ __align__(256) uint32_t g_noalloc_scratch[kHeaderWords + ASP_NOALLOC_MAX_SCORES];

constexpr int kMaxDevicesNa = 64;
std::mutex g_na_mu;
uint32_t* g_na_ptr[kMaxDevicesNa] = {};

// Device address of the scratch array on the current device (set-up on first use).
cudaError_t noalloc_scratch(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevicesNa) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_na_mu);
  if (!g_na_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_na_ptr[dev] = static_cast<uint32_t*>(ptr);
  }
  *out = g_na_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace asp

extern "C" asp_status asp_coverage_select_noalloc(const asp_paged_kv* kv, const float* q,
                                                  float gamma, int32_t budget, int32_t* lists,
                                                  int32_t* lens, uint32_t* dev_error,
                                                  asp_stream stream) {
  using namespace asp;
  NvtxRange range("asp_coverage_select_noalloc");
  if (!kv || !q || !lists || !lens) return ASP_EINVAL;
  // the capacity limit comes first, before anything touches the device
  if (kv->batch > 0 && kv->num_kv_heads > 0 && kv->max_pages > 0 &&
      (unsigned long long)kv->batch * kv->num_kv_heads * kv->max_pages > ASP_NOALLOC_MAX_SCORES)
    return ASP_EUNSUPPORTED;
  size_t unused = 0;
  asp_status st = asp_workspace_size(kv, &unused);  // validates the shape and pointers
  if (st != ASP_OK) return st;
  if (reinterpret_cast<uintptr_t>(q) & 15u) return ASP_EINVAL;
  if (budget < 0) return ASP_EINVAL;
  if (budget == 0 && !(gamma > 0.0f && gamma <= 1.0f)) return ASP_EINVAL;
  uint32_t* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return ASP_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* err = dev_error;
  if (!err) {  // no caller word: use (and clear) the spare one in the array
    err = scratch;
    if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return ASP_ECUDA;
  }
  SelectArgs a{kv, q, gamma, budget, lists, lens,
               reinterpret_cast<float*>(scratch + kHeaderWords), err,
               current_device_sm_count()};
  return launch_select(a, s) == cudaSuccess ? ASP_OK : ASP_ECUDA;
}
