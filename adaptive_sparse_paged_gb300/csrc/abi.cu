// abi.cu - the extern "C" entry points of libasp.so declared in asp.h:
// host-side argument checks, workspace layout, launches and the device error
// word. No call here allocates memory; only asp_get_device_error synchronises.
#include <atomic>
#include <cmath>
#include <mutex>

#include "asp_internal.cuh"

namespace asp {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

bool is_pow2_le8(int x) { return x == 1 || x == 2 || x == 4 || x == 8; }

asp_status check_kv(const asp_paged_kv* kv) {
  if (!kv || !kv->k_cache || !kv->v_cache || !kv->summaries || !kv->block_table || !kv->seq_lens)
    return ASP_EINVAL;
  if (kv->batch <= 0 || kv->num_q_heads <= 0 || kv->num_kv_heads <= 0 || kv->max_pages <= 0 ||
      kv->num_phys_pages <= 0)
    return ASP_EINVAL;
  if (kv->num_q_heads % kv->num_kv_heads != 0) return ASP_EINVAL;
  if (kv->head_dim != 64 && kv->head_dim != 128) return ASP_EUNSUPPORTED;
  if (kv->page_size != 16 && kv->page_size != 32 && kv->page_size != 64) return ASP_EUNSUPPORTED;
  if (!is_pow2_le8(kv->num_kv_heads)) return ASP_EUNSUPPORTED;
  if (!is_pow2_le8(kv->num_q_heads / kv->num_kv_heads)) return ASP_EUNSUPPORTED;
  if ((long long)kv->batch * kv->num_kv_heads > kMaxSegments) return ASP_EUNSUPPORTED;
  if (kv->max_pages > kMaxPages) return ASP_EUNSUPPORTED;
  // page-space (with the decode's split weights) and TMA row coordinates are int32
  if ((long long)kv->batch * kv->num_kv_heads * (kv->max_pages + kMaxPieceCost) >= (1LL << 31))
    return ASP_EUNSUPPORTED;
  if ((long long)kv->num_phys_pages * kv->num_kv_heads * kv->page_size >= (1LL << 31))
    return ASP_EUNSUPPORTED;
  // 16-byte alignment of the cache bases (bulk and tensor copies)
  if ((reinterpret_cast<uintptr_t>(kv->k_cache) | reinterpret_cast<uintptr_t>(kv->v_cache) |
       reinterpret_cast<uintptr_t>(kv->summaries)) & 15u)
    return ASP_EINVAL;
  return ASP_OK;
}

asp_status check_ws(const asp_paged_kv* kv, void* ws, size_t ws_bytes, WsLayout* lay) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return ASP_EWORKSPACE;
  const int sms = current_device_sm_count();
  if (sms <= 0) return ASP_ECUDA;
  *lay = ws_layout(*kv, sms);
  if (ws_bytes < lay->total) return ASP_EWORKSPACE;
  return ASP_OK;
}

asp_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ASP_OK : ASP_ECUDA; }

// One warp; thread 0 waits on a barrier that expects one arrival which never
// comes, through the library's bounded wait, and reports the timeout.
__global__ void selftest_wait_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) report(err, ASP_DEVERR_TIMEOUT);
}
}  // namespace

int current_device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t set_max_dynamic_smem(const void* func, int bytes) {
  // The attribute belongs to the function; setting it again is cheap but it
  // is done once per (function, device) to keep capture-time calls minimal.
  static std::mutex mu;
  static const void* done_func[256];
  static int done_dev[256];
  static int done_bytes[256];
  static int n_done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done_func[i] == func && done_dev[i] == dev && done_bytes[i] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  // Every kernel of the library asks for the largest shared-memory carveout,
  // so consecutive kernels never make an SM flush L1 and repartition it.
  e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  if (n_done < 256) {
    done_func[n_done] = func;
    done_dev[n_done] = dev;
    done_bytes[n_done] = bytes;
    ++n_done;
  }
  return cudaSuccess;
}

}  // namespace asp

using namespace asp;

extern "C" {

int32_t asp_abi_version(void) { return ASP_ABI_VERSION; }

const char* asp_status_string(asp_status st) {
  switch (st) {
    case ASP_OK: return "ASP_OK";
    case ASP_EINVAL: return "ASP_EINVAL: invalid argument";
    case ASP_EUNSUPPORTED: return "ASP_EUNSUPPORTED: shape outside the supported set";
    case ASP_EWORKSPACE: return "ASP_EWORKSPACE: workspace null, misaligned or too small";
    case ASP_ECUDA: return "ASP_ECUDA: CUDA runtime call or launch failed";
    case ASP_EDEVICE: return "ASP_EDEVICE: device error word set";
  }
  return "unknown asp_status";
}

asp_status asp_workspace_size(const asp_paged_kv* kv, size_t* bytes) {
  if (!bytes) return ASP_EINVAL;
  asp_status st = check_kv(kv);
  if (st != ASP_OK) return st;
  const int sms = current_device_sm_count();
  if (sms <= 0) return ASP_ECUDA;
  *bytes = ws_layout(*kv, sms).total;
  return ASP_OK;
}

asp_status asp_workspace_init(void* ws, size_t ws_bytes, asp_stream stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256) return ASP_EWORKSPACE;
  // only the error word has to start at zero; zeroing the whole buffer is
  // simplest and still cheap
  return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

asp_status asp_page_summarize(const asp_paged_kv* kv, int32_t mode, const uint16_t* k_new,
                              const uint16_t* v_new, void* ws, size_t ws_bytes,
                              asp_stream stream) {
  NvtxRange range("asp_page_summarize");
  asp_status st = check_kv(kv);
  if (st != ASP_OK) return st;
  if (mode == ASP_SUMMARIZE_BULK) {
    if (k_new || v_new) return ASP_EINVAL;
  } else if (mode == ASP_SUMMARIZE_APPEND) {
    if (!k_new || !v_new) return ASP_EINVAL;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 7u)
      return ASP_EINVAL;
  } else {
    return ASP_EINVAL;
  }
  WsLayout lay;
  if ((st = check_ws(kv, ws, ws_bytes, &lay)) != ASP_OK) return st;
  SummarizeArgs a{kv, mode, k_new, v_new, static_cast<uint32_t*>(ws)};
  return from_cuda(launch_summarize(a, static_cast<cudaStream_t>(stream)));
}

asp_status asp_coverage_select(const asp_paged_kv* kv, const float* q, float gamma,
                               int32_t budget, int32_t* lists, int32_t* lens, void* ws,
                               size_t ws_bytes, asp_stream stream) {
  NvtxRange range("asp_coverage_select");
  asp_status st = check_kv(kv);
  if (st != ASP_OK) return st;
  if (!q || !lists || !lens) return ASP_EINVAL;
  if (reinterpret_cast<uintptr_t>(q) & 15u) return ASP_EINVAL;
  if (budget < 0) return ASP_EINVAL;
  if (budget == 0 && !(gamma > 0.0f && gamma <= 1.0f)) return ASP_EINVAL;
  WsLayout lay;
  if ((st = check_ws(kv, ws, ws_bytes, &lay)) != ASP_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(ws);
  SelectArgs a{kv, q, gamma, budget, lists, lens, reinterpret_cast<float*>(w + lay.scores_off),
               reinterpret_cast<uint32_t*>(w), current_device_sm_count()};
  return from_cuda(launch_select(a, static_cast<cudaStream_t>(stream)));
}

asp_status asp_select_plan(const asp_paged_kv* kv, float gamma, int32_t budget, int32_t append,
                           int32_t* kernels, int32_t* cluster_ctas) {
  asp_status st = check_kv(kv);
  if (st != ASP_OK) return st;
  if (!kernels || !cluster_ctas) return ASP_EINVAL;
  if (budget < 0) return ASP_EINVAL;
  if (budget == 0 && !(gamma > 0.0f && gamma <= 1.0f)) return ASP_EINVAL;
  const int sms = current_device_sm_count();
  if (sms <= 0) return ASP_ECUDA;
  const bool all = budget == 0 && gamma >= 1.0f;
  int C = 0;
  if (!all) C = cluster_select_ctas(*kv, sms);
  *cluster_ctas = C;
  *kernels = C > 0 ? 1 : (all && !append ? 1 : 2);
  return ASP_OK;
}

asp_status asp_coverage_select_append(const asp_paged_kv* kv, const uint16_t* k_new,
                                      const uint16_t* v_new, const float* q, float gamma,
                                      int32_t budget, int32_t* lists, int32_t* lens, void* ws,
                                      size_t ws_bytes, asp_stream stream) {
  NvtxRange range("asp_coverage_select_append");
  asp_status st = check_kv(kv);
  if (st != ASP_OK) return st;
  if (!q || !lists || !lens || !k_new || !v_new) return ASP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_new) |
       reinterpret_cast<uintptr_t>(v_new)) & 15u)
    return ASP_EINVAL;
  if (budget < 0) return ASP_EINVAL;
  if (budget == 0 && !(gamma > 0.0f && gamma <= 1.0f)) return ASP_EINVAL;
  WsLayout lay;
  if ((st = check_ws(kv, ws, ws_bytes, &lay)) != ASP_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(ws);
  SelectArgs a{kv, q, gamma, budget, lists, lens, reinterpret_cast<float*>(w + lay.scores_off),
               reinterpret_cast<uint32_t*>(w), current_device_sm_count(), k_new, v_new};
  return from_cuda(launch_select(a, static_cast<cudaStream_t>(stream)));
}

asp_status asp_page_scores(const asp_paged_kv* kv, const float* q, float* scores, void* ws,
                           size_t ws_bytes, asp_stream stream) {
  NvtxRange range("asp_page_scores");
  asp_status st = check_kv(kv);
  if (st != ASP_OK) return st;
  if (!q || !scores) return ASP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(scores) & 3u))
    return ASP_EINVAL;
  WsLayout lay;
  if ((st = check_ws(kv, ws, ws_bytes, &lay)) != ASP_OK) return st;
  SelectArgs a{kv, q, 0.5f, 0, nullptr, nullptr, scores, static_cast<uint32_t*>(ws),
               current_device_sm_count()};
  return from_cuda(launch_scores(a, static_cast<cudaStream_t>(stream)));
}

asp_status asp_sparse_decode(const asp_paged_kv* kv, const float* q, const int32_t* lists,
                             const int32_t* lens, float sm_scale, float* out, float* lse,
                             void* ws, size_t ws_bytes, asp_stream stream) {
  NvtxRange range("asp_sparse_decode");
  asp_status st = check_kv(kv);
  if (st != ASP_OK) return st;
  if (!q || !lists || !lens || !out || !lse) return ASP_EINVAL;
  if (reinterpret_cast<uintptr_t>(q) & 7u) return ASP_EINVAL;
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale)) return ASP_EINVAL;
  WsLayout lay;
  if ((st = check_ws(kv, ws, ws_bytes, &lay)) != ASP_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(ws);
  DecodeArgs a{kv, q, lists, lens, sm_scale, out, lse,
               reinterpret_cast<float*>(w + lay.partials_off),
               reinterpret_cast<int32_t*>(w + lay.arrivals_off), reinterpret_cast<uint32_t*>(w),
               lay.decode_grid, lay.slot_floats};
  return from_cuda(launch_decode(a, static_cast<cudaStream_t>(stream)));
}

asp_status asp_selftest_wait_timeout(void* ws, size_t ws_bytes, asp_stream stream) {
  NvtxRange range("asp_selftest_wait_timeout");
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256) return ASP_EWORKSPACE;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint32_t*>(ws));
  return from_cuda(cudaGetLastError());
}

asp_status asp_get_device_error(void* ws, uint32_t* code_out, asp_stream stream) {
  if (!ws || !code_out) return ASP_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t code = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&code, ws, sizeof(code), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && code) e = cudaMemset(ws, 0, sizeof(code));
  if (e != cudaSuccess) return ASP_ECUDA;
  *code_out = code;
  return code ? ASP_EDEVICE : ASP_OK;
}

}  // extern "C"
