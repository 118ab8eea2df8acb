// asp_internal.cuh - device primitives and workspace layout shared by the
// kernels of libasp.so (sm_103a). Nothing here is part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "asp.h"

namespace asp {

// Named NVTX range over one host entry point, so a profiler that reads NVTX
// (Nsight Systems, or ncu with --nvtx and --nvtx-include) attributes the
// kernels a call launches to that call. With no tool attached, push and pop
// only test a null hook.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kMaxSegments = 4096;     // batch * Hkv handled by one call
constexpr int kMaxPages = 1 << 20;     // max_pages bound (int32 page-space arithmetic)
// The decode splits its page sequence by weight: a list's first page weighs
// 1 + decode_piece_cost(d, P) pages, about the K and V a CTA streams in the
// time that ending a piece stalls it (its 8 warp pipelines drift 2-4 us
// apart over a piece and all wait for the last, then merge). The measured
// step time is flat for weights of 160-384 KiB and worse at 48 or 512 KiB.
constexpr int kDecodePieceBytes = 256 * 1024;
constexpr int kMaxPieceCost = 128;
inline int decode_piece_cost(int head_dim, int page_size) {
  const int page_bytes = 4 * page_size * head_dim;  // K and V, bf16
  const int c = (kDecodePieceBytes + page_bytes / 2) / page_bytes;
  return c < kMaxPieceCost ? c : kMaxPieceCost;
}
constexpr int kMaxGroup = 8;           // query heads per KV head (padded mma width)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a bounded on-chip wait gives up after 2 s

// ----------------------------------------------------------------- workspace
// [ header 256 B | arrivals int32[S] | scores f32[S*max_pages] | partials ]
// arrivals[s] counts the decode CTAs done with split segment s; the CTA that
// completes it merges s and puts the count back to zero.
// header word 0 is the sticky device error mask.
struct WsLayout {
  size_t arrivals_off = 0;
  size_t scores_off = 0;
  size_t partials_off = 0;
  size_t total = 0;
  int decode_grid = 0;   // CTAs of the decode kernel
  int slot_floats = 0;   // floats per partial slot: m[8], l[8], o[8][d]
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(const asp_paged_kv& kv, int num_sms) {
  WsLayout w;
  const size_t S = size_t(kv.batch) * kv.num_kv_heads;
  w.decode_grid = num_sms;
  w.slot_floats = 2 * kMaxGroup + kMaxGroup * kv.head_dim;
  w.arrivals_off = 256;
  w.scores_off = align256(w.arrivals_off + S * sizeof(int32_t));
  w.partials_off = align256(w.scores_off + S * size_t(kv.max_pages) * sizeof(float));
  w.total = align256(w.partials_off +
                     (S + size_t(w.decode_grid)) * size_t(w.slot_floats) * sizeof(float));
  return w;
}

// ------------------------------------------------------------- device errors
__device__ __forceinline__ void report(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

// ------------------------------------------------------------------- helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Valid tokens of request b: seq_lens clamped to [0, max_pages*P]; a clamp
// raises ASP_DEVERR_SEQ_RANGE.
__device__ __forceinline__ int clamp_seq_len(int T, int max_pages, int P, uint32_t* err) {
  const long long cap = (long long)max_pages * P;
  if (T < 0 || (long long)T > cap) {
    report(err, ASP_DEVERR_SEQ_RANGE);
    return T < 0 ? 0 : (int)cap;
  }
  return T;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits until the phase with the given parity has completed. Returns false
// (and the caller reports ASP_DEVERR_TIMEOUT) if that takes longer than
// kWaitLimitNs: no wait in this library can spin forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ----------------------------------------------------------- bulk / TMA copy
// 1-D bulk copy global -> shared, completing `bytes` on the mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled TMA load of one box at (x, y). x is the innermost coordinate in
// elements and must be a multiple of 8 for bf16 (16-byte rule).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data read exactly once per call (K/V pages, page summaries):
// evict it first, so that it does not push out the small structures that the
// dependent lookups of every kernel read (lengths, lists, block table, scores).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s and tma_load_2d with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gsrc, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* map, int x,
                                                 int y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------- even splits
// Part i of n of [0, total): the first total % n parts hold one item more.
// 32-bit only (total < 2^31): 64-bit division is a called routine, and at a
// kernel's start its code fetch alone costs microseconds.
struct EvenSplit {
  int q, r;  // items per part, parts with one more
  __device__ __forceinline__ EvenSplit(int total, int n) : q(total / n), r(total % n) {}
  __device__ __forceinline__ int begin(int i) const { return i * q + min(i, r); }
  __device__ __forceinline__ int end(int i) const { return begin(i) + q + (i < r ? 1 : 0); }
  // part holding item x (x < total)
  __device__ __forceinline__ int part_of(int x) const {
    const int big = r * (q + 1);
    return x < big ? x / (q + 1) : r + (x - big) / q;
  }
};

// ------------------------------------------- programmatic dependent launch
// Every kernel of the library is launched with programmatic stream
// serialisation: the next kernel in the stream may be scheduled onto SMs as
// this one's CTAs retire, instead of after the whole grid has drained. Each
// kernel first allows its dependents to launch, then waits for its
// predecessor grid to complete and its memory to be visible before touching
// global memory; only shared-memory and mbarrier set-up come before the wait.
// Stream order is therefore unchanged. Without the launch attribute (or
// after a non-kernel node) both instructions are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_predecessor() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------ bf16 channel min/max
// Exact: the min or max of two bf16 values is one of them.
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmin2(*reinterpret_cast<__nv_bfloat162*>(&a),
                             *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a),
                             *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint2 vmin(uint2 a, uint2 b) {
  return make_uint2(bmin2(a.x, b.x), bmin2(a.y, b.y));
}
__device__ __forceinline__ uint2 vmax(uint2 a, uint2 b) {
  return make_uint2(bmax2(a.x, b.x), bmax2(a.y, b.y));
}
__device__ __forceinline__ uint32_t vmin(uint32_t a, uint32_t b) { return bmin2(a, b); }
__device__ __forceinline__ uint32_t vmax(uint32_t a, uint32_t b) { return bmax2(a, b); }


// ------------------------------------------------------ warp-level mma (bf16)
// ldmatrix of four 8x8 b16 matrices; lane i supplies the row address of
// matrix i / 8, row i % 8.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// c += a * b for one m16n8k16 tile, bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Two floats rounded to bf16 and packed, `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Orders this thread's generic-proxy global writes before its later
// async-proxy (bulk copy) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Asks L2 to fetch `bytes` (a multiple of 16) at a 16-byte aligned global
// address; nothing is returned and nothing waits on it.
__device__ __forceinline__ void prefetch_l2_bulk(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

// Named barrier over a subset of the CTA's warps.
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// -------------------------------------------------------------------- launch
// Launchers implemented in the kernel translation units. Each returns a
// cudaError_t from the launch (cudaSuccess when nothing needed launching).
struct SummarizeArgs {
  const asp_paged_kv* kv;
  int mode;
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint32_t* err;
};
cudaError_t launch_summarize(const SummarizeArgs& a, cudaStream_t stream);

struct SelectArgs {
  const asp_paged_kv* kv;
  const float* q;
  float gamma;
  int budget;
  int32_t* lists;
  int32_t* lens;
  float* scores;
  uint32_t* err;
  int num_sms;
  // optional fused append (asp_coverage_select_append): bf16 [B, Hkv, d]
  const uint16_t* k_new = nullptr;
  const uint16_t* v_new = nullptr;
};
cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream);
// The score kernel alone (a.scores: [B, Hkv, max_pages]; lists/lens unused).
cudaError_t launch_scores(const SelectArgs& a, cudaStream_t stream);
// Scoring and selection in one cluster kernel (select_cluster.cu): the
// cluster size C to use for this shape on the current device (0: the shape
// takes the two-kernel path), and the launch. Segments of kClusterSelectMinPages
// to 8192 pages qualify; a.scores is not used.
constexpr int kClusterSelectMinPages = 64;
int cluster_select_ctas(const asp_paged_kv& kv, int num_sms);
cudaError_t launch_cluster_select(const SelectArgs& a, int C, cudaStream_t stream);

struct DecodeArgs {
  const asp_paged_kv* kv;
  const float* q;
  const int32_t* lists;
  const int32_t* lens;
  float sm_scale;
  float* out;
  float* lse;
  float* partials;
  int32_t* arrivals;  // [S], zero between calls
  uint32_t* err;
  int grid;
  int slot_floats;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// A 2-D bf16 tensor map over [rows, inner] (row stride inner * 2 bytes) with
// boxes of [box_rows, box_inner] elements, the 128-byte swizzle and zero
// fill out of bounds (decode.cu). box_inner * 2 must be 128.
cudaError_t encode_bf16_2d_swizzled(CUtensorMap* map, const void* base, unsigned long long inner,
                                    unsigned long long rows, unsigned box_inner, unsigned box_rows);

// Per-device helpers (abi.cu).
int current_device_sm_count();
cudaError_t set_max_dynamic_smem(const void* func, int bytes);

}  // namespace asp
