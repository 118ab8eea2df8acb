// summarize.cu - per-(page, KV head) channel min/max of K (the Quest page
// summary behind the coverage rule's estimate; MOIRA abstract, with Quest as
// named in the HiSparse abstract).
//
// BULK: one warp per logical page (b, p < N_b) loops over the KV heads; each
// lane owns d/32 channels, so every token row is one coalesced warp load of
// 2*d bytes, and 16 rows are in flight per lane. bf16 min/max is exact: each
// result is one of the inputs.
// APPEND: one warp per (request, KV head) writes the new K/V row and folds it
// into its page's summary. Summaries live in logical page order
// [B, Hkv, max_pages, 2, d], so each segment's summaries are contiguous.
#include "asp_internal.cuh"

namespace asp {
namespace {

// One lane's slice of a d-channel bf16 row: d/32 channels.
template <int D>
struct LaneVec;
template <>
struct LaneVec<128> {
  using T = uint2;  // 4 channels
};
template <>
struct LaneVec<64> {
  using T = uint32_t;  // 2 channels
};

struct BulkParams {
  const uint16_t* k;
  uint16_t* summ;
  const int32_t* bt;
  const int32_t* seq_lens;
  uint32_t* err;
  int Hkv, max_pages, num_phys;
};

template <int D, int P>
__global__ void __launch_bounds__(256) summarize_bulk_kernel(BulkParams p) {
  using V = typename LaneVec<D>::T;
  constexpr int kRow = 2 * D / sizeof(V);  // lane slices per row (= 32)
  constexpr int kChunk = 16;               // rows loaded before folding
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int page = blockIdx.x * 8 + (threadIdx.x >> 5);
  pdl_launch_dependents();
  pdl_wait_predecessor();
  const int T = clamp_seq_len(p.seq_lens[b], p.max_pages, P, p.err);
  if (page >= ceil_div(T, P)) return;
  const int phys = p.bt[(size_t)b * p.max_pages + page];
  if (phys < 0 || phys >= p.num_phys) {
    if (lane == 0) report(p.err, ASP_DEVERR_PAGE_RANGE);
    return;
  }
  const int valid = min(P, T - page * P);
  for (int h = 0; h < p.Hkv; ++h) {
    const V* rows = reinterpret_cast<const V*>(p.k + ((size_t)phys * p.Hkv + h) * P * D) + lane;
    V mn = __ldg(rows), mx = mn;
#pragma unroll
    for (int t0 = 0; t0 < P; t0 += kChunk) {
      V v[kChunk];
#pragma unroll
      for (int t = 0; t < kChunk; ++t)
        if (t0 + t < valid) v[t] = __ldg(rows + (t0 + t) * kRow);
#pragma unroll
      for (int t = 0; t < kChunk; ++t)
        if (t0 + t < valid) {
          mn = vmin(mn, v[t]);
          mx = vmax(mx, v[t]);
        }
    }
    V* out = reinterpret_cast<V*>(p.summ + (((size_t)b * p.Hkv + h) * p.max_pages + page) * 2 * D) + lane;
    out[0] = mn;     // row 0: minimum
    out[kRow] = mx;  // row 1: maximum
  }
}

struct AppendParams {
  uint16_t* k;
  uint16_t* v;
  uint16_t* summ;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int32_t* bt;
  const int32_t* seq_lens;
  uint32_t* err;
  int B, Hkv, max_pages, num_phys;
};

template <int D, int P>
__global__ void __launch_bounds__(256) summarize_append_kernel(AppendParams p) {
  using V = typename LaneVec<D>::T;
  constexpr int kRow = 2 * D / sizeof(V);
  const int lane = threadIdx.x & 31;
  const int unit = blockIdx.x * 8 + (threadIdx.x >> 5);  // (b, h)
  pdl_launch_dependents();
  pdl_wait_predecessor();
  if (unit >= p.B * p.Hkv) return;
  const int b = unit / p.Hkv, h = unit % p.Hkv;
  const int T = clamp_seq_len(p.seq_lens[b], p.max_pages, P, p.err);
  if (T <= 0) return;
  const int lp = (T - 1) / P, slot = (T - 1) % P;
  const int phys = p.bt[(size_t)b * p.max_pages + lp];
  if (phys < 0 || phys >= p.num_phys) {
    if (lane == 0) report(p.err, ASP_DEVERR_PAGE_RANGE);
    return;
  }
  const size_t head_block = (size_t)phys * p.Hkv + h;
  const V kn = reinterpret_cast<const V*>(p.k_new + (size_t)unit * D)[lane];
  const V vn = reinterpret_cast<const V*>(p.v_new + (size_t)unit * D)[lane];
  reinterpret_cast<V*>(p.k + (head_block * P + slot) * D)[lane] = kn;
  reinterpret_cast<V*>(p.v + (head_block * P + slot) * D)[lane] = vn;
  V* s = reinterpret_cast<V*>(p.summ + ((size_t)unit * p.max_pages + lp) * 2 * D) + lane;
  if (slot == 0) {  // a fresh page: its only token is both min and max
    s[0] = kn;
    s[kRow] = kn;
  } else {
    s[0] = vmin(s[0], kn);
    s[kRow] = vmax(s[kRow], kn);
  }
}

template <int D, int P>
cudaError_t launch_summarize_t(const SummarizeArgs& a, cudaStream_t stream) {
  const asp_paged_kv& kv = *a.kv;
  if (a.mode == ASP_SUMMARIZE_BULK) {
    BulkParams p{kv.k_cache, kv.summaries, kv.block_table, kv.seq_lens, a.err,
                 kv.num_kv_heads, kv.max_pages, kv.num_phys_pages};
    dim3 grid(ceil_div(kv.max_pages, 8), kv.batch);
    cudaError_t e = set_max_dynamic_smem((const void*)summarize_bulk_kernel<D, P>, 0);
    if (e != cudaSuccess) return e;
    return launch_pdl(summarize_bulk_kernel<D, P>, grid, dim3(256), 0, stream, p);
  } else {
    AppendParams p{kv.k_cache, kv.v_cache, kv.summaries, a.k_new, a.v_new, kv.block_table,
                   kv.seq_lens, a.err, kv.batch, kv.num_kv_heads, kv.max_pages, kv.num_phys_pages};
    const int units = kv.batch * kv.num_kv_heads;
    cudaError_t e = set_max_dynamic_smem((const void*)summarize_append_kernel<D, P>, 0);
    if (e != cudaSuccess) return e;
    return launch_pdl(summarize_append_kernel<D, P>, dim3(ceil_div(units, 8)), dim3(256), 0, stream,
                      p);
  }
}

}  // namespace

cudaError_t launch_summarize(const SummarizeArgs& a, cudaStream_t stream) {
  const int d = a.kv->head_dim, P = a.kv->page_size;
  if (d == 128 && P == 16) return launch_summarize_t<128, 16>(a, stream);
  if (d == 128 && P == 32) return launch_summarize_t<128, 32>(a, stream);
  if (d == 128 && P == 64) return launch_summarize_t<128, 64>(a, stream);
  if (d == 64 && P == 16) return launch_summarize_t<64, 16>(a, stream);
  if (d == 64 && P == 32) return launch_summarize_t<64, 32>(a, stream);
  if (d == 64 && P == 64) return launch_summarize_t<64, 64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace asp
