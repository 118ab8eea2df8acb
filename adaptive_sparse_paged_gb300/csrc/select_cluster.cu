// select_cluster.cu - coverage selection of one segment per thread-block
// cluster: score and select in one kernel (MOIRA abstract: per request,
// layer, KV head and step, keep the smallest page set whose estimated
// attention mass reaches gamma; the estimate is the Quest bound named in the
// HiSparse abstract).
//
// The two-kernel path (select.cu) streams every segment's summaries over the
// whole GPU, writes the scores to global memory, and then selects each
// segment on one CTA while HBM sits idle. Here a cluster of C CTAs (C = 1,
// 2 or 4; one CTA per SM) owns one segment of up to 2048 C pages: CTA r
// streams the summaries of pages [r M, r M + M), M = ceil(N / C), as 2-D
// tensor copies (8 KiB pieces, 128-byte swizzle) into per-warp rings, keeps
// their scores in shared memory, and the C CTAs then select together through
// distributed shared memory, with three cluster barriers:
//
//   1. min and max score: every CTA pushes its own into every CTA (barrier);
//   2. fixed-point softmax weights (2^37 = the top page; budget mode: 1 per
//      page) and a 4096-bin histogram linear in max - s, condensed into 256
//      coarse bins of 16, per CTA (barrier);
//   3. every CTA reads the cluster's coarse bins, takes the total weight Z
//      and the target ceil(gamma Z) (budget mode: the budget), and finds the
//      bin where the running weight from the top reaches it: the coarse bin,
//      then its 16 fine bins read from every CTA;
//   4. every CTA pushes the pages of that bin (score, id) and the count of
//      its pages above the bin to every CTA (barrier);
//   5. every CTA resolves the cutoff key among those candidates (one per
//      lane when they are few, exact radix rounds otherwise), the number of
//      ties kept (lowest ids first) and its own output offset;
//   6. every CTA writes its kept ids in ascending order at its offset, and
//      asks L2 for the K/V of its first kept pages: the decode that follows
//      reads them, and HBM is idle until its first copies.
//
// All branches before a barrier depend only on values that are the same in
// the whole cluster, so every thread of every CTA reaches every barrier. The
// scores are computed by score::GroupQuery, the instructions of the
// two-kernel path, and the weights, target and tie count by the same integer
// arithmetic, so both paths select the same pages.
#include <cooperative_groups.h>

#include <mutex>
#include <type_traits>

#include "score_common.cuh"

namespace asp {
namespace {

namespace cg = cooperative_groups;
using score::kFull;

constexpr int kCsWarps = 8;
constexpr int kCsThreads = kCsWarps * 32;
constexpr int kCsPages = 2048;                  // pages one CTA scores and holds
constexpr int kCsPer = kCsPages / kCsThreads;   // elements per thread
constexpr int kCsBins = 4096;                   // bins of the linear histogram
constexpr int kCsMaxC = 4;                      // CTAs per cluster
constexpr int kCsSlots = 3;                     // ring slots per warp
constexpr int kCsPieceBytes = 8192;             // summaries one ring slot holds
constexpr int kRxBins = 256;                    // bins of one radix round
constexpr int kLoBits = 19;                     // a weight is lo + hi << 19 in the histogram
constexpr int kLimb = 14;                       // radix rounds: 3 limbs of 14 bits
constexpr int kFine = 16;                       // histogram bins per coarse bin

struct CsParams {
  uint16_t* summ;  // written only by the append variant
  const float* q;
  const int32_t* seq_lens;
  int32_t* lists;
  int32_t* lens;
  uint32_t* err;
  int Hq, Hkv, P, max_pages;
  float inv_sqrt_d;
  float gamma;
  int budget;
  int pf_pieces;  // pieces per warp fetched into L2 before the predecessor ends
  // K/V of kept pages fetched into L2 for the decode that follows: the first
  // kv_pf_pages kept pages (in id order) of each CTA's range
  const int32_t* bt;
  uint16_t* k_cache;  // written only by the append variant
  uint16_t* v_cache;
  int num_phys;
  int kv_pf_pages;
  // append variant: the new token's K and V rows, bf16 [B, Hkv, d]
  const uint16_t* k_new;
  const uint16_t* v_new;
};

// Cluster exchange block, one per CTA. Every field a CTA reads after a
// barrier was pushed into it (remote stores) before that barrier.
struct CsCtl {
  float cmin[kCsMaxC], cmax[kCsMaxC];  // step 1: from CTA c
  uint32_t above_c[kCsMaxC];           // step 4: pages of CTA c above the crossing bin
  uint32_t cand_cnt[kCsMaxC];          // step 4: candidates of CTA c
};

// Shared-memory map (1 KiB aligned): [ring | mbarriers | scores]; after the
// stream the ring is reused for the selection's histograms and candidates.
// A ring slot holds one piece of kRows consecutive pages as 2d / 64
// tensor-copy sub-tiles [kRows pages x 128 B] with the 128-byte swizzle
// (16 pages at d = 128, 32 at d = 64: 8 KiB).
template <int D, int G>
struct CsLayout {
  static constexpr int kRows = kCsPieceBytes / (4 * D);    // pages per piece
  static constexpr int kSubTiles = 2 * D / 64;              // 64-element columns of a page
  static constexpr int kSubBytes = kRows * 128;
  static constexpr int kRingBytes = kCsWarps * kCsSlots * kCsPieceBytes;
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kScoresOff = kBarOff + kCsWarps * kCsSlots * 8;
  static constexpr int kBtOff = kScoresOff + kCsPages * 4;  // block-table slice, int32
  static constexpr int kBytes = kBtOff + kCsPages * 4 + 1024;  // + alignment slack
  // aliases of the ring after the stream
  static constexpr int kHistOff = 0;                          // u32 lo[4096], hi[4096]
  static constexpr int kCandOff = kHistOff + 2 * kCsBins * 4;  // f32 score[8192], i32 id[8192]
  static constexpr int kRxOff = kCandOff + 2 * kCsMaxC * kCsPages * 4;  // u32 [warp][bin][4]
  static_assert(kRxOff + kCsWarps * kRxBins * 16 <= kRingBytes, "selection scratch fits the ring");
};

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

template <int D, int G, int C, bool Append>
__global__ void __launch_bounds__(kCsThreads, 1)
    cluster_select_kernel(const __grid_constant__ CUtensorMap tm_summ, const CsParams p) {
  using L = CsLayout<D, G>;
  constexpr int kPiecePages = L::kRows, kPageBytes = 4 * D;
  extern __shared__ uint8_t cs_raw[];
  uint8_t* cs_smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(cs_raw) + 1023) & ~uintptr_t(1023));
  __shared__ CsCtl ctl;
  __shared__ float red_f[2 * kCsWarps];
  __shared__ unsigned long long red_w[kCsWarps];
  __shared__ uint32_t red_c[kCsWarps];
  __shared__ uint32_t slab_cnt[kCsPer * kCsWarps][2];
    __shared__ unsigned long long rx_w[kRxBins];
  __shared__ uint32_t rx_pick[3];
  __shared__ unsigned long long rx_pick_w;
  __shared__ uint32_t rank_cnt[kCsMaxC][2];  // candidates above / at tau, per CTA
  __shared__ unsigned long long coarse[kCsBins / kFine];  // this CTA's coarse bins
  __shared__ int sel_coarse, sel_bin;
  __shared__ unsigned long long sel_coarse_w, sel_bin_w;
  __shared__ uint32_t loc_n;  // this CTA's candidates
  __shared__ uint32_t res_off, res_eq;

  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = (int)cluster.block_rank();
  const int s = blockIdx.x / C;
  const int b = s / p.Hkv, h = s % p.Hkv;

  uint8_t* ring = cs_smem + warp * kCsSlots * kCsPieceBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(cs_smem + L::kBarOff) + warp * kCsSlots;
  float* sc = reinterpret_cast<float*>(cs_smem + L::kScoresOff);
  uint32_t* hist_lo = reinterpret_cast<uint32_t*>(cs_smem + L::kHistOff);
  uint32_t* hist_hi = hist_lo + kCsBins;
  float* cand_s = reinterpret_cast<float*>(cs_smem + L::kCandOff);
  int32_t* cand_id = reinterpret_cast<int32_t*>(cand_s + kCsMaxC * kCsPages);
  uint32_t* rx_hist = reinterpret_cast<uint32_t*>(cs_smem + L::kRxOff);

  if (lane == 0) {
    for (int i = 0; i < kCsSlots; ++i) mbar_init(&full[i], 1);
    mbar_fence_init();
  }
  if (tid == 0) loc_n = 0;
  // Distributed shared memory may be touched only once every CTA of the
  // cluster runs: arrive now, wait before the first remote access.
  if (C > 1) cluster_arrive_relaxed();
  pdl_launch_dependents();

  const size_t seg_page0 = (size_t)s * p.max_pages;  // first summary of the segment
  auto slice = [&](int n_seg, int& lo, int& hi) {    // this warp's pages [lo, hi)
    const int m = ceil_div(n_seg, C);
    const int r0 = min(n_seg, rank * m), r1 = min(n_seg, r0 + m);
    const EvenSplit sp(r1 - r0, kCsWarps);
    lo = r0 + sp.begin(warp);
    hi = r0 + sp.end(warp);
  };
  // Before the predecessor ends HBM is mostly idle: fetch this warp's first
  // pieces into L2 on a racy read of the length (a stale length only wastes
  // a prefetch; everything is recomputed after the wait).
  if (p.pf_pieces > 0) {
    const long long Tr = __ldcg(p.seq_lens + b);
    const long long cap = (long long)p.max_pages * p.P;
    const int nr = ceil_div((int)(Tr < 0 ? 0 : (Tr > cap ? cap : Tr)), p.P);
    int lo, hi;
    slice(nr, lo, hi);
    const int end = min(hi, lo + p.pf_pieces * kPiecePages);
    for (int pg = lo + lane; pg < end; pg += 32)
      prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(p.summ) + (seg_page0 + pg) * kPageBytes,
                       kPageBytes);
  }
  pdl_wait_predecessor();

  const int T = clamp_seq_len(p.seq_lens[b], p.max_pages, p.P, p.err);
  const int N = ceil_div(T, p.P);
  const int M = ceil_div(N, C);
  const int base = min(N, rank * M);              // first page id of this CTA
  const int Mr = min(N, base + M) - base;         // pages of this CTA
  int32_t* out = p.lists + (size_t)s * p.max_pages;
  const bool mass_mode = p.budget <= 0;
  // Append variant: before the piece holding the segment's last page is
  // copied, its warp writes the new token's K and V rows into slot
  // (T - 1) % P of that page and folds the key into the page's summary (a
  // fresh page, slot 0, takes the key as both bounds), as the APPEND
  // summarize does; the fence orders those writes before the copy reads.
  using LV = typename std::conditional<D == 128, uint2, uint32_t>::type;  // d / 32 channels
  constexpr int kLRow = 2 * D / (int)sizeof(LV);                          // lane units per row
  auto append_token = [&]() {
    const int lp = N - 1, slot = (T - 1) % p.P;
    const int phys = __ldg(p.bt + (size_t)b * p.max_pages + lp);
    if (phys < 0 || phys >= p.num_phys) {
      if (lane == 0) report(p.err, ASP_DEVERR_PAGE_RANGE);
      return;
    }
    const size_t unit = (size_t)b * p.Hkv + h;
    const size_t row = ((size_t)phys * p.Hkv + h) * p.P + slot;
    const LV kn = reinterpret_cast<const LV*>(p.k_new + unit * D)[lane];
    const LV vn = reinterpret_cast<const LV*>(p.v_new + unit * D)[lane];
    reinterpret_cast<LV*>(p.k_cache + row * D)[lane] = kn;
    reinterpret_cast<LV*>(p.v_cache + row * D)[lane] = vn;
    LV* sm = reinterpret_cast<LV*>(p.summ + (seg_page0 + lp) * 2 * D) + lane;
    if (slot == 0) {
      sm[0] = kn;
      sm[kLRow] = kn;
    } else {
      sm[0] = vmin(sm[0], kn);
      sm[kLRow] = vmax(sm[kLRow], kn);
    }
    fence_proxy_async_global();
  };
  // cluster-uniform early exits: no remote access has happened yet
  if (N == 0 || (mass_mode && p.gamma >= 1.0f) || (!mass_mode && p.budget >= N)) {
    if (Append && N > 0 && warp == 0 && base <= N - 1 && N - 1 < base + Mr) append_token();
    for (int i = tid; i < Mr; i += kCsThreads) out[base + i] = base + i;
    if (rank == 0 && tid == 0) p.lens[s] = N;
    if (C > 1) cluster_wait();
    return;
  }

  // The block-table entries of this CTA's pages, for the K/V prefetch at
  // the end; the loads complete while the first summary copies fly.
  int32_t* bt_s = reinterpret_cast<int32_t*>(cs_smem + L::kBtOff);
  if (p.kv_pf_pages > 0)
    for (int i = tid; i < Mr; i += kCsThreads) bt_s[i] = __ldg(p.bt + (size_t)b * p.max_pages + base + i);

  // ------------------------------------------------------------ the stream
  {
    int wlo, whi;
    slice(N, wlo, whi);
    const uint64_t pol = l2_evict_first_policy();  // summaries are read once per call
    int issue_pg = wlo, issued = 0;
    // one piece: kSubTiles boxes of [kRows pages x 64 elements]; rows past
    // the segment belong to the next one (or are zero-filled past the end)
    // and are not scored
    auto issue = [&]() {
      const int slot = issued % kCsSlots;
      if (Append && issue_pg + min(kPiecePages, whi - issue_pg) == N) {  // warp-uniform
        append_token();
        __syncwarp();
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[slot], kCsPieceBytes);
        const int row = (int)seg_page0 + issue_pg;
#pragma unroll
        for (int t = 0; t < L::kSubTiles; ++t)
          tma_load_2d_hint(ring + slot * kCsPieceBytes + t * L::kSubBytes, &tm_summ, t * 64, row,
                           &full[slot], pol);
      }
      issue_pg += min(kPiecePages, whi - issue_pg);
      ++issued;
    };
    if (lane == 0) prefetch_tensormap(&tm_summ);
    for (int k = 0; k < kCsSlots && issue_pg < whi; ++k) issue();
    score::GroupQuery<D, G> gq;
    gq.load(p.q + ((size_t)b * p.Hq + h * G) * D, lane);
    const int g = lane >> 2, t = lane & 3;
    int k = 0;
    bool aborted = false;
#pragma unroll 1
    for (int pg = wlo; pg < whi; ++k) {
      const int slot = k % kCsSlots;
      if (!__all_sync(kFull, mbar_wait(&full[slot], (k / kCsSlots) & 1))) {
        if (lane == 0) report(p.err, ASP_DEVERR_TIMEOUT);
        aborted = true;
        break;
      }
      const int n = min(kPiecePages, whi - pg);
      const uint32_t sb = smem_u32(ring + slot * kCsPieceBytes);
#pragma unroll
      for (int nt = 0; nt < kPiecePages / 8; ++nt) {
        if (nt * 8 >= n) break;  // warp-uniform
        float x0, x1;
        gq.tile_swz(sb, nt, kPiecePages, lane, x0, x1);
        const int q0 = nt * 8 + 2 * t;
        if (g == 0) {
          if (q0 < n) sc[pg - base + q0] = x0 * p.inv_sqrt_d;
          if (q0 + 1 < n) sc[pg - base + q0 + 1] = x1 * p.inv_sqrt_d;
        }
      }
      pg += n;
      __syncwarp();  // every lane is done reading the slot
      if (issue_pg < whi) {
        fence_proxy_async_smem();
        issue();
      }
    }
    // never reuse the ring with copies in flight (only after a timeout can any remain)
    if (aborted && lane == 0)
      for (int j = k; j < issued; ++j) mbar_wait(&full[j % kCsSlots], (j / kCsSlots) & 1);
    __syncwarp();
  }
  __syncthreads();  // every score of this CTA is in shared memory; the ring is free

  // ------------------------------------------------------- 1. min and max
  float v[kCsPer];
  float lo_s = INFINITY, hi_s = -INFINITY;
#pragma unroll
  for (int k = 0; k < kCsPer; ++k) {
    const int i = k * kCsThreads + tid;
    v[k] = -INFINITY;
    if (i < Mr) {
      v[k] = sc[i];
      lo_s = fminf(lo_s, v[k]);
      hi_s = fmaxf(hi_s, v[k]);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    lo_s = fminf(lo_s, __shfl_xor_sync(kFull, lo_s, o));
    hi_s = fmaxf(hi_s, __shfl_xor_sync(kFull, hi_s, o));
  }
  if (lane == 0) {
    red_f[warp] = lo_s;
    red_f[kCsWarps + warp] = hi_s;
  }
  __syncthreads();
  if (C > 1) cluster_wait();  // every CTA of the cluster is running
  if (tid < C) {              // push this CTA's pair into CTA tid
    float mn = INFINITY, mx = -INFINITY;
    for (int w = 0; w < kCsWarps; ++w) {
      mn = fminf(mn, red_f[w]);
      mx = fmaxf(mx, red_f[kCsWarps + w]);
    }
    CsCtl* dst = cluster.map_shared_rank(&ctl, tid);
    dst->cmin[rank] = mn;
    dst->cmax[rank] = mx;
  }
  cluster.sync();  // barrier 1
  float smin = INFINITY, smax = -INFINITY;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    smin = fminf(smin, ctl.cmin[c]);
    smax = fmaxf(smax, ctl.cmax[c]);
  }

  // ------------------------------------------- 2. weights and the histogram
  unsigned long long mw[kCsPer];
#pragma unroll
  for (int k = 0; k < kCsPer; ++k)
    mw[k] = k * kCsThreads + tid < Mr
                ? (mass_mode ? score::mass_fixed(v[k], smax, score::kUnitFast) : 1ull)
                : 0ull;
  // bins linear in smax - s over at most 28 units in mass mode (a page
  // further down has zero weight); the bin index never increases with the
  // score, so the bin where the running weight from the top reaches the
  // target holds one interval of keys
  const float span = mass_mode ? fminf(smax - smin, 28.f) : smax - smin;
  const float inv_w = span > 0.f ? (float)kCsBins / span : 0.f;
  auto lin_bin = [&](float x) { return min(kCsBins - 1, (int)((smax - x) * inv_w)); };
  for (int i = tid; i < 2 * kCsBins / 4; i += kCsThreads)
    reinterpret_cast<uint4*>(hist_lo)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kCsPer; ++k)
    if (mw[k]) {
      const int bin = lin_bin(v[k]);
      atomicAdd(&hist_lo[bin], (uint32_t)mw[k] & ((1u << kLoBits) - 1u));
      const uint32_t hw = (uint32_t)(mw[k] >> kLoBits);
      if (hw) atomicAdd(&hist_hi[bin], hw);
    }
  __syncthreads();
  {  // coarse bin tid: the 16 bins [16 tid, 16 tid + 16) of this CTA
    unsigned long long cw = 0;
    const uint4* lo4 = reinterpret_cast<const uint4*>(hist_lo + tid * kFine);
    const uint4* hi4 = reinterpret_cast<const uint4*>(hist_hi + tid * kFine);
#pragma unroll
    for (int u = 0; u < kFine / 4; ++u) {
      const uint4 x4 = lo4[u], z4 = hi4[u];
      cw += (unsigned long long)x4.x + x4.y + x4.z + x4.w +
            (((unsigned long long)z4.x + z4.y + z4.z + z4.w) << kLoBits);
    }
    coarse[tid] = cw;
  }
  cluster.sync();  // barrier 2: every histogram of the cluster is complete

  // ------------------------------ 3. the crossing bin, found by every CTA
  // Every CTA reads the cluster's coarse bins, takes the total weight Z and
  // the target, finds the coarse bin where the running weight from the top
  // reaches it, then the fine bin inside: the same values in every CTA.
  unsigned long long target = (unsigned long long)p.budget;
  {
    unsigned long long cw = 0;
#pragma unroll
    for (int c = 0; c < C; ++c) cw += cluster.map_shared_rank(coarse, c)[tid];
    unsigned long long x = cw;  // inclusive scan over the threads (coarse bins in order)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) red_w[warp] = x;
    __syncthreads();
    unsigned long long woff = 0, Z = 0;
#pragma unroll
    for (int ww = 0; ww < kCsWarps; ++ww) {
      const unsigned long long t = red_w[ww];
      if (ww < warp) woff += t;
      Z += t;
    }
    if (mass_mode) {
      target = score::ceil_gamma_times(p.gamma, Z);
      if (target < 1) target = 1;
    }
    const unsigned long long run = woff + x - cw;  // weight of the coarse bins above this one
    if (run < target && run + cw >= target) {      // exactly one coarse bin
      sel_coarse = tid;
      sel_coarse_w = run;
    }
  }
  __syncthreads();
  if (warp == 0) {  // the fine bins of that coarse bin, one per lane
    const int jc = sel_coarse;
    unsigned long long fw = 0;
    if (lane < kFine) {
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const uint32_t* rlo = cluster.map_shared_rank(hist_lo, c);
        fw += rlo[jc * kFine + lane] + ((unsigned long long)rlo[kCsBins + jc * kFine + lane] << kLoBits);
      }
    }
    unsigned long long x = fw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    const unsigned long long run = sel_coarse_w + x - fw;
    if (lane < kFine && run < target && run + fw >= target) {
      sel_bin = jc * kFine + lane;
      sel_bin_w = run;
    }
  }
  __syncthreads();
  const int jbin = sel_bin;
  const unsigned long long above_w = sel_bin_w;

  // ------------- 4. candidates and the count of pages above, to every CTA
  {
    const unsigned lt = (1u << lane) - 1u;
    uint32_t above = 0;
#pragma unroll
    for (int k = 0; k < kCsPer; ++k) {
      const bool valid = k * kCsThreads + tid < Mr;
      const int bin = valid ? lin_bin(v[k]) : kCsBins;
      above += bin < jbin;
      const unsigned m = __ballot_sync(kFull, bin == jbin);
      if (m) {  // warp-uniform
        uint32_t at = 0;
        if (lane == __ffs(m) - 1) at = atomicAdd(&loc_n, (uint32_t)__popc(m));
        at = __shfl_sync(kFull, at, __ffs(m) - 1);
        if (bin == jbin) {  // region `rank` of every CTA's candidate buffer
          const uint32_t i = rank * kCsPages + at + __popc(m & lt);
          const int id = base + k * kCsThreads + tid;
#pragma unroll
          for (int c = 0; c < C; ++c) {
            cluster.map_shared_rank(cand_s, c)[i] = v[k];
            cluster.map_shared_rank(cand_id, c)[i] = id;
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) above += __shfl_xor_sync(kFull, above, o);
    if (lane == 0) red_c[warp] = above;
    __syncthreads();
    if (tid < C) {
      uint32_t a = 0;
      for (int ww = 0; ww < kCsWarps; ++ww) a += red_c[ww];
      CsCtl* dst = cluster.map_shared_rank(&ctl, tid);
      dst->above_c[rank] = a;
      dst->cand_cnt[rank] = loc_n;
    }
  }
  cluster.sync();  // barrier 3: every CTA holds every candidate

  // ----------------------------- 5. the cutoff (every CTA, redundantly)
  uint32_t pc[kCsMaxC + 1];  // candidates of CTAs before c
  pc[0] = 0;
  uint32_t above_c = 0;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    pc[c + 1] = pc[c] + ctl.cand_cnt[c];
    above_c += ctl.above_c[c];
  }
  const uint32_t nc = pc[C];
  auto slot_of = [&](uint32_t j, int& r) {  // candidate j's slot and its CTA
    r = 0;
    uint32_t first = 0;
#pragma unroll
    for (int c = 1; c < C; ++c)
      if (j >= pc[c]) {
        r = c;
        first = pc[c];
      }
    return r * kCsPages + (j - first);
  };
  auto wgt = [&](float xs) -> unsigned long long {
    return mass_mode ? score::mass_fixed(xs, smax, score::kUnitFast) : 1ull;
  };
  // Ties kept: the fewest that reach the target (at least one), lowest ids
  // first; `above_tau` is the weight (count) of every page above tau, below
  // the target by the choice of tau. From the candidates above / at tau per
  // CTA (gtc, eqc) it sets this CTA's output offset and its share of the
  // ties, and CTA 0 writes the list length. Run by one thread.
  auto finish = [&](uint32_t tau, unsigned long long above_tau, const uint32_t* gtc,
                    const uint32_t* eqc) {
    uint32_t n_eq = 0;
#pragma unroll
    for (int c = 0; c < C; ++c) n_eq += eqc[c];
    unsigned long long t;
    if (mass_mode) {
      const unsigned long long wt = wgt(score::key_score(tau));
      t = wt ? (target > above_tau ? score::ceil_div_count(target - above_tau, wt) : 1ull) : n_eq;
    } else {
      t = target > above_tau ? target - above_tau : 1ull;
    }
    if (t < 1) t = 1;
    if (t > n_eq) t = n_eq;
    uint32_t off = 0, eq_before = 0;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const uint32_t keep_eq =
          (uint32_t)min((unsigned long long)eqc[c], t > eq_before ? t - eq_before : 0ull);
      if (c == rank) {
        res_off = off;
        res_eq = keep_eq;
      }
      off += ctl.above_c[c] + gtc[c] + keep_eq;
      eq_before += eqc[c];
    }
    if (rank == 0) p.lens[s] = (int32_t)off;
  };
  // weight (mass mode) or count (budget mode) of every page with a key above
  // the current candidate range
  unsigned long long above = mass_mode ? above_w : (unsigned long long)above_c;
  uint32_t tau;
  if (nc <= 32) {
    if (warp == 0) {  // one candidate per lane
      const bool has = lane < (int)nc;
      int r = 0;
      const float cv = has ? cand_s[slot_of(lane, r)] : 0.f;
      const uint32_t ck = score::score_key(cv);
      const unsigned long long cm = has ? wgt(cv) : 0ull;
      unsigned long long gt_w = 0, ge_w = 0;
      for (int o = 0; o < (int)nc; ++o) {
        const uint32_t k2 = __shfl_sync(kFull, ck, o);
        const unsigned long long m2 = __shfl_sync(kFull, cm, o);
        if (k2 > ck) gt_w += m2;
        if (k2 >= ck) ge_w += m2;
      }
      // tau: the largest key whose weight from the top, ties included, reaches the target
      const bool reach = has && above + ge_w >= target;
      uint32_t best = reach ? ck : 0u;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) best = max(best, __shfl_xor_sync(kFull, best, o));
      const unsigned at = __ballot_sync(kFull, reach && ck == best);
      const unsigned long long above_tau = __shfl_sync(kFull, above + gt_w, __ffs(at) - 1);
      // candidates above and at tau, per CTA (their lanes' regions)
      uint32_t gtc[kCsMaxC], eqc[kCsMaxC];
#pragma unroll
      for (int c = 0; c < C; ++c) {
        gtc[c] = __popc(__ballot_sync(kFull, has && r == c && ck > best));
        eqc[c] = __popc(__ballot_sync(kFull, has && r == c && ck == best));
      }
      if (lane == 0) {
        rx_pick[0] = best;
        finish(best, above_tau, gtc, eqc);
      }
    }
    __syncthreads();
    tau = rx_pick[0];
  } else {
    // exact radix rounds over the candidate keys until one key is left
    uint32_t klo = 0xffffffffu, khi = 0u;
    for (uint32_t j = tid; j < nc; j += kCsThreads) {
      int r;
      const uint32_t kk = score::score_key(cand_s[slot_of(j, r)]);
      klo = min(klo, kk);
      khi = max(khi, kk);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      klo = min(klo, __shfl_xor_sync(kFull, klo, o));
      khi = max(khi, __shfl_xor_sync(kFull, khi, o));
    }
    if (lane == 0) {
      red_c[warp] = klo;
      slab_cnt[warp][0] = khi;
    }
    __syncthreads();
    klo = 0xffffffffu;
    khi = 0u;
    for (int ww = 0; ww < kCsWarps; ++ww) {
      klo = min(klo, red_c[ww]);
      khi = max(khi, slab_cnt[ww][0]);
    }
    __syncthreads();
    uint32_t* my_rx = rx_hist + warp * kRxBins * 4;
    constexpr uint32_t kLimbMask = (1u << kLimb) - 1u;
    while (klo != khi) {
      const uint32_t range = khi - klo;
      const int bits = 32 - __clz(range);
      const int shift = bits > 8 ? bits - 8 : 0;
      for (int i = tid; i < kCsWarps * kRxBins; i += kCsThreads)
        reinterpret_cast<uint4*>(rx_hist)[i] = make_uint4(0, 0, 0, 0);
      __syncthreads();
      for (uint32_t j = tid; j < nc; j += kCsThreads) {
        int r;
        const float xs = cand_s[slot_of(j, r)];
        const uint32_t kk = score::score_key(xs);
        if (kk >= klo && kk <= khi) {
          uint32_t* hb = my_rx + ((kk - klo) >> shift) * 4;
          atomicAdd(hb, 1u);
          if (mass_mode) {
            const unsigned long long m = wgt(xs);
            atomicAdd(hb + 1, (uint32_t)m & kLimbMask);
            atomicAdd(hb + 2, (uint32_t)(m >> kLimb) & kLimbMask);
            atomicAdd(hb + 3, (uint32_t)(m >> (2 * kLimb)));
          }
        }
      }
      __syncthreads();
      {  // merge the private histograms: thread tid owns bin tid
        uint32_t c = 0;
        unsigned long long l0 = 0, l1 = 0, l2 = 0;
        for (int ww = 0; ww < kCsWarps; ++ww) {
          const uint4 hv = reinterpret_cast<const uint4*>(rx_hist)[ww * kRxBins + tid];
          c += hv.x;
          l0 += hv.y;
          l1 += hv.z;
          l2 += hv.w;
        }
        rx_w[tid] = mass_mode ? l0 + (l1 << kLimb) + (l2 << (2 * kLimb)) : c;
      }
      __syncthreads();
      if (warp == 0) {  // the highest bin j with above + (weight of bins >= j) >= target
        unsigned long long lw = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) lw += rx_w[lane * 8 + i];
        unsigned long long sw = lw;  // inclusive suffix over lanes >= lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long y = __shfl_down_sync(kFull, sw, o);
          if (lane + o < 32) sw += y;
        }
        const unsigned bal = __ballot_sync(kFull, above + sw >= target);
        const int ls = bal ? 31 - __clz(bal) : 0;
        if (lane == ls) {
          unsigned long long run = above + (sw - lw);
          int j = lane * 8;
          for (int i = 7; i >= 0; --i) {
            const unsigned long long nw = run + rx_w[lane * 8 + i];
            if (nw >= target) {
              j = lane * 8 + i;
              break;
            }
            run = nw;
          }
          rx_pick[0] = (uint32_t)j;
          rx_pick_w = run;
        }
      }
      __syncthreads();
      const uint32_t j = rx_pick[0];
      above = rx_pick_w;
      const unsigned long long nlo = (unsigned long long)klo + ((unsigned long long)j << shift);
      const unsigned long long nhi = nlo + ((1ull << shift) - 1ull);
      klo = (uint32_t)nlo;
      khi = nhi < khi ? (uint32_t)nhi : khi;
      __syncthreads();  // rx_pick is rewritten by the next round
    }
    tau = klo;  // and `above` is everything above it
    // candidates above tau and at tau, per CTA of the cluster (ids are contiguous per CTA)
    if (tid < kCsMaxC) rank_cnt[tid][0] = rank_cnt[tid][1] = 0;
    __syncthreads();
    for (uint32_t j = tid; j < nc; j += kCsThreads) {
      int r;
      const uint32_t kk = score::score_key(cand_s[slot_of(j, r)]);
      if (kk > tau) atomicAdd(&rank_cnt[r][0], 1u);
      else if (kk == tau) atomicAdd(&rank_cnt[r][1], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t gtc[kCsMaxC], eqc[kCsMaxC];
#pragma unroll
      for (int c = 0; c < C; ++c) {
        gtc[c] = rank_cnt[c][0];
        eqc[c] = rank_cnt[c][1];
      }
      finish(tau, above, gtc, eqc);
    }
    __syncthreads();
  }

  // ------------------------------------- 7. kept ids, ascending, per CTA
  const uint32_t out_off = res_off, eq_keep = res_eq;
  uint32_t gtm[kCsPer], eqm[kCsPer];
#pragma unroll
  for (int k = 0; k < kCsPer; ++k) {
    const bool valid = k * kCsThreads + tid < Mr;
    const uint32_t key = score::score_key(v[k]);
    gtm[k] = __ballot_sync(kFull, valid && key > tau);
    eqm[k] = __ballot_sync(kFull, valid && key == tau);
    if (lane == 0) {
      slab_cnt[k * kCsWarps + warp][0] = __popc(gtm[k]);
      slab_cnt[k * kCsWarps + warp][1] = __popc(eqm[k]);
    }
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan over the (slab, warp) counts in id order
    constexpr int kE = kCsPer * kCsWarps / 32;
    uint32_t ga[kE], ea[kE], gs = 0, es = 0;
#pragma unroll
    for (int u = 0; u < kE; ++u) {
      ga[u] = slab_cnt[lane * kE + u][0];
      ea[u] = slab_cnt[lane * kE + u][1];
      gs += ga[u];
      es += ea[u];
    }
    uint32_t xg = gs, xe = es;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t yg = __shfl_up_sync(kFull, xg, o);
      const uint32_t ye = __shfl_up_sync(kFull, xe, o);
      if (lane >= o) {
        xg += yg;
        xe += ye;
      }
    }
    uint32_t rg = xg - gs, re = xe - es;
#pragma unroll
    for (int u = 0; u < kE; ++u) {
      slab_cnt[lane * kE + u][0] = rg;
      slab_cnt[lane * kE + u][1] = re;
      rg += ga[u];
      re += ea[u];
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int k = 0; k < kCsPer; ++k) {
    const uint32_t gb = slab_cnt[k * kCsWarps + warp][0] + __popc(gtm[k] & lt);
    const uint32_t eb = slab_cnt[k * kCsWarps + warp][1] + __popc(eqm[k] & lt);
    const bool is_gt = (gtm[k] >> lane) & 1u, is_eq = (eqm[k] >> lane) & 1u;
    if (is_gt || (is_eq && eb < eq_keep)) {
      const uint32_t pos = gb + min(eb, eq_keep);  // among this CTA's kept pages
      out[out_off + pos] = base + k * kCsThreads + tid;
      // The decode reads the K/V of every kept page next; HBM is idle until
      // its first copies, so move the first kept pages into L2 now (a stale or
      // out-of-range table entry only skips the prefetch: the decode checks it).
      if ((int)pos < p.kv_pf_pages) {
        const int phys = bt_s[k * kCsThreads + tid];
        if (phys >= 0 && phys < p.num_phys) {
          const size_t blk = ((size_t)phys * p.Hkv + h) * (size_t)p.P * D;
          prefetch_l2_bulk(p.k_cache + blk, (uint32_t)(p.P * D * 2));
          prefetch_l2_bulk(p.v_cache + blk, (uint32_t)(p.P * D * 2));
        }
      }
    }
  }
}

// Pieces per warp fetched into L2 before the previous kernel ends, and kept
// pages per CTA whose K/V the kernel fetches into L2 for the decode (8 KiB
// each at P = 16, d = 128). Outstanding bulk prefetches hold this kernel
// open, so more pages make it slower than they make the decode faster. At
// 128k, gamma = 0.99 on one GB300 (builds alternated on one box, steps/s):
// (pages, pieces) = (0, 3) 365.5, (32, 3) 372.6, (64, 3) 369.1, (128, 3)
// 364.9, (256, 3) 339.4; on a later build of the decode, (32, 3) 390.7,
// (24, 6) 393.6, (28, 6) 393.6, (24, 8) 393.6, and on another box (16, 3)
// 391.9, (48, 3) 391.9, (32, 4) 394.8, (24, 4) 395.3 against (32, 3) 393.7.
constexpr int kCsPrefetchPieces = 6;
constexpr int kCsKvPrefetchPages = 24;

template <int D, int G, int C, bool Append>
cudaError_t launch_cs(const SelectArgs& a, cudaStream_t stream) {
  const asp_paged_kv& kv = *a.kv;
  using L = CsLayout<D, G>;
  const void* fn = (const void*)cluster_select_kernel<D, G, C, Append>;
  cudaError_t e = set_max_dynamic_smem(fn, L::kBytes);
  if (e != cudaSuccess) return e;
  CUtensorMap tm;
  // summaries as [B * Hkv * max_pages rows, 2d elements]
  e = encode_bf16_2d_swizzled(&tm, kv.summaries, 2ull * D,
                              (unsigned long long)kv.batch * kv.num_kv_heads * kv.max_pages, 64,
                              (unsigned)L::kRows);
  if (e != cudaSuccess) return e;
  CsParams p{kv.summaries, a.q, kv.seq_lens, a.lists, a.lens, a.err, kv.num_q_heads,
             kv.num_kv_heads, kv.page_size, kv.max_pages, 1.0f / sqrtf((float)D), a.gamma,
             a.budget, kCsPrefetchPieces, kv.block_table, kv.k_cache, kv.v_cache,
             kv.num_phys_pages, kCsKvPrefetchPages, a.k_new, a.v_new};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kv.batch * kv.num_kv_heads * C);
  cfg.blockDim = dim3(kCsThreads);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, cluster_select_kernel<D, G, C, Append>, tm, p);
}

// Clusters of C CTAs that the current device runs at once (0: none fit).
template <int D, int G, int C>
int active_clusters() {
  using L = CsLayout<D, G>;
  const void* fn = (const void*)cluster_select_kernel<D, G, C, false>;
  if (set_max_dynamic_smem(fn, L::kBytes) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(kCsThreads);
  cfg.dynamicSmemBytes = L::kBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, cluster_select_kernel<D, G, C, false>, &cfg) != cudaSuccess)
    return 0;
  return n;
}

// Per (device, D, G, C): clusters resident at once, looked up on first use.
template <int D, int G, int C>
int resident_clusters() {
  static std::mutex mu;
  static int cache[64];
  static bool known[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!known[dev]) {
    cache[dev] = active_clusters<D, G, C>();
    known[dev] = true;
  }
  return cache[dev];
}

template <int D, int G>
cudaError_t launch_cs_c(const SelectArgs& a, int C, cudaStream_t stream) {
  switch (C) {
    case 1: return a.k_new ? launch_cs<D, G, 1, true>(a, stream) : launch_cs<D, G, 1, false>(a, stream);
    case 2: return a.k_new ? launch_cs<D, G, 2, true>(a, stream) : launch_cs<D, G, 2, false>(a, stream);
    case 4: return a.k_new ? launch_cs<D, G, 4, true>(a, stream) : launch_cs<D, G, 4, false>(a, stream);
  }
  return cudaErrorInvalidValue;
}

template <int D, int G>
int resident_c(int C) {
  switch (C) {
    case 1: return resident_clusters<D, G, 1>();
    case 2: return resident_clusters<D, G, 2>();
    case 4: return resident_clusters<D, G, 4>();
  }
  return 0;
}

template <int D>
cudaError_t launch_cs_g(const SelectArgs& a, int C, cudaStream_t stream) {
  switch (a.kv->num_q_heads / a.kv->num_kv_heads) {
    case 1: return launch_cs_c<D, 1>(a, C, stream);
    case 2: return launch_cs_c<D, 2>(a, C, stream);
    case 4: return launch_cs_c<D, 4>(a, C, stream);
    case 8: return launch_cs_c<D, 8>(a, C, stream);
  }
  return cudaErrorInvalidValue;
}

template <int D>
int resident_g(const asp_paged_kv& kv, int C) {
  switch (kv.num_q_heads / kv.num_kv_heads) {
    case 1: return resident_c<D, 1>(C);
    case 2: return resident_c<D, 2>(C);
    case 4: return resident_c<D, 4>(C);
    case 8: return resident_c<D, 8>(C);
  }
  return 0;
}

}  // namespace

int cluster_select_ctas(const asp_paged_kv& kv, int num_sms) {
  if (kv.max_pages < kClusterSelectMinPages || kv.max_pages > kCsMaxC * kCsPages) return 0;
  const int S = kv.batch * kv.num_kv_heads;
  int C = 1;
  while (C * kCsPages < kv.max_pages) C *= 2;
  // spread each segment over more SMs while the grid would leave a quarter idle
  while (C < kCsMaxC && S * C * 4 < num_sms * 3) C *= 2;
  // Every cluster pays the selection's latency (~8 us) once: only when all of
  // them run in one wave does that beat the two-kernel path, whose score pass
  // spreads every page over the whole GPU and whose select kernel runs a
  // 1024-thread CTA per segment (at 128k one wave: 32 clusters of 4 CTAs;
  // with 64 requests of up to 8192 pages, 512 clusters of 4 would take 14).
  const int n = kv.head_dim == 128 ? resident_g<128>(kv, C) : resident_g<64>(kv, C);
  return n >= S ? C : 0;
}

cudaError_t launch_cluster_select(const SelectArgs& a, int C, cudaStream_t stream) {
  return a.kv->head_dim == 128 ? launch_cs_g<128>(a, C, stream) : launch_cs_g<64>(a, C, stream);
}

}  // namespace asp
