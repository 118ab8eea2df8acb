// select.cu - coverage selection (MOIRA abstract: per request, layer, KV
// head and step, keep the smallest page set whose estimated attention mass
// reaches gamma). Two kernels:
//
// score_kernel   HBM-bound stream over the page summaries, which are kept in
//                logical page order per (request, KV head) segment. Every
//                warp of a persistent grid streams its own even slice of all
//                segments' pages in 4 KiB pieces into a private mbarrier ring
//                (no warp waits on another). The Quest bound
//                sum_i max(q_i*mn_i, q_i*mx_i) = sum_i q-_i*mn_i + q+_i*mx_i
//                is a dense contraction of the group's queries with 2d
//                summary channels per page, so it runs on the tensor cores
//                (mma.sync m16n8k16, 8 pages per tile) with each fp32 query
//                split into three bf16 terms: the dot products keep fp32
//                precision (bf16 queries alone would move scores by ~1e-3
//                and change lists) at a few instructions per page, which
//                leaves the pass bound by HBM rather than by issue.
//                (Gathering 512-byte per-(page, head) summaries scattered by
//                the block table runs at under half the copy bandwidth;
//                contiguous runs reach it.)
//
// select_kernel  One CTA (1024 threads) per segment. Softmax weights
//                exp(s - max) are turned into fixed point (2^37 = weight of
//                the top page on segments of up to 8192 pages, 2^42 on
//                longer ones), so every sum is exact and order-independent
//                and the result is deterministic. Rounding each weight to
//                the unit errs by at most half a unit per page, i.e. by at
//                most N * 2^-38 (N <= 8192: 3.0e-8) or N * 2^-43 (N <= 2^20:
//                1.2e-7) of the total mass. A first pass histograms
//                the weights over 4096 bins linear in max - s; the bin where
//                the running weight from the top reaches gamma times the
//                total is one interval of score keys, usually a handful of
//                pages, which one warp resolves exactly (exact radix rounds
//                over the keys when many pages tie closely). Ties at the
//                cutoff go to the lower page ids; per-warp ballots and one
//                scan compact the kept ids in ascending order. Segments of
//                up to 8192 pages keep scores and weights in registers;
//                longer ones read them from global memory (that general path
//                is compiled out of the variant launched when max_pages is
//                at most 8192).

#include "score_common.cuh"

#include <type_traits>

namespace asp {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ============================================================== score kernel
constexpr int kScoreWarps = 8;
constexpr int kScoreThreads = kScoreWarps * 32;

struct ScoreParams {
  uint16_t* summ;  // written only by the fused append
  const float* q;
  const int32_t* seq_lens;
  float* scores;
  uint32_t* err;
  int B, Hq, Hkv, P, max_pages;
  float inv_sqrt_d;
  // fused append (null k_new: none): new token rows bf16 [B, Hkv, d]
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_cache;
  uint16_t* v_cache;
  const int32_t* bt;
  int num_phys;
  int pf_pieces;  // pieces per warp fetched into L2 before the predecessor ends
};

// Summaries are stored per segment (request b, KV head h) in logical page
// order, so this pass is one sequential stream with no block-table lookups.
// The concatenated page space of all segments (segment-major) is split evenly
// over the warps of a persistent grid. Each warp walks its slice as pieces of
// up to 4 KiB of one segment's pages; lane p bulk-copies page p of a piece
// into the warp's own ring of slots (one mbarrier per slot, so no warp ever
// waits on another). The scores of 8 pages at a time come from
// score::GroupQuery (the group's queries against the pages' summaries on the
// tensor cores).
template <int D, int G>
struct ScoreCfg : score::Cfg<D, G> {
  static constexpr int kCtas = score::Cfg<D, G>::kBlocks > 2 ? 1 : 2;  // CTAs per SM (registers)
  static constexpr int kSlots = kCtas == 2 ? 3 : 6;                     // ring depth per warp
};

// Position in a warp's slice: segment (b, h), logical page lp, and the index
// in the concatenated page space. Every lane of the warp holds the same one.
struct SegCursor {
  int b, h, lp, pos;
};

template <int D, int G, bool Append>
__global__ void __launch_bounds__(kScoreThreads, ScoreCfg<D, G>::kCtas)
    score_kernel(ScoreParams p) {
  using C = ScoreCfg<D, G>;
  constexpr int kPiecePages = C::kPiecePages, kPageBytes = C::kPageBytes, kStride = C::kStride;
  constexpr int kSlots = C::kSlots;
  extern __shared__ __align__(128) uint8_t score_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kRingBytes = kScoreWarps * kSlots * C::kSlotBytes;
  uint8_t* ring = score_smem + warp * kSlots * C::kSlotBytes;  // this warp's slots
  uint64_t* full = reinterpret_cast<uint64_t*>(score_smem + kRingBytes) + warp * kSlots;
  int* rprefix = reinterpret_cast<int*>(score_smem + kRingBytes +
                                        kScoreWarps * kSlots * sizeof(uint64_t));  // [B + 1]
  int* tlen = rprefix + p.B + 1;  // [B] clamped sequence lengths (for the fused append)
  int* pre = tlen + p.B;          // [B + 1] the early plan's prefix (below)

  if (lane == 0) {
    for (int i = 0; i < kSlots; ++i) mbar_init(&full[i], 1);
    mbar_fence_init();
  }
  pdl_launch_dependents();
  // Until the previous kernel in the stream finishes, HBM is mostly idle and
  // this grid is resident but may read nothing that kernel writes. Each warp
  // plans its slice from a racy read of seq_lens (bypassing L1) and asks L2
  // for its first pieces. A prefetch only moves lines into L2, which every
  // write passes through, so a stale length costs a useless prefetch and
  // never a wrong result; the plan is redone from scratch after the wait.
  if (p.pf_pieces > 0) {
    if (warp == 0) {
      int carry = 0;
      if (lane == 0) pre[0] = 0;
      for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int n = 0;
        if (b < p.B) {
          const long long T = __ldcg(p.seq_lens + b);
          const long long cap = (long long)p.max_pages * p.P;
          n = ceil_div((int)(T < 0 ? 0 : (T > cap ? cap : T)), p.P);
        }
        int x = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(kFull, x, o);
          if (lane >= o) x += y;
        }
        if (b < p.B) pre[b + 1] = carry + x;
        carry += __shfl_sync(kFull, x, 31);
      }
    }
    __syncthreads();
    const EvenSplit sp(p.Hkv * pre[p.B], gridDim.x * kScoreWarps);
    const int gw = blockIdx.x * kScoreWarps + warp;
    int pos = sp.begin(gw);
    const int pend = sp.end(gw);
    if (pos < pend) {
      int b = 0, hi = p.B - 1;  // the request holding page pos (N_b > 0)
      while (b < hi) {
        const int mid = (b + hi + 1) >> 1;
        if (p.Hkv * pre[mid] <= pos) b = mid; else hi = mid - 1;
      }
      const int off = pos - p.Hkv * pre[b];
      int h = off / (pre[b + 1] - pre[b]), lp = off % (pre[b + 1] - pre[b]);
      for (int k = 0; k < p.pf_pieces && pos < pend; ++k) {
        const int nb = pre[b + 1] - pre[b];
        const int n = min(min(kPiecePages, nb - lp), pend - pos);
        if (lane < n) {
          const size_t page = ((size_t)b * p.Hkv + h) * p.max_pages + lp + lane;
          prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(p.summ) + page * kPageBytes,
                           kPageBytes);
        }
        pos += n;
        lp += n;
        if (lp == nb) {
          lp = 0;
          if (++h == p.Hkv) {
            h = 0;
            do ++b; while (b < p.B && pre[b + 1] == pre[b]);
          }
        }
      }
    }
  }
  pdl_wait_predecessor();
  // prefix of the requests' page counts N_b (clamped sequence lengths)
  if (warp == 0) {
    int carry = 0;
    if (lane == 0) rprefix[0] = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < p.B) {
        const int T = clamp_seq_len(p.seq_lens[b], p.max_pages, p.P, p.err);
        if (Append) tlen[b] = T;
        n = ceil_div(T, p.P);
      }
      int x = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      if (b < p.B) rprefix[b + 1] = carry + x;
      carry += __shfl_sync(kFull, x, 31);
    }
  }
  __syncthreads();
  // this warp's slice of the Hkv * sum_b N_b pages (< 2^31, checked on the host)
  const EvenSplit split(p.Hkv * rprefix[p.B], gridDim.x * kScoreWarps);
  const int gw = blockIdx.x * kScoreWarps + warp;
  const int wbeg = split.begin(gw), wend = split.end(gw);
  if (wbeg >= wend) return;

  auto seg_pages = [&](int b) { return rprefix[b + 1] - rprefix[b]; };
  SegCursor ic;  // issue cursor: the request holding page wbeg has N_b > 0
  {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.Hkv * rprefix[mid] <= wbeg) lo = mid; else hi = mid - 1;
    }
    const int n = seg_pages(lo), off = wbeg - p.Hkv * rprefix[lo];
    ic = SegCursor{lo, off / n, off % n, wbeg};
  }
  SegCursor cc = ic;  // consume cursor: the same sequence of pieces, later
  auto piece_pages = [&](const SegCursor& c) {
    return min(min(kPiecePages, seg_pages(c.b) - c.lp), wend - c.pos);
  };
  auto advance = [&](SegCursor& c, int n) {
    c.pos += n;
    c.lp += n;
    if (c.lp == seg_pages(c.b)) {
      c.lp = 0;
      if (++c.h == p.Hkv) {
        c.h = 0;
        do ++c.b; while (c.b < p.B && seg_pages(c.b) == 0);
      }
    }
  };
  const uint64_t pol = l2_evict_first_policy();  // summaries are read once per call
  int issued = 0;
  // Fused append (asp_coverage_select_append): before the piece that holds
  // a segment's last page is copied, its warp writes the new token's K and V
  // rows and folds the key into that page's summary (a fresh page, slot 0,
  // takes the key as both bounds), exactly as the APPEND summarize does.
  using LV = typename std::conditional<D == 128, uint2, uint32_t>::type;  // d / 32 channels
  constexpr int kLRow = 2 * D / (int)sizeof(LV);                          // lane units per row
  auto append_token = [&](int b, int h, int lp_last) {
    const int T = tlen[b], slot = (T - 1) % p.P;
    const int phys = __ldg(p.bt + (size_t)b * p.max_pages + lp_last);
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
    LV* sm = reinterpret_cast<LV*>(p.summ + (unit * p.max_pages + lp_last) * 2 * D) + lane;
    if (slot == 0) {
      sm[0] = kn;
      sm[kLRow] = kn;
    } else {
      sm[0] = vmin(sm[0], kn);
      sm[kLRow] = vmax(sm[kLRow], kn);
    }
  };
  auto issue = [&]() {  // next piece of the slice into slot issued % kSlots
    const int n = piece_pages(ic);
    const int slot = issued % kSlots;
    const bool app = Append && ic.lp + n == seg_pages(ic.b);  // warp-uniform
    if (app) append_token(ic.b, ic.h, ic.lp + n - 1);
    if (lane == 0) mbar_arrive_expect_tx(&full[slot], n * kPageBytes);
    __syncwarp();
    if (app) fence_proxy_async_global();  // the fold, before this warp's copy reads the page
    if (lane < n) {
      const size_t page = ((size_t)ic.b * p.Hkv + ic.h) * p.max_pages + ic.lp + lane;
      bulk_g2s_hint(ring + slot * C::kSlotBytes + lane * kStride,
                    reinterpret_cast<const uint8_t*>(p.summ) + page * kPageBytes, kPageBytes,
                    &full[slot], pol);
    }
    advance(ic, n);
    ++issued;
  };
  for (int k = 0; k < kSlots && ic.pos < wend; ++k) issue();

  const int g = lane >> 2, t = lane & 3;
  score::GroupQuery<D, G> gq;
  auto load_q = [&](int b, int h) { gq.load(p.q + ((size_t)b * p.Hq + h * G) * D, lane); };
  int qseg = cc.b * p.Hkv + cc.h, k = 0;
  load_q(cc.b, cc.h);  // the first piece's queries load while its copies fly
  bool aborted = false;
  const uint32_t lane_row = score::GroupQuery<D, G>::lane_row(lane);
#pragma unroll 1
  for (; cc.pos < wend; ++k) {
    const int slot = k % kSlots;
    if (!__all_sync(kFull, mbar_wait(&full[slot], (k / kSlots) & 1))) {
      if (lane == 0) report(p.err, ASP_DEVERR_TIMEOUT);
      aborted = true;
      break;
    }
    const int n = piece_pages(cc), seg = cc.b * p.Hkv + cc.h;
    if (seg != qseg) {
      load_q(cc.b, cc.h);
      qseg = seg;
    }
    const uint32_t sb = smem_u32(ring + slot * C::kSlotBytes) + lane_row;
    float* out = p.scores + (size_t)seg * p.max_pages + cc.lp;
#pragma unroll
    for (int nt = 0; nt < kPiecePages / 8; ++nt) {
      if (nt * 8 >= n) break;  // warp-uniform
      float x0, x1;
      gq.tile(sb + nt * 8 * kStride, x0, x1);
      const int pg = nt * 8 + 2 * t;
      if (g == 0) {
        if (pg < n) out[pg] = x0 * p.inv_sqrt_d;
        if (pg + 1 < n) out[pg + 1] = x1 * p.inv_sqrt_d;
      }
    }
    advance(cc, n);
    __syncwarp();  // every lane is done reading the slot
    if (ic.pos < wend) {
      fence_proxy_async_smem();
      issue();
    }
  }
  // never leave with copies in flight (only after a timeout can any remain)
  if (aborted && lane == 0)
    for (int j = k; j < issued; ++j) mbar_wait(&full[j % kSlots], (j / kSlots) & 1);
}

// ============================================================= select kernel
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCache = 8192;  // N up to this: the fast path (scores in registers and smem)
constexpr int kPer = kSelCache / kSelThreads;  // elements per thread on the fast path
constexpr int kBins = 256;
constexpr int kLimbBits = 14;    // mass = l0 + l1 << 14 + l2 << 28, each limb < 2^14
constexpr int kWarpCand = 4096;  // candidates one warp finishes on (fits the histogram area)
constexpr int kLinBins = 4096;   // bins of the first, linear round
constexpr int kLinLoBits = 19;   // fast path: a weight is lo + hi << 19, both < 2^19
constexpr size_t kSelSmem = (size_t)kSelWarps * kBins * 4 * sizeof(uint32_t) +  // private hists
                            kSelCache * sizeof(float);                            // score cache

struct SelectParams {
  const float* scores;
  const int32_t* seq_lens;
  int32_t* lists;
  int32_t* lens;
  uint32_t* err;
  int Hkv, P, max_pages;
  float gamma;
  int budget;
};

using score::ceil_gamma_times;
using score::key_score;
using score::kUnitFast;
using score::kUnitLong;
using score::mass_fixed;
using score::score_key;

// Block min and max of one float pair in a single pass (scratch: 2 x warps).
__device__ __forceinline__ void block_minmax(float& mn, float& mx, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  }
  if (lane == 0) {
    scratch[warp] = mn;
    scratch[kSelWarps + warp] = mx;
  }
  __syncthreads();
  mn = lane < kSelWarps ? scratch[lane] : INFINITY;
  mx = lane < kSelWarps ? scratch[kSelWarps + lane] : -INFINITY;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  }
  __syncthreads();  // scratch is free again
}

// General = false: every segment fits the fast path (max_pages <= kSelCache,
// known on the host), so the general path is compiled out and the kernel's
// code, fetched afresh on every SM at each launch, is smaller.
template <bool General>
__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectParams p) {
  extern __shared__ __align__(16) uint8_t sel_smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(sel_smem);  // [warp][bin][count, l0, l1, l2]
  float* cache = reinterpret_cast<float*>(hist + kSelWarps * kBins * 4);
  __shared__ uint32_t m_cnt[kBins];
  __shared__ unsigned long long m_mass[kBins];
  __shared__ unsigned long long red_u64[kSelWarps];
  __shared__ uint32_t red_u32[2 * kSelWarps];
  __shared__ float red_f[2 * kSelWarps];
  __shared__ uint32_t pick[4];
  __shared__ unsigned long long pick_m[1];
  __shared__ unsigned long long sel_target, tie_t;  // computed by one thread
  __shared__ uint32_t slab_cnt[kPer * kSelWarps][2];  // fast compaction: (gt, eq) per (slab, warp)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x;
  const int b = s / p.Hkv;
  pdl_launch_dependents();
  pdl_wait_predecessor();
  const int T = clamp_seq_len(p.seq_lens[b], p.max_pages, p.P, p.err);
  const int N = ceil_div(T, p.P);
  int32_t* out = p.lists + (size_t)s * p.max_pages;
  const bool mass_mode = p.budget <= 0;
  if (N == 0) {
    if (tid == 0) p.lens[s] = 0;
    return;
  }
  if ((!mass_mode && p.budget >= N) || (mass_mode && p.gamma >= 1.0f)) {
    for (int i = tid; i < N; i += kSelThreads) out[i] = i;
    if (tid == 0) p.lens[s] = N;
    return;
  }
  const float* gsc = p.scores + (size_t)s * p.max_pages;
  // fast path: element k of this thread is page id k * kSelThreads + tid, so a
  // warp's elements of one slab k are 32 consecutive ids
  const bool fast = !General || N <= kSelCache;
  float v[kPer];
  float lo_s = INFINITY, hi_s = -INFINITY;
  if (fast) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = k * kSelThreads + tid;
      v[k] = -INFINITY;
      if (i < N) {
        v[k] = gsc[i];
        cache[i] = v[k];
        lo_s = fminf(lo_s, v[k]);
        hi_s = fmaxf(hi_s, v[k]);
      }
    }
  } else {
    for (int i = tid; i < N; i += kSelThreads) {
      const float x = gsc[i];
      lo_s = fminf(lo_s, x);
      hi_s = fmaxf(hi_s, x);
    }
  }
  block_minmax(lo_s, hi_s, red_f);
  const float* sc = fast ? cache : gsc;
  const float smax = hi_s;
  const float unit = fast ? kUnitFast : kUnitLong;
  auto weight = [&](float x) -> unsigned long long {
    return mass_mode ? mass_fixed(x, smax, unit) : 1ull;
  };

  // selection weights: fixed-point softmax mass, or 1 in budget mode. The
  // target (gamma times the total mass) comes out of the first pass's bin scan.
  unsigned long long mw[kPer];
  unsigned long long target = (unsigned long long)p.budget;
  if (fast) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) mw[k] = k * kSelThreads + tid < N ? weight(v[k]) : 0ull;
  }

  // state of the cutoff search: candidates are the keys in [lo, hi]; above_m
  // (above_c) is the weight (count) of every element with a larger key
  uint32_t lo = 0, hi = 0;
  unsigned long long above_m = 0;
  uint32_t above_c = 0, cnt_eq = 0;
  uint32_t* my_hist = hist + warp * kBins * 4;
  constexpr uint32_t kLimbMask = (1u << kLimbBits) - 1u;

  // First pass: one histogram of bins linear in the distance from the top score,
  // smax - s, over at most 28 units in mass mode, 31 on the general path (a
  // page further down has zero fixed-point mass). The bin index never increases with the score, so
  // the bin where the running weight from the top reaches the target holds
  // one interval of keys, usually a handful.
  // (28 units: e^-28 * 2^37 < 0.5; 31 units: e^-31 * 2^42 < 0.5)
  const float span = mass_mode ? fminf(hi_s - lo_s, fast ? 28.f : 31.f) : hi_s - lo_s;
  const float inv_w = span > 0.f ? (float)kLinBins / span : 0.f;
  auto lin_bin = [&](float x) { return min(kLinBins - 1, (int)((smax - x) * inv_w)); };
  int jbin;
  {
    uint32_t* lin_lo = hist;             // fast: weight limbs; general: count
    uint32_t* lin_hi = hist + kLinBins;  // fast: weight limbs
    unsigned long long* lin_w = reinterpret_cast<unsigned long long*>(hist + kLinBins);  // general
    const int words = fast ? 2 * kLinBins : 3 * kLinBins;
    for (int i = tid; i < words / 4; i += kSelThreads)
      reinterpret_cast<uint4*>(hist)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) pick[3] = 0;  // candidate counter of the fast path
    __syncthreads();
    if (fast) {
#pragma unroll
      for (int k = 0; k < kPer; ++k)
        if (mw[k]) {
          const int bin = lin_bin(v[k]);
          atomicAdd(&lin_lo[bin], (uint32_t)mw[k] & ((1u << kLinLoBits) - 1u));
          const uint32_t h = (uint32_t)(mw[k] >> kLinLoBits);
          if (h) atomicAdd(&lin_hi[bin], h);
        }
    } else {
      for (int i = tid; i < N; i += kSelThreads) {
        const float x = sc[i];
        const int bin = lin_bin(x);
        atomicAdd(&lin_lo[bin], 1u);
        atomicAdd(&lin_w[bin], weight(x));
      }
    }
    __syncthreads();
    // block scan over the bins; thread tid owns bins [kPb tid, kPb tid + kPb)
    constexpr int kPb = kLinBins / kSelThreads;
    unsigned long long w[kPb], ws = 0;
    uint32_t c[kPb], cs = 0;
#pragma unroll
    for (int u = 0; u < kPb; ++u) {
      const int bin = tid * kPb + u;
      w[u] = fast ? lin_lo[bin] + ((unsigned long long)lin_hi[bin] << kLinLoBits) : lin_w[bin];
      c[u] = fast ? 0u : lin_lo[bin];
      ws += w[u];
      cs += c[u];
    }
    unsigned long long xw = ws;
    uint32_t xc = cs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long yw = __shfl_up_sync(kFull, xw, o);
      if (lane >= o) xw += yw;
    }
    if (!fast) {  // counts per bin exist only on the general path
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t yc = __shfl_up_sync(kFull, xc, o);
        if (lane >= o) xc += yc;
      }
    }
    if (lane == 31) {
      red_u64[warp] = xw;
      red_u32[warp] = xc;
    }
    __syncthreads();
    if (warp == 0) {
      const unsigned long long w0 = lane < kSelWarps ? red_u64[lane] : 0ull;
      const uint32_t c0 = lane < kSelWarps ? red_u32[lane] : 0u;
      unsigned long long aw = w0;
      uint32_t ac = c0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long yw = __shfl_up_sync(kFull, aw, o);
        const uint32_t yc = __shfl_up_sync(kFull, ac, o);
        if (lane >= o) {
          aw += yw;
          ac += yc;
        }
      }
      if (lane < kSelWarps) {
        red_u64[lane] = aw - w0;  // exclusive warp offsets
        red_u32[lane] = ac - c0;
      }
      if (lane == 31) {  // gamma times the total weight, once (fp64 is slow on this part)
        unsigned long long tg = target;
        if (mass_mode) {
          tg = ceil_gamma_times(p.gamma, aw);
          if (tg < 1) tg = 1;
        }
        sel_target = tg;
      }
    }
    __syncthreads();
    target = sel_target;
    unsigned long long run_w = red_u64[warp] + xw - ws;
    uint32_t run_c = red_u32[warp] + xc - cs;
    // exactly one bin has run_w < target <= run_w + w (target <= total weight)
#pragma unroll
    for (int u = 0; u < kPb; ++u) {
      if (run_w < target && run_w + w[u] >= target) {
        pick[0] = (uint32_t)(tid * kPb + u);
        pick[1] = run_c;
        pick[2] = c[u];
        pick_m[0] = run_w;
      }
      run_w += w[u];
      run_c += c[u];
    }
    __syncthreads();  // every thread has read the total; pick[] holds the bin
    jbin = (int)pick[0];
    above_m = pick_m[0];
    // counts are tracked only where the weight is not already a count
    above_c = fast ? (mass_mode ? 0u : (uint32_t)above_m) : pick[1];
    cnt_eq = pick[2];
    __syncthreads();  // pick[0..2] are rewritten below
  }

  // warp 0: lane owns bins [8*lane, 8*lane+8) of m_cnt/m_mass; finds the
  // largest bin j with above + (sum over bins >= j) >= target
  auto pick_bin = [&]() {
    unsigned long long lm = 0;
    uint32_t lc = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lm += m_mass[lane * 8 + i];
      lc += m_cnt[lane * 8 + i];
    }
    unsigned long long sm = lm;  // inclusive suffix over lanes >= lane
    uint32_t scn = lc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long ym = __shfl_down_sync(kFull, sm, o);
      const uint32_t yc = __shfl_down_sync(kFull, scn, o);
      if (lane + o < 32) {
        sm += ym;
        scn += yc;
      }
    }
    const bool reach = mass_mode ? (above_m + sm >= target)
                                 : ((unsigned long long)above_c + scn >= target);
    const unsigned ballot = __ballot_sync(kFull, reach);
    const int lstar = ballot ? 31 - __clz(ballot) : 0;  // lane 0 reaches by the invariant
    if (lane == lstar) {
      unsigned long long run_m = above_m + (sm - lm);
      uint32_t run_c = above_c + (scn - lc);
      int j = lane * 8;
      for (int i = 7; i >= 0; --i) {
        const int bin = lane * 8 + i;
        const unsigned long long nm = run_m + m_mass[bin];
        const uint32_t nc = run_c + m_cnt[bin];
        if (mass_mode ? (nm >= target) : ((unsigned long long)nc >= target)) {
          j = bin;
          break;
        }
        run_m = nm;
        run_c = nc;
      }
      pick[0] = (uint32_t)j;
      pick[1] = run_c;
      pick[2] = m_cnt[j];
      pick_m[0] = run_m;
    }
  };
  // narrows [lo, hi] to the picked bin; returns the shift the round used
  auto narrow = [&](int shift) {
    const uint32_t j = pick[0];
    above_c = pick[1];
    cnt_eq = pick[2];
    above_m = pick_m[0];
    const unsigned long long nlo = (unsigned long long)lo + ((unsigned long long)j << shift);
    const unsigned long long nhi = nlo + ((1ull << shift) - 1ull);
    lo = (uint32_t)nlo;
    hi = nhi < hi ? (uint32_t)nhi : hi;
  };
  auto shift_of = [&]() {
    const uint32_t range = hi - lo;
    const int bits = range ? 32 - __clz(range) : 0;
    return bits > 8 ? bits - 8 : 0;
  };
  // Exact radix rounds on the keys in [lo, hi] until one key is left: block
  // rounds over every element while more than kWarpCand remain, then warp 0
  // alone on the gathered candidates. Leaves the cutoff key in lo.
  auto radix_resolve = [&]() {
    bool resolved = lo == hi;
    while (!resolved && cnt_eq > kWarpCand) {
      const int shift = shift_of();
      for (int i = tid; i < kSelWarps * kBins; i += kSelThreads)
        reinterpret_cast<uint4*>(hist)[i] = make_uint4(0, 0, 0, 0);
      __syncthreads();
      for (int i = tid; i < N; i += kSelThreads) {
        const float x = sc[i];
        const uint32_t k = score_key(x);
        if (k >= lo && k <= hi) {
          uint32_t* h = my_hist + ((k - lo) >> shift) * 4;
          atomicAdd(h, 1u);
          if (mass_mode) {
            const unsigned long long m = mass_fixed(x, smax, unit);
            atomicAdd(h + 1, (uint32_t)m & kLimbMask);
            atomicAdd(h + 2, (uint32_t)(m >> kLimbBits) & kLimbMask);
            atomicAdd(h + 3, (uint32_t)(m >> (2 * kLimbBits)));
          }
        }
      }
      __syncthreads();
      if (tid < kBins) {  // merge the private histograms of bin tid
        uint32_t c = 0;
        unsigned long long l0 = 0, l1 = 0, l2 = 0;
        for (int w = 0; w < kSelWarps; ++w) {
          const uint4 h = reinterpret_cast<const uint4*>(hist)[w * kBins + tid];
          c += h.x;
          l0 += h.y;
          l1 += h.z;
          l2 += h.w;
        }
        m_cnt[tid] = c;
        m_mass[tid] = l0 + (l1 << kLimbBits) + (l2 << (2 * kLimbBits));
      }
      __syncthreads();
      if (warp == 0) pick_bin();
      __syncthreads();
      narrow(shift);
      resolved = shift == 0;
      __syncthreads();
    }
    if (!resolved) {
      // gather the candidates (scores with keys in [lo, hi]) and let warp 0
      // run the remaining rounds on them with warp-level synchronisation only
      float* cand = reinterpret_cast<float*>(hist + kBins * 4);  // after warp 0's histogram
      if (tid == 0) pick[3] = 0;
      __syncthreads();
      for (int i = tid; i < N; i += kSelThreads) {
        const float x = sc[i];
        const uint32_t k = score_key(x);
        if (k >= lo && k <= hi) cand[atomicAdd(&pick[3], 1u)] = x;
      }
      __syncthreads();
      if (warp == 0) {
        const int nc = (int)pick[3];
        while (true) {
          const int shift = shift_of();
          for (int i = lane; i < kBins; i += 32)
            reinterpret_cast<uint4*>(hist)[i] = make_uint4(0, 0, 0, 0);
          __syncwarp();
          for (int i = lane; i < nc; i += 32) {
            const float x = cand[i];
            const uint32_t k = score_key(x);
            if (k >= lo && k <= hi) {
              uint32_t* h = hist + ((k - lo) >> shift) * 4;
              atomicAdd(h, 1u);
              if (mass_mode) {
                const unsigned long long m = mass_fixed(x, smax, unit);
                atomicAdd(h + 1, (uint32_t)m & kLimbMask);
                atomicAdd(h + 2, (uint32_t)(m >> kLimbBits) & kLimbMask);
                atomicAdd(h + 3, (uint32_t)(m >> (2 * kLimbBits)));
              }
            }
          }
          __syncwarp();
          for (int i = lane; i < kBins; i += 32) {
            const uint4 h = reinterpret_cast<const uint4*>(hist)[i];
            m_cnt[i] = h.x;
            m_mass[i] = (unsigned long long)h.y + ((unsigned long long)h.z << kLimbBits) +
                        ((unsigned long long)h.w << (2 * kLimbBits));
          }
          __syncwarp();
          pick_bin();
          __syncwarp();
          narrow(shift);
          __syncwarp();
          if (shift == 0) break;
        }
        if (lane == 0) {  // publish the result for the whole block
          pick[0] = lo;
          pick[1] = above_c;
          pick[2] = cnt_eq;
          pick_m[0] = above_m;
        }
      }
      __syncthreads();
      lo = pick[0];
      above_c = pick[1];
      cnt_eq = pick[2];
      above_m = pick_m[0];
    }
  };
  // ties at the cutoff key tau: keep the first t of the n_eq (lowest ids)
  auto tie_take = [&](uint32_t tau, unsigned long long above_w, unsigned long long n_eq) {
    unsigned long long t;
    if (mass_mode) {
      // t = ceil(rem / w): a float estimate corrected exactly in integers
      const unsigned long long w = mass_fixed(key_score(tau), smax, unit);
      const unsigned long long rem = target - above_w;
      if (w) {
        const float est = ceilf((float)rem / (float)w);
        t = est > (float)n_eq ? n_eq : (unsigned long long)est;
        while (t < n_eq && t * w < rem) ++t;
        while (t > 1 && (t - 1) * w >= rem) --t;
      } else {
        t = n_eq;
      }
    } else {
      t = target - above_w;
    }
    if (t < 1) t = 1;
    if (t > n_eq) t = n_eq;
    return t;
  };

  // Mass mode, fast path: the tie count before its clamp to [1, n_eq],
  // ceil((target - above_w) / w(tau)), computed by one thread as soon as tau
  // is known so that it stays off the compaction's critical path. Counts
  // from 2^22 up exceed every n_eq (at most 2^20) and need no refinement;
  // below that the float estimate is within one of the exact value.
  auto tie_mass = [&](uint32_t tau, unsigned long long above_w) -> unsigned long long {
    const unsigned long long w = mass_fixed(key_score(tau), smax, unit);
    if (!w) return 1ull << 40;  // ties of zero mass: all of them
    const unsigned long long rem = target - above_w;
    const float est = ceilf((float)rem / (float)w);
    if (est >= 4194304.0f) return 1ull << 40;
    unsigned long long t = (unsigned long long)est;
    while (t * w < rem) ++t;
    while (t > 1 && (t - 1) * w >= rem) --t;
    return t;
  };

  if (fast) {
    // candidates of the cutoff bin (weights recomputed from the scores)
    float* cand = reinterpret_cast<float*>(hist + kBins * 4);
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (k * kSelThreads + tid < N && lin_bin(v[k]) == jbin) {
        const uint32_t idx = atomicAdd(&pick[3], 1u);
        if (idx < kWarpCand) cand[idx] = v[k];
      }
    __syncthreads();
    const uint32_t nc = pick[3];
    if (nc <= 32) {
      // one candidate per lane: tau is the largest key whose weight from the
      // top, ties included, reaches the target
      if (warp == 0) {
        const bool has = lane < (int)nc;
        const float cv = has ? cand[lane] : 0.f;
        const uint32_t ck = score_key(cv);
        const unsigned long long cm = has ? weight(cv) : 0ull;
        unsigned long long gt_w = 0, ge_w = 0;
        for (int o = 0; o < (int)nc; ++o) {
          const uint32_t k2 = __shfl_sync(kFull, ck, o);
          const unsigned long long m2 = __shfl_sync(kFull, cm, o);
          if (k2 > ck) gt_w += m2;
          if (k2 >= ck) ge_w += m2;
        }
        const bool reach = has && above_m + ge_w >= target;
        uint32_t best = reach ? ck : 0u;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) best = max(best, __shfl_xor_sync(kFull, best, o));
        const unsigned at = __ballot_sync(kFull, has && reach && ck == best);
        if (lane == __ffs(at) - 1) {
          pick[0] = best;
          pick_m[0] = above_m + gt_w;
          if (mass_mode) tie_t = tie_mass(best, above_m + gt_w);
        }
      }
      __syncthreads();
      lo = pick[0];
      above_m = pick_m[0];
    } else {
      // many candidates: the key interval of the bin, then exact radix rounds
      uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
      for (int k = 0; k < kPer; ++k)
        if (k * kSelThreads + tid < N && lin_bin(v[k]) == jbin) {
          const uint32_t key = score_key(v[k]);
          kmin = min(kmin, key);
          kmax = max(kmax, key);
        }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
        kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
      }
      if (lane == 0) {
        red_u32[warp] = kmin;
        red_u32[kSelWarps + warp] = kmax;
      }
      __syncthreads();
      kmin = lane < kSelWarps ? red_u32[lane] : 0xffffffffu;
      kmax = lane < kSelWarps ? red_u32[kSelWarps + lane] : 0u;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
        kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
      }
      lo = kmin;
      hi = kmax;
      cnt_eq = nc;
      __syncthreads();
      radix_resolve();
      if (tid == 0 && mass_mode) tie_t = tie_mass(lo, above_m);
    }
    const uint32_t tau = lo;
    // compaction in id order: per (slab, warp) counts of keys above and at
    // tau, one warp-0 scan over them, then every thread writes its kept ids
    uint32_t gtm[kPer], eqm[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const bool valid = k * kSelThreads + tid < N;
      const uint32_t key = score_key(v[k]);
      gtm[k] = __ballot_sync(kFull, valid && key > tau);
      eqm[k] = __ballot_sync(kFull, valid && key == tau);
      if (lane == 0) {
        slab_cnt[k * kSelWarps + warp][0] = __popc(gtm[k]);
        slab_cnt[k * kSelWarps + warp][1] = __popc(eqm[k]);
      }
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scan over the kPer * kSelWarps entries in id order
      constexpr int kE = kPer * kSelWarps / 32;
      uint32_t g[kE], e[kE], gs = 0, es = 0;
#pragma unroll
      for (int u = 0; u < kE; ++u) {
        g[u] = slab_cnt[lane * kE + u][0];
        e[u] = slab_cnt[lane * kE + u][1];
        gs += g[u];
        es += e[u];
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
        rg += g[u];
        re += e[u];
      }
      if (lane == 31) {
        pick[1] = xg;  // keys above tau
        const unsigned long long t0 = mass_mode ? tie_t : target - xg;
        tie_t = t0 < 1 ? 1 : (t0 > xe ? (unsigned long long)xe : t0);
      }
    }
    __syncthreads();
    const uint32_t n_gt = pick[1];
    const unsigned long long t = tie_t;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const uint32_t gb = slab_cnt[k * kSelWarps + warp][0] + __popc(gtm[k] & lt);
      const uint32_t eb = slab_cnt[k * kSelWarps + warp][1] + __popc(eqm[k] & lt);
      const bool is_gt = (gtm[k] >> lane) & 1u, is_eq = (eqm[k] >> lane) & 1u;
      if (is_gt || (is_eq && eb < t))
        out[gb + (uint32_t)min((unsigned long long)eb, t)] = k * kSelThreads + tid;
    }
    if (tid == 0) p.lens[s] = (int32_t)(n_gt + t);
    return;
  }

  // ---- general path (N > kSelCache): the bin's key interval, exact rounds
  {
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int i = tid; i < N; i += kSelThreads) {
      const float x = sc[i];
      if (lin_bin(x) == jbin) {
        const uint32_t k = score_key(x);
        kmin = min(kmin, k);
        kmax = max(kmax, k);
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
    }
    if (lane == 0) {
      red_u32[warp] = kmin;
      red_u32[kSelWarps + warp] = kmax;
    }
    __syncthreads();
    kmin = lane < kSelWarps ? red_u32[lane] : 0xffffffffu;
    kmax = lane < kSelWarps ? red_u32[kSelWarps + lane] : 0u;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
    }
    lo = kmin;
    hi = kmax;
    __syncthreads();
  }
  radix_resolve();
  const uint32_t tau = lo;
  if (tid == 0) tie_t = tie_take(tau, mass_mode ? above_m : above_c, cnt_eq);
  __syncthreads();
  const unsigned long long t = tie_t;

  // compaction in id order: thread owns ids [i0, i1)
  const int ipt = ceil_div(N, kSelThreads);
  const int i0 = min(N, tid * ipt), i1 = min(N, i0 + ipt);
  uint32_t gt = 0, eq = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t k = score_key(sc[i]);
    gt += k > tau;
    eq += k == tau;
  }
  // block exclusive scan of (gt, eq) packed as hi/lo 32 bits
  unsigned long long pv = ((unsigned long long)gt << 32) | eq, x = pv;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red_u64[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = lane < kSelWarps ? red_u64[lane] : 0ull, xx = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, xx, o);
      if (lane >= o) xx += y;
    }
    if (lane < kSelWarps) red_u64[lane] = xx - w;  // exclusive warp offsets
  }
  __syncthreads();
  const unsigned long long pre = red_u64[warp] + x - pv;
  const uint32_t gt_pre = (uint32_t)(pre >> 32), eq_pre = (uint32_t)(pre & 0xffffffffu);
  uint32_t pos = gt_pre + (uint32_t)min((unsigned long long)eq_pre, t);
  uint32_t eq_rank = eq_pre;
  for (int i = i0; i < i1; ++i) {
    const uint32_t k = score_key(sc[i]);
    if (k > tau) {
      out[pos++] = i;
    } else if (k == tau) {
      if (eq_rank < t) out[pos++] = i;
      ++eq_rank;
    }
  }
  if (tid == 0) p.lens[s] = (int32_t)(above_c + t);
}

// Pieces per warp that the score pass fetches into L2 before the previous
// kernel in the stream ends (the first three of its ring: 29 MB over the
// grid at 128k and d = 128). Measured over a 32-layer step at 128k: none
// 356.6 steps/s, one 358.5, two 360.5, three 361.0.
constexpr int kScorePrefetchPieces = 3;

template <int D, int G, bool Append>
cudaError_t launch_score_tt(const SelectArgs& a, cudaStream_t stream) {
  const asp_paged_kv& kv = *a.kv;
  ScoreParams p{kv.summaries, a.q, kv.seq_lens, a.scores, a.err, kv.batch, kv.num_q_heads,
                kv.num_kv_heads, kv.page_size, kv.max_pages, 1.0f / sqrtf((float)D),
                a.k_new, a.v_new, kv.k_cache, kv.v_cache, kv.block_table, kv.num_phys_pages,
                kScorePrefetchPieces};
  using C = ScoreCfg<D, G>;
  const size_t smem = (size_t)kScoreWarps * C::kSlots * (C::kSlotBytes + sizeof(uint64_t)) +
                      (3 * kv.batch + 2) * sizeof(int);
  cudaError_t e = set_max_dynamic_smem((const void*)score_kernel<D, G, Append>, (int)smem);
  if (e != cudaSuccess) return e;
  // persistent: the kernel splits the pages it finds in seq_lens itself
  return launch_pdl(score_kernel<D, G, Append>, dim3(C::kCtas * a.num_sms), dim3(kScoreThreads),
                    smem, stream, p);
}

template <int D, int G>
cudaError_t launch_score_t(const SelectArgs& a, cudaStream_t stream) {
  return a.k_new ? launch_score_tt<D, G, true>(a, stream) : launch_score_tt<D, G, false>(a, stream);
}

template <int D>
cudaError_t launch_score_d(const SelectArgs& a, cudaStream_t stream) {
  switch (a.kv->num_q_heads / a.kv->num_kv_heads) {
    case 1: return launch_score_t<D, 1>(a, stream);
    case 2: return launch_score_t<D, 2>(a, stream);
    case 4: return launch_score_t<D, 4>(a, stream);
    case 8: return launch_score_t<D, 8>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_scores(const SelectArgs& a, cudaStream_t stream) {
  return a.kv->head_dim == 128 ? launch_score_d<128>(a, stream) : launch_score_d<64>(a, stream);
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream) {
  const asp_paged_kv& kv = *a.kv;
  const bool all = a.budget <= 0 && a.gamma >= 1.0f;
  if (!all) {  // one cluster per segment scores (and appends) and selects it in one pass
    const int C = cluster_select_ctas(kv, a.num_sms);
    if (C > 0) return launch_cluster_select(a, C, stream);
  }
  if (!all || a.k_new) {  // gamma >= 1 keeps every page: no scores needed (but the append)
    cudaError_t e = launch_scores(a, stream);
    if (e != cudaSuccess) return e;
  }
  SelectParams p{a.scores, kv.seq_lens, a.lists, a.lens, a.err, kv.num_kv_heads, kv.page_size,
                 kv.max_pages, a.gamma, a.budget};
  const bool general = kv.max_pages > kSelCache;
  const void* fn = general ? (const void*)select_kernel<true> : (const void*)select_kernel<false>;
  cudaError_t e = set_max_dynamic_smem(fn, (int)kSelSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid(kv.batch * kv.num_kv_heads);
  return general ? launch_pdl(select_kernel<true>, grid, dim3(kSelThreads), kSelSmem, stream, p)
                 : launch_pdl(select_kernel<false>, grid, dim3(kSelThreads), kSelSmem, stream, p);
}

}  // namespace asp
