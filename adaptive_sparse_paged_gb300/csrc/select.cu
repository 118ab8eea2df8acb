// select.cu - coverage selection (MOIRA abstract: per request, layer, KV
// head and step, keep the smallest page set whose estimated attention mass
// reaches gamma). Two kernels:
//
// score_kernel   HBM-bound stream over the page summaries, which are kept in
//                logical page order per (request, KV head) segment. Every
//                warp of a persistent grid streams its own even slice of all
//                segments' pages with 4 KiB bulk copies into a private
//                3-slot ring. 16 lanes (32 when the group's queries would
//                not fit in registers) score one page. A lane holds channels
//                of either the min row or the max row, together with the
//                matching sign part of the group's queries, so
//                sum_i max(q_i*mn_i, q_i*mx_i) = sum_i q-_i*mn_i + q+_i*mx_i
//                is one fp32 FMA per element (paired with fma.rn.f32x2). A
//                transpose-reduce leaves each head's sum on a lane group; the
//                group max times 1/sqrt(d) is the page score. Scores stay
//                fp32: bf16 queries would move them by ~1e-3 and change lists.
//                (Gathering 512-byte per-(page, head) summaries scattered by
//                the block table runs at under half the copy bandwidth;
//                contiguous 4 KiB runs reach it.)
//
// select_kernel  One CTA per segment. Softmax weights exp(s - max) are turned
//                into fixed point (2^38 = weight of the top page), so every
//                sum is exact and order-independent. A radix select over
//                order-preserving score keys, with histograms of count and
//                mass over the candidates' actual key range, finds the cutoff
//                score in at most four rounds; ties at the cutoff go to the
//                lower page ids; one block scan compacts the kept ids in
//                ascending order. Each warp fills a private histogram of
//                32-bit words (a mass is three 13-bit limbs, so no word can
//                overflow), which keeps hot bins from serialising the CTA.
#include "asp_internal.cuh"

namespace asp {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ============================================================== score kernel
constexpr int kScoreWarps = 8;
constexpr int kScoreThreads = kScoreWarps * 32;

struct ScoreParams {
  const uint16_t* summ;
  const float* q;
  const int32_t* seq_lens;
  float* scores;
  uint32_t* err;
  int B, Hq, Hkv, P, max_pages;
  float inv_sqrt_d;
};

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// bf16x2 word -> (low element, high element) as an fp32 pair
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
  return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Sum of v[j] over the LPU lanes of a unit for each j < G, then the max over
// j. The halving steps leave each lane with head j(lane) (bits of the lane
// index); the final max is on every lane of the unit.
template <int G, int LPU>
__device__ __forceinline__ float group_bound_max(float (&v)[G], int lane) {
#pragma unroll
  for (int n = G, mask = LPU / 2; n > 1; n >>= 1, mask >>= 1) {
    const bool up = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? v[i] : v[i + n / 2];
      const float keep = up ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, mask);
    }
  }
  float s = v[0];
#pragma unroll
  for (int mask = LPU / 2 / G; mask >= 1; mask >>= 1) s += __shfl_xor_sync(kFull, s, mask);
#pragma unroll
  for (int mask = LPU / G; mask <= LPU / 2; mask <<= 1)
    s = fmaxf(s, __shfl_xor_sync(kFull, s, mask));
  return s;
}

// One lane's slice of a page's summary.
template <int Bytes>
struct Chunk {
  uint4 v[Bytes / 16];
};

// Summaries are stored per segment (request b, KV head h) in logical page
// order, so this pass is one sequential stream with no block-table lookups.
// The concatenated page space of all segments (segment-major) is split evenly
// over the warps of a persistent grid. Each warp walks its slice as pieces of
// up to kPieceBytes (whole pages of one segment); lane 0 bulk-copies every
// piece into the warp's own ring of kScoreSlots slots, one mbarrier per slot,
// so no warp ever waits on another. LPU lanes score one page (lanes
// [0, LPU/2) take the min row with q-, the rest the max row with q+), 32 / LPU
// pages per warp step.
constexpr int kPieceBytes = 4096;
constexpr int kScoreSlots = 3;

template <int D, int LPU>
struct ScoreCfg {
  static constexpr int kVals = 2 * D / LPU;  // channels per lane (one row)
  static constexpr int kBpl = kVals * 2;     // bytes per lane per page
  static constexpr int kPpi = 32 / LPU;      // pages per warp step
  static constexpr int kPageBytes = 4 * D;   // min and max rows of one page
  static constexpr int kPiecePages = kPieceBytes / kPageBytes;
};

// Position in a warp's slice: segment (b, h), logical page lp, and the index
// in the concatenated page space. Every lane of the warp holds the same one.
struct SegCursor {
  int b, h, lp, pos;
};

template <int D, int G, int LPU>
__global__ void __launch_bounds__(kScoreThreads, 2) score_kernel(ScoreParams p) {
  using C = ScoreCfg<D, LPU>;
  constexpr int kVals = C::kVals, kBpl = C::kBpl, kPpi = C::kPpi;
  constexpr int kPiecePages = C::kPiecePages, kPageBytes = C::kPageBytes;
  extern __shared__ __align__(128) uint8_t score_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kRingBytes = kScoreWarps * kScoreSlots * kPieceBytes;
  uint8_t* ring = score_smem + warp * kScoreSlots * kPieceBytes;  // this warp's slots
  uint64_t* full = reinterpret_cast<uint64_t*>(score_smem + kRingBytes) + warp * kScoreSlots;
  int* rprefix = reinterpret_cast<int*>(score_smem + kRingBytes +
                                        kScoreWarps * kScoreSlots * sizeof(uint64_t));  // [B + 1]

  if (lane == 0) {
    for (int i = 0; i < kScoreSlots; ++i) mbar_init(&full[i], 1);
    mbar_fence_init();
  }
  // prefix of the requests' page counts N_b (clamped sequence lengths)
  if (warp == 0) {
    int carry = 0;
    if (lane == 0) rprefix[0] = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < p.B) n = ceil_div(clamp_seq_len(p.seq_lens[b], p.max_pages, p.P, p.err), p.P);
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
  const long long units = (long long)p.Hkv * rprefix[p.B];
  const long long nw = (long long)gridDim.x * kScoreWarps;
  const long long gw = (long long)blockIdx.x * kScoreWarps + warp;
  const int wbeg = (int)(gw * units / nw), wend = (int)((gw + 1) * units / nw);
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
  int issued = 0;
  auto issue = [&]() {  // next piece of the slice into slot issued % kScoreSlots
    const int n = piece_pages(ic);
    if (lane == 0) {
      const int slot = issued % kScoreSlots;
      const size_t first = ((size_t)ic.b * p.Hkv + ic.h) * p.max_pages + ic.lp;
      mbar_arrive_expect_tx(&full[slot], n * kPageBytes);
      bulk_g2s(ring + slot * kPieceBytes,
               reinterpret_cast<const uint8_t*>(p.summ) + first * kPageBytes, n * kPageBytes,
               &full[slot]);
    }
    advance(ic, n);
    ++issued;
  };
  for (int k = 0; k < kScoreSlots && ic.pos < wend; ++k) issue();

  const int ul = lane % LPU, part = ul >= LPU / 2, ur = ul % (LPU / 2), pslot = lane / LPU;
  // chunk c of this lane = bytes [(c * LPU/2 + ur) * 16, +16) of its row
  const int lane_off = part * 2 * D + ur * 16;
  uint64_t qv[G][kVals / 2];
  auto load_q = [&](int b, int h) {
    const float* qp = p.q + ((size_t)b * p.Hq + h * G) * D + ur * 8;
#pragma unroll
    for (int jj = 0; jj < G; ++jj)
#pragma unroll
      for (int i = 0; i < kVals; i += 4) {  // chunk i/8 holds channels (i/8 * LPU/2 + ur) * 8 + [0, 8)
        const float4 x = *reinterpret_cast<const float4*>(
            qp + (size_t)jj * D + (i / 8) * (LPU / 2) * 8 + (i % 8));
        const float a0 = part ? fmaxf(x.x, 0.f) : fminf(x.x, 0.f);
        const float a1 = part ? fmaxf(x.y, 0.f) : fminf(x.y, 0.f);
        const float a2 = part ? fmaxf(x.z, 0.f) : fminf(x.z, 0.f);
        const float a3 = part ? fmaxf(x.w, 0.f) : fminf(x.w, 0.f);
        qv[jj][i / 2] = pack2(a0, a1);
        qv[jj][i / 2 + 1] = pack2(a2, a3);
      }
  };
  int qseg = -1, k = 0;
  bool aborted = false;
#pragma unroll 1
  for (; cc.pos < wend; ++k) {
    const int slot = k % kScoreSlots;
    if (!__all_sync(kFull, mbar_wait(&full[slot], (k / kScoreSlots) & 1))) {
      if (lane == 0) report(p.err, ASP_DEVERR_TIMEOUT);
      aborted = true;
      break;
    }
    const int n = piece_pages(cc), seg = cc.b * p.Hkv + cc.h;
    if (seg != qseg) {
      load_q(cc.b, cc.h);
      qseg = seg;
    }
    const uint8_t* sb = ring + slot * kPieceBytes + lane_off;
    float* out = p.scores + (size_t)seg * p.max_pages + cc.lp;
#pragma unroll 2
    for (int i0 = 0; i0 < n; i0 += kPpi) {
      const int pg = i0 + pslot;
      const int pr = min(pg, n - 1);  // lanes past the piece re-read its last page
      Chunk<kBpl> x;
#pragma unroll
      for (int c = 0; c < kBpl / 16; ++c)
        x.v[c] = *reinterpret_cast<const uint4*>(sb + pr * kPageBytes + c * (LPU / 2) * 16);
      const uint32_t* w = reinterpret_cast<const uint32_t*>(&x);
      uint64_t xv[kVals / 2];
#pragma unroll
      for (int m = 0; m < kVals / 2; ++m) xv[m] = bf16x2_to_f32x2(w[m]);
      float acc[G];
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        uint64_t a2 = 0;
#pragma unroll
        for (int m = 0; m < kVals / 2; ++m) a2 = ffma2(qv[jj][m], xv[m], a2);
        const float2 f = unpack2(a2);
        acc[jj] = f.x + f.y;
      }
      const float sc = group_bound_max<G, LPU>(acc, lane) * p.inv_sqrt_d;
      if (ul == 0 && pg < n) out[pg] = sc;
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
    for (int j = k; j < issued; ++j) mbar_wait(&full[j % kScoreSlots], (j / kScoreSlots) & 1);
}

// ============================================================= select kernel
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCache = 8192;  // scores cached in shared memory when N fits
constexpr int kBins = 256;
constexpr int kLimbBits = 13;    // mass = l0 + l1 << 13 + l2 << 26, each limb < 2^13
constexpr int kWarpCand = 4096;  // candidates one warp finishes on (fits the histogram area)
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

// Order-preserving key: a larger score gives a larger key; -0 maps like +0.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t f = __float_as_uint(s);
  if (f == 0x80000000u) f = 0u;
  return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// Softmax weight of a page relative to the top page, in 2^-38 units (<= 2^38).
__device__ __forceinline__ unsigned long long mass_fixed(float s, float smax) {
  return __float2ull_rn(expf(s - smax) * 274877906944.0f);
}

template <typename T>
__device__ __forceinline__ T block_reduce(T v, T* scratch, int op /*0 sum, 1 min, 2 max*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const T y = __shfl_xor_sync(kFull, v, o);
    v = op == 0 ? v + y : (op == 1 ? (y < v ? y : v) : (y > v ? y : v));
  }
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = scratch[lane];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const T y = __shfl_xor_sync(kFull, v, o);
      v = op == 0 ? v + y : (op == 1 ? (y < v ? y : v) : (y > v ? y : v));
    }
    if (lane == 0) scratch[0] = v;
  }
  __syncthreads();
  const T r = scratch[0];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectParams p) {
  extern __shared__ __align__(16) uint8_t sel_smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(sel_smem);  // [warp][bin][count, l0, l1, l2]
  float* cache = reinterpret_cast<float*>(hist + kSelWarps * kBins * 4);
  __shared__ uint32_t m_cnt[kBins];
  __shared__ unsigned long long m_mass[kBins];
  __shared__ unsigned long long red_u64[kSelWarps];
  __shared__ float red_f[kSelWarps];
  __shared__ uint32_t pick[4];
  __shared__ unsigned long long pick_m[1];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x;
  const int b = s / p.Hkv;
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
  const bool cached = N <= kSelCache;
  float lo_s = INFINITY, hi_s = -INFINITY;
  for (int i = tid; i < N; i += kSelThreads) {
    const float v = gsc[i];
    if (cached) cache[i] = v;
    lo_s = fminf(lo_s, v);
    hi_s = fmaxf(hi_s, v);
  }
  lo_s = block_reduce<float>(lo_s, red_f, 1);
  hi_s = block_reduce<float>(hi_s, red_f, 2);
  const float* sc = cached ? cache : gsc;
  const float smax = hi_s;

  unsigned long long target;
  if (mass_mode) {
    unsigned long long z = 0;
    for (int i = tid; i < N; i += kSelThreads) z += mass_fixed(sc[i], smax);
    z = block_reduce<unsigned long long>(z, red_u64, 0);
    target = (unsigned long long)ceil((double)p.gamma * (double)z);
    if (target < 1) target = 1;
  } else {
    target = (unsigned long long)p.budget;
  }

  // radix select of the cutoff key over the candidates' key range
  uint32_t lo = score_key(lo_s), hi = score_key(hi_s);
  unsigned long long above_m = 0;
  uint32_t above_c = 0, cnt_eq = 0;
  uint32_t* my_hist = hist + warp * kBins * 4;
  constexpr uint32_t kLimbMask = (1u << kLimbBits) - 1u;
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

  // Block-wide rounds over every element while the picked bin is large.
  bool resolved = false;
  while (true) {
    const int shift = shift_of();
    for (int i = tid; i < kSelWarps * kBins; i += kSelThreads)
      reinterpret_cast<uint4*>(hist)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    for (int i = tid; i < N; i += kSelThreads) {
      const float v = sc[i];
      const uint32_t k = score_key(v);
      if (k >= lo && k <= hi) {
        uint32_t* h = my_hist + ((k - lo) >> shift) * 4;
        atomicAdd(h, 1u);
        if (mass_mode) {
          const unsigned long long m = mass_fixed(v, smax);
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
    if (shift == 0) {
      resolved = true;
      break;
    }
    if (cnt_eq <= kWarpCand) break;  // few candidates left: one warp finishes
    __syncthreads();
  }
  if (!resolved) {
    // gather the candidates (scores with keys in [lo, hi]) and let warp 0
    // run the remaining rounds on them with warp-level synchronisation only
    float* cand = reinterpret_cast<float*>(hist + kBins * 4);  // after warp 0's histogram
    if (tid == 0) pick[3] = 0;
    __syncthreads();
    for (int i = tid; i < N; i += kSelThreads) {
      const float v = sc[i];
      const uint32_t k = score_key(v);
      if (k >= lo && k <= hi) cand[atomicAdd(&pick[3], 1u)] = v;
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
          const float v = cand[i];
          const uint32_t k = score_key(v);
          if (k >= lo && k <= hi) {
            uint32_t* h = hist + ((k - lo) >> shift) * 4;
            atomicAdd(h, 1u);
            if (mass_mode) {
              const unsigned long long m = mass_fixed(v, smax);
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
  const uint32_t tau = lo;
  // ties at the cutoff key: keep the first t (lowest ids)
  unsigned long long t;
  if (mass_mode) {
    const unsigned long long w = mass_fixed(key_score(tau), smax);
    t = w ? (target - above_m + w - 1) / w : cnt_eq;
  } else {
    t = target - above_c;
  }
  if (t < 1) t = 1;
  if (t > cnt_eq) t = cnt_eq;

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
  unsigned long long v = ((unsigned long long)gt << 32) | eq, x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red_u64[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = red_u64[lane], xx = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, xx, o);
      if (lane >= o) xx += y;
    }
    red_u64[lane] = xx - w;  // exclusive warp offsets
  }
  __syncthreads();
  const unsigned long long pre = red_u64[warp] + x - v;
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

template <int D, int G>
cudaError_t launch_score_t(const SelectArgs& a, cudaStream_t stream) {
  const asp_paged_kv& kv = *a.kv;
  ScoreParams p{kv.summaries, a.q, kv.seq_lens, a.scores, a.err, kv.batch, kv.num_q_heads,
                kv.num_kv_heads, kv.page_size, kv.max_pages, 1.0f / sqrtf((float)D)};
  // 16 lanes per page while the group's queries fit in 64 registers, else 32
  constexpr int kLpu = (G * 2 * D / 16 > 64) ? 32 : 16;
  const size_t smem = (size_t)kScoreWarps * kScoreSlots * (kPieceBytes + sizeof(uint64_t)) +
                      (kv.batch + 1) * sizeof(int);
  cudaError_t e = set_max_dynamic_smem((const void*)score_kernel<D, G, kLpu>, (int)smem);
  if (e != cudaSuccess) return e;
  // persistent: two CTAs per SM; the kernel splits the pages from seq_lens itself
  score_kernel<D, G, kLpu><<<2 * a.num_sms, kScoreThreads, smem, stream>>>(p);
  return cudaGetLastError();
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

cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream) {
  const asp_paged_kv& kv = *a.kv;
  const bool all = a.budget <= 0 && a.gamma >= 1.0f;
  if (!all) {  // gamma >= 1 keeps every page: no scores needed
    cudaError_t e = kv.head_dim == 128 ? launch_score_d<128>(a, stream)
                                       : launch_score_d<64>(a, stream);
    if (e != cudaSuccess) return e;
  }
  SelectParams p{a.scores, kv.seq_lens, a.lists, a.lens, a.err, kv.num_kv_heads, kv.page_size,
                 kv.max_pages, a.gamma, a.budget};
  cudaError_t e = set_max_dynamic_smem((const void*)select_kernel, (int)kSelSmem);
  if (e != cudaSuccess) return e;
  select_kernel<<<kv.batch * kv.num_kv_heads, kSelThreads, kSelSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace asp
