// decode.cu - self-planning sparse attention over ragged page lists (MOIRA
// abstract: each thread block derives its own share of the work from the
// list lengths, so the decode step needs no host-side plan and stays inside
// the CUDA graph).
//
// Plan (every CTA, on the device): load lens[B*Hkv] into shared memory and
// take their inclusive prefix; the concatenated lists form one sequence of
// `total` pages. Each (segment, CTA) piece ends in a CTA-wide merge of the
// warps' states: the warps, which drift apart over a piece, all wait for the
// last one, so the CTA's copy pipeline idles for several microseconds. The
// first page of every non-empty list therefore weighs 1 + piece_cost pages
// (about 256 KiB of K and V) and the sequence is split evenly by weight over the G
// CTAs: a CTA whose range starts more lists takes fewer pages, and the split
// still depends on the list lengths alone. Each piece produces one partial
// (m, l, o) in slot segment + CTA of the workspace, which is unique because
// both indices grow along the sequence; a segment held whole by one CTA is
// written out directly. A split segment is merged by log-sum-exp by the last
// of its CTAs to finish: each counts its piece in with one atomic after its
// stream has ended (never at a piece end, where the round trip, 1.5-2 us
// under full HBM load, would stall the copy pipeline), and the CTA that
// completes the count folds the pieces in CTA order, so the result does not
// depend on timing. No CTA ever waits on another.
//
// Data path (per CTA: 8 warps, one CTA per SM): every warp runs its own
// pipeline. Warp w takes stages w, w+8, ... of the CTA's slice (a stage is a
// 16-token sub-tile of one page: K then V, [16 rows x 64 channels] 2-D TMA
// boxes with the 128-byte swizzle), keeps kSlots of them in flight in its own
// shared-memory slots, each with its own mbarrier, and refills a slot as soon
// as it has consumed it. Its lanes resolve list entry -> logical page ->
// physical row for the next 32 stages ahead of time. Independent issuers per
// SM are what reach the copy bandwidth on this gather; one issuing thread per
// CTA does not. Each warp keeps its own online-softmax state; the warps are
// merged in shared memory at the end of each piece.
//
// Per page the contraction is small (g <= 8 queries against P tokens), so it
// runs on mma.sync m16n8k16 bf16 with tokens as the M dimension and the query
// group (padded to 8) as N:
//   S^T[16 x 8] = K[16 x d] . Q^T[d x 8]      (Q split into bf16 hi + lo)
//   O^T[d x 8] += V^T[d x 16] . P^T[16 x 8]   (probabilities rounded to bf16)
// The S^T accumulator becomes the P^T operand through movmatrix.trans, and the
// swizzled tiles make every ldmatrix conflict-free. A page is 4-32 KiB of HBM
// against 4-8 flop per byte, far below any tensor-core limit: the kernel is
// bound by HBM, and the ring (128 KiB, or 192 KiB when the segment prefix
// leaves room in shared memory) keeps that much per SM in flight.
#include "asp_internal.cuh"

#include <cudaTypedefs.h>

#include <climits>

#include <mutex>

namespace asp {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;

// A stage is a 16-token sub-tile of a page (P/16 stages per page): 8 KiB (d=128)
// or 4 KiB (d=64). Each warp owns kSlots stages of the ring: 128 KiB per CTA,
// or 192 KiB (Deep) when the segment prefix leaves room in shared memory.
// While a warp computes on one stage the others stay in flight, so the extra
// slot is what keeps each SM's share of the copy bandwidth requested.
template <int D, int P, bool Deep>
struct Cfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kSubs = P / 16;                      // stages per page
  static constexpr int kTileBytes = 16 * 128;               // [16 rows x 64 bf16], swizzled
  static constexpr int kPartBytes = kHalves * kTileBytes;   // K (or V) of 16 tokens
  static constexpr int kStageBytes = 2 * kPartBytes;        // K then V
  static constexpr int kSlots = (D == 128 ? 2 : 4) * (Deep ? 3 : 2) / 2;  // stages per warp
  static constexpr int kRingBytes = kDecWarps * kSlots * kStageBytes;
  static constexpr int kMergeFloats = kDecWarps * (2 * 8 + 8 * D);
  static constexpr int kSlotFloats = 2 * 8 + 8 * D;
};

struct DecParams {
  const float* q;
  const int32_t* lists;
  const int32_t* lens;
  const int32_t* bt;
  const int32_t* seq_lens;
  float* out;
  float* lse;
  float* partials;
  int32_t* arrivals;  // [S]: pieces of each split segment done; zero between calls
  uint32_t* err;
  int B, Hq, Hkv, g, max_pages, num_phys, slot_floats;
  int piece_cost;  // extra weight of a list's first page in the split, in pages
  float scale_log2;
};

// ------------------------------------------------------------ mma helpers
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// Byte offset of (row r < 16, channel c, c % 8 == 0) inside a stage's K or V
// part, laid out as kHalves tiles of [16 rows x 128 B] with the 128-byte
// swizzle (16-byte chunk index XOR row % 8; tiles start on 1 KiB boundaries).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  const int hh = c >> 6, chunk = (c & 63) >> 3;
  return hh * (16 * 128) + r * 128 + ((chunk ^ (r & 7)) << 4);
}

__device__ __forceinline__ int seg_of(const int* prefix, int S, int pos) {
  int lo = 0, hi = S - 1;  // largest s with prefix[s] <= pos
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= pos) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Log-sum-exp merge of four output elements (query column col, channels
// o_off .. o_off + 3 with o_off = col * d + channel) over the np partials
// (m, l, o) of a segment, stored slot_floats apart from base: pieces are
// folded in CTA order with an online rescale in the log2 domain, eight
// pieces' loads in flight at once. The partials were written by other CTAs
// of this grid: loads go through L2.
__device__ __forceinline__ void fold_pieces4(const float* base, int np, int slot_floats, int col,
                                             int o_off, float& M, float& L, float4& acc) {
  M = -INFINITY;
  L = 0.f;
  acc = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int kU = 8;
  for (int c = 0; c < np; c += kU) {
    float m[kU], l[kU];
    float4 o[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      m[u] = -INFINITY;
      if (c + u < np) {
        const float* q = base + (size_t)(c + u) * slot_floats;
        m[u] = __ldcg(q + col);
        l[u] = __ldcg(q + 8 + col);
        o[u] = __ldcg(reinterpret_cast<const float4*>(q + 16 + o_off));
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (m[u] == -INFINITY) continue;  // a piece with no valid token (or none)
      if (m[u] > M) {
        const float sc = exp2f(M - m[u]);  // 0 while M is still -inf
        acc.x *= sc;
        acc.y *= sc;
        acc.z *= sc;
        acc.w *= sc;
        L *= sc;
        M = m[u];
      }
      const float w = exp2f(m[u] - M);
      acc.x += w * o[u].x;
      acc.y += w * o[u].y;
      acc.z += w * o[u].z;
      acc.w += w * o[u].w;
      L += w * l[u];
    }
  }
}

template <int D, int P, bool Deep>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecParams p) {
  using C = Cfg<D, P, Deep>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;                                                  // [warp][slot][stage]
  float* merge = reinterpret_cast<float*>(ring + C::kRingBytes);
  int4* meta = reinterpret_cast<int4*>(merge + C::kMergeFloats);         // [warp][slot]
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + kDecWarps * C::kSlots);
  int* flags = reinterpret_cast<int*>(full + kDecWarps * C::kSlots);    // [0..1] merge, [8..] scan
  int* prefix = flags + 48;                                              // [S + 1]

  // Split weight at the start of each segment, W(prefix[s]) = prefix[s] +
  // piece_cost * (non-empty segments before s); [S + 1] ints in the ring,
  // read only while planning, before the first copy lands there.
  int* wstart = reinterpret_cast<int*>(ring);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.B * p.Hkv;
  const int G = gridDim.x, cta = blockIdx.x;

  if (tid == 0) {
    for (int i = 0; i < kDecWarps * C::kSlots; ++i) mbar_init(&full[i], 1);
    mbar_fence_init();
    prefix[0] = 0;
    wstart[0] = 0;
  }
  pdl_launch_dependents();
  pdl_wait_predecessor();
  // ---- self-plan: lengths (validated) -> inclusive prefix of pages and of
  // non-empty segments in shared memory
  const int per = ceil_div(S, kDecThreads);
  const int a0 = min(S, tid * per), a1 = min(S, a0 + per);
  int run = 0, nzr = 0;
  // Range errors are collected and reported once after the loop: an atomic
  // on the error word between loads would keep the later loads in order.
  uint32_t bad = 0;
  const long long t_cap = (long long)p.max_pages * P;
  for (int s = a0; s < a1; ++s) {  // wstart[s + 1] first holds non-empty segments up to s
    int Tb = p.seq_lens[s / p.Hkv];
    int n = p.lens[s];
    if (Tb < 0 || (long long)Tb > t_cap) {
      bad |= ASP_DEVERR_SEQ_RANGE;
      Tb = Tb < 0 ? 0 : (int)t_cap;
    }
    const int n_b = ceil_div(Tb, P);
    if (n < 0 || n > n_b) {
      bad |= ASP_DEVERR_LEN_RANGE;
      n = n < 0 ? 0 : n_b;
    }
    run += n;
    nzr += n > 0 ? 1 : 0;
    prefix[s + 1] = run;
    wstart[s + 1] = nzr;
  }
  if (bad) report(p.err, bad);
  int x = run, y = nzr;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int xo = __shfl_up_sync(kFull, x, o), yo = __shfl_up_sync(kFull, y, o);
    if (lane >= o) {
      x += xo;
      y += yo;
    }
  }
  if (lane == 31) {
    flags[8 + warp] = x;
    flags[16 + warp] = y;
  }
  __syncthreads();
  int off = 0, offn = 0, total = 0;
  for (int w = 0; w < kDecWarps; ++w) {
    if (w < warp) {
      off += flags[8 + w];
      offn += flags[16 + w];
    }
    total += flags[8 + w];  // < 2^31, checked on the host
  }
  off += x - run;
  offn += y - nzr;
  // Every share of the weight must hold a page (X + 1 <= share size), so that
  // the CTAs holding pieces of one segment are consecutive, as the merge at
  // the end assumes (it folds the partial slots of CTAs cf..cl): X is capped
  // at total / G - 1.
  const int X = max(0, min(p.piece_cost, total / G - 1));
  for (int s = a0; s < a1; ++s) {
    prefix[s + 1] += off;
    wstart[s + 1] = prefix[s + 1] + X * (wstart[s + 1] + offn);
  }
  __syncthreads();

  // Weighted split: page j of segment s weighs 1, plus X when j = prefix[s];
  // W(j) = weight of the pages before j. CTA c takes the pages whose W lies
  // in the c-th even share of the total weight (< 2^31: the host checks
  // B * Hkv * (max_pages + 128)).
  const int wtotal = wstart[S];
  const int geff = wtotal < G ? wtotal : G;
  const EvenSplit split(wtotal, geff > 0 ? geff : 1);
  auto weight_at = [&](int s, int j) {  // W(j) for page j of segment s
    return j == prefix[s] ? wstart[s] : j + (wstart[s] - prefix[s]) + X;
  };
  auto page_at = [&](int cut) {  // first page j with W(j) >= cut
    if (cut >= wtotal) return total;
    int lo = 0, hi = S - 1;  // largest s with wstart[s] <= cut: a non-empty segment
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (wstart[mid] <= cut) lo = mid; else hi = mid - 1;
    }
    const int j0 = prefix[lo];
    if (cut <= wstart[lo]) return j0;
    return min(max(cut - (wstart[lo] - j0) - X, j0 + 1), prefix[lo + 1]);
  };
  long long beg = 0, end = 0;
  if (cta < geff) {
    beg = page_at(split.begin(cta));
    end = page_at(split.end(cta));
  }
  const float kLn2 = 0.69314718055994530942f;

  // segments with an empty list: out = 0, lse = -inf
  for (int s = cta; s < S; s += G) {
    if (prefix[s + 1] != prefix[s]) continue;
    const int b = s / p.Hkv, h = s % p.Hkv;
    for (int e = tid; e < p.g * D; e += kDecThreads)
      p.out[((size_t)b * p.Hq + h * p.g + e / D) * D + e % D] = 0.f;
    for (int e = tid; e < p.g; e += kDecThreads) p.lse[(size_t)b * p.Hq + h * p.g + e] = -INFINITY;
  }
  // Only a CTA's first and last pieces can hold part of a segment (a middle
  // piece holds a whole one). For each, the CTAs cf..cf+np-1 holding that
  // segment: the last of them to finish merges it.
  int seg_a = -1, seg_b = -1, cf_a = 0, cf_b = 0, np_a = 0, np_b = 0;
  if (beg < end) {
    auto holders = [&](int s, int& cf) {
      cf = split.part_of(wstart[s]);
      return split.part_of(weight_at(s, prefix[s + 1] - 1)) - cf + 1;
    };
    seg_a = seg_of(prefix, S, (int)beg);
    seg_b = seg_of(prefix, S, (int)(end - 1));
    np_a = holders(seg_a, cf_a);
    if (seg_b != seg_a) np_b = holders(seg_b, cf_b);
  }
  __syncthreads();  // the weights are done with: the ring is free for copies
  if (beg >= end) return;
  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }

  // ---- this warp's stages: CTA stage it = warp + 8n covers page position
  // beg + it / kSubs, sub-tile it % kSubs (= warp % kSubs, since kSubs | 8)
  const long long nst = (end - beg) * C::kSubs;
  const int n_total = nst > warp ? (int)((nst - warp + kDecWarps - 1) / kDecWarps) : 0;
  const int sub = warp % C::kSubs;
  uint8_t* my_ring = ring + warp * C::kSlots * C::kStageBytes;
  uint64_t* my_full = full + warp * C::kSlots;
  int4* my_meta = meta + warp * C::kSlots;

  // Lookups for warp stages [nb, nb + 32): lane j owns stage nb + j. The
  // list entry (and sequence length) are fetched two batches ahead and the
  // block-table entry one batch ahead of the stages being issued.
  constexpr int kNoPage = INT_MIN;
  auto lookup_list = [&](int nb, int& seg, int& T, int& lp) {
    seg = 0; T = 0; lp = -1;
    const int n = nb + lane;
    if (n < n_total) {
      const long long pos = beg + (warp + (long long)kDecWarps * n) / C::kSubs;
      seg = seg_of(prefix, S, (int)pos);
      T = __ldg(p.seq_lens + seg / p.Hkv);
      lp = __ldg(p.lists + (size_t)seg * p.max_pages + (int)(pos - prefix[seg]));
    }
  };
  auto lookup_page = [&](int nb, int seg, int T, int lp) {
    int phys = kNoPage;
    if (nb + lane < n_total) {
      T = min(max(T, 0), p.max_pages * P);
      if (lp < 0 || lp >= ceil_div(T, P)) {
        if (sub == 0) report(p.err, ASP_DEVERR_LIST_RANGE);
      } else {
        phys = __ldg(p.bt + (size_t)(seg / p.Hkv) * p.max_pages + lp);
      }
    }
    return phys;
  };
  // (row of the sub-tile in the [rows, d] view, valid tokens in it) or ntok 0
  auto finalize = [&](int seg, int T, int lp, int phys, int& row, int& ntok) {
    row = 0; ntok = 0;
    if (phys == kNoPage) return;
    if (phys < 0 || phys >= p.num_phys) {
      if (sub == 0) report(p.err, ASP_DEVERR_PAGE_RANGE);
      return;
    }
    T = min(max(T, 0), p.max_pages * P);
    row = (phys * p.Hkv + seg % p.Hkv) * P + 16 * sub;
    ntok = min(16, max(0, min(P, T - lp * P) - 16 * sub));
  };

  int sB, TB, lpB, sC, TC, lpC, rowA, ntokA, phB;
  {
    int sA, TA, lpA;
    lookup_list(0, sA, TA, lpA);
    lookup_list(32, sB, TB, lpB);
    const int phA = lookup_page(0, sA, TA, lpA);
    finalize(sA, TA, lpA, phA, rowA, ntokA);
    phB = lookup_page(32, sB, TB, lpB);
    lookup_list(64, sC, TC, lpC);
  }
  const uint64_t pol = l2_evict_first_policy();  // K/V pages are read once
  int ib = 0;   // first warp stage of batch A
  int ni = 0;   // next warp stage to issue
  bool aborted = false;
  auto issue_next = [&]() {
    if (ni >= ib + 32) {  // rotate the lookup batches (warp-uniform)
      finalize(sB, TB, lpB, phB, rowA, ntokA);
      ib += 32;
      const int phC = lookup_page(ib + 32, sC, TC, lpC);
      sB = sC; TB = TC; lpB = lpC; phB = phC;
      lookup_list(ib + 64, sC, TC, lpC);
    }
    const int r_row = __shfl_sync(kFull, rowA, ni - ib);
    const int r_ntok = __shfl_sync(kFull, ntokA, ni - ib);
    if (lane == 0) {
      const int slot = ni % C::kSlots;
      my_meta[slot] = make_int4(r_ntok, 0, 0, 0);
      if (r_ntok > 0) {
        uint8_t* dst = my_ring + slot * C::kStageBytes;
        mbar_arrive_expect_tx(&my_full[slot], C::kStageBytes);
#pragma unroll
        for (int hh = 0; hh < C::kHalves; ++hh) {
          tma_load_2d_hint(dst + hh * C::kTileBytes, &tmK, hh * 64, r_row, &my_full[slot], pol);
          tma_load_2d_hint(dst + C::kPartBytes + hh * C::kTileBytes, &tmV, hh * 64, r_row,
                           &my_full[slot], pol);
        }
      } else {
        mbar_arrive(&my_full[slot]);
      }
    }
    ++ni;
  };
  while (ni < min(C::kSlots, n_total)) issue_next();

  // ================================================================ pieces
  const int gid = lane >> 2, tq = lane & 3;
  int nc = 0;      // next warp stage to consume
  int waited = 0;  // stages whose copies are known complete
  // Q^T fragments (B operand): rows d = kk*16 + 2*tq (+1, +8, +9), column gid
  uint32_t qhi[D / 16][2], qlo[D / 16][2];
  auto load_q = [&](int seg) {
    const int qb = seg / p.Hkv, qh = seg % p.Hkv;
    const bool live = gid < p.g;
    const float* qr = p.q + ((size_t)qb * p.Hq + qh * p.g + (live ? gid : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float2 v = make_float2(0.f, 0.f);
        if (live) v = *reinterpret_cast<const float2*>(qr + kk * 16 + half * 8 + 2 * tq);
        v.x *= p.scale_log2;
        v.y *= p.scale_log2;
        const __nv_bfloat162 hv = __floats2bfloat162_rn(v.x, v.y);
        const float2 hf = __bfloat1622float2(hv);
        qhi[kk][half] = *reinterpret_cast<const uint32_t*>(&hv);
        qlo[kk][half] = pack_bf16(v.x - hf.x, v.y - hf.y);
      }
  };
  long long pos = beg;
  load_q(seg_of(prefix, S, (int)pos));
  while (pos < end) {
    const int s = seg_of(prefix, S, (int)pos);
    const long long seg_lo = prefix[s], seg_hi = prefix[s + 1];
    const long long pe = seg_hi < end ? seg_hi : end;
    const int b = s / p.Hkv, h = s % p.Hkv;

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[D / 16][4];
#pragma unroll
    for (int dt = 0; dt < D / 16; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;

    const long long it_end = (pe - beg) * C::kSubs;
    while (nc < n_total && warp + (long long)kDecWarps * nc < it_end) {
      const int slot = nc % C::kSlots;
      if (!aborted) {
        // warp-uniform outcome: the refill below shuffles across all lanes
        const bool got = mbar_wait(&my_full[slot], (nc / C::kSlots) & 1);
        if (__all_sync(kFull, got)) {
          waited = nc + 1;
        } else {
          if (lane == 0) report(p.err, ASP_DEVERR_TIMEOUT);
          aborted = true;
        }
      }
      const int ntok = my_meta[slot].x;
      if (!aborted && ntok > 0) {
        const uint32_t kb = smem_u32(my_ring + slot * C::kStageBytes);
        const uint32_t vb = kb + C::kPartBytes;
        const int j = lane >> 3;
        // ---- S^T[16 x 8] = K[16 x d] . Q^T[d x 8]
        float sv[4];
        {
          // four independent accumulator chains (hi/lo x even/odd k-step)
          float acc[4][4] = {};
          const int r = (j & 1) * 8 + (lane & 7);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4];
            ldsm_x4(kb + swz(r, kk * 16 + (j >> 1) * 8), a);
            mma16816(acc[(kk & 1) * 2], a, qhi[kk][0], qhi[kk][1]);
            mma16816(acc[(kk & 1) * 2 + 1], a, qlo[kk][0], qlo[kk][1]);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) sv[i] = (acc[0][i] + acc[2][i]) + (acc[1][i] + acc[3][i]);
        }
        // ---- mask tokens past the sequence, online softmax (log2 domain)
        if (gid >= ntok) sv[0] = sv[1] = -INFINITY;
        if (gid + 8 >= ntok) sv[2] = sv[3] = -INFINITY;
        float cm0 = fmaxf(sv[0], sv[2]), cm1 = fmaxf(sv[1], sv[3]);
#pragma unroll
        for (int off2 = 4; off2 < 32; off2 <<= 1) {
          cm0 = fmaxf(cm0, __shfl_xor_sync(kFull, cm0, off2));
          cm1 = fmaxf(cm1, __shfl_xor_sync(kFull, cm1, off2));
        }
        const float n0 = fmaxf(m0, cm0), n1 = fmaxf(m1, cm1);
        const float al0 = exp2f(m0 - n0), al1 = exp2f(m1 - n1);
        m0 = n0;
        m1 = n1;
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) {
          o[dt][0] *= al0;
          o[dt][1] *= al1;
          o[dt][2] *= al0;
          o[dt][3] *= al1;
        }
        const float p0 = exp2f(sv[0] - n0), p1 = exp2f(sv[1] - n1);
        const float p2 = exp2f(sv[2] - n0), p3 = exp2f(sv[3] - n1);
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
        const uint32_t pb0 = movm_t(pack_bf16(p0, p1));
        const uint32_t pb1 = movm_t(pack_bf16(p2, p3));
        // ---- rows past the sequence may hold anything: zero them in V
        if (ntok < 16) {
          uint8_t* vpart = my_ring + slot * C::kStageBytes + C::kPartBytes;
          const int chunks = (16 - ntok) * C::kHalves * 8;
          for (int e = lane; e < chunks; e += 32) {
            const int r = ntok + e / (C::kHalves * 8);
            const int hh = (e / 8) % C::kHalves;
            *reinterpret_cast<uint4*>(vpart + hh * C::kTileBytes + r * 128 + (e % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        // ---- O^T[d x 8] += V^T[d x 16] . P^T[16 x 8]
        {
          const int r = (j >> 1) * 8 + (lane & 7);
#pragma unroll
          for (int dt = 0; dt < D / 16; ++dt) {
            uint32_t a[4];
            ldsm_x4_t(vb + swz(r, dt * 16 + (j & 1) * 8), a);
            mma16816(o[dt], a, pb0, pb1);
          }
        }
      }
      // the slot's reads (and any zeroing writes) are done: refill it
      __syncwarp();
      if (!aborted && ni < n_total) {
        fence_proxy_async_smem();
        issue_next();
      }
      ++nc;
    }

    // ---- merge the 8 warps' states of this piece
#pragma unroll
    for (int off2 = 4; off2 < 32; off2 <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, off2);
      l1 += __shfl_xor_sync(kFull, l1, off2);
    }
    float* mw = merge + warp * C::kSlotFloats;  // m[8], l[8], o[8][D]
    if (gid == 0) {
      mw[2 * tq] = m0;
      mw[2 * tq + 1] = m1;
      mw[8 + 2 * tq] = l0;
      mw[8 + 2 * tq + 1] = l1;
    }
#pragma unroll
    for (int dt = 0; dt < D / 16; ++dt) {
      const int d0 = dt * 16 + gid;
      mw[16 + (2 * tq) * D + d0] = o[dt][0];
      mw[16 + (2 * tq + 1) * D + d0] = o[dt][1];
      mw[16 + (2 * tq) * D + d0 + 8] = o[dt][2];
      mw[16 + (2 * tq + 1) * D + d0 + 8] = o[dt][3];
    }
    if (pe < end) load_q(seg_of(prefix, S, (int)pe));  // next piece's queries overlap the merge
    __syncthreads();
    const bool whole = (pos == seg_lo) && (pe == seg_hi);
    float* pslot = p.partials + (size_t)(s + cta) * p.slot_floats;
    for (int e = tid; e < p.g * D; e += kDecThreads) {
      const int col = e / D, d = e % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, merge[w * C::kSlotFloats + col]);
      float L = 0.f, acc = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
          const float* q = merge + w * C::kSlotFloats;
          const float sc = exp2f(q[col] - M);
          L += sc * q[8 + col];
          acc += sc * q[16 + col * D + d];
        }
      }
      if (whole) {
        const size_t row = (size_t)b * p.Hq + h * p.g + col;
        p.out[row * D + d] = L > 0.f ? acc / L : 0.f;
        if (d == 0) p.lse[row] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
      } else {
        pslot[16 + col * D + d] = acc;
        if (d == 0) {
          pslot[col] = M;
          pslot[8 + col] = L;
        }
      }
    }
    __syncthreads();  // the merge area is rewritten by the next piece
    pos = pe;
  }
  // never leave the CTA with copies in flight (only after a timeout can any remain)
  if (lane == 0)
    for (int n = waited; n < ni; ++n) mbar_wait(&my_full[n % C::kSlots], (n / C::kSlots) & 1);

  // ---- split segments: count this CTA's pieces in; the CTA that brings a
  // segment's count to its number of pieces merges that segment's partials
  // (in CTA order, so the result does not depend on which CTA it is) and
  // resets the count for the next call.
  if (np_a < 2 && np_b < 2) return;  // CTA-uniform
  __syncthreads();  // every partial store of this CTA has been issued
  if (tid == 0) {
    __threadfence();  // ... and is ordered before the arrivals (cumulative over the CTA)
    const int oa = np_a > 1 ? atomicAdd(&p.arrivals[seg_a], 1) : -1;
    const int ob = np_b > 1 ? atomicAdd(&p.arrivals[seg_b], 1) : -1;
    flags[0] = np_a > 1 && oa == np_a - 1 ? 1 : 0;
    flags[1] = np_b > 1 && ob == np_b - 1 ? 1 : 0;
    __threadfence();  // the other CTAs' partials, seen through the arrivals, before the loads
  }
  __syncthreads();
#pragma unroll 1
  for (int k = 0; k < 2; ++k) {
    if (!flags[k]) continue;  // CTA-uniform
    const int ms = k ? seg_b : seg_a, cf = k ? cf_b : cf_a, np = k ? np_b : np_a;
    const float* base = p.partials + (size_t)(ms + cf) * p.slot_floats;
    const int mb = ms / p.Hkv, mh = ms % p.Hkv;
    for (int e = 4 * tid; e < p.g * D; e += 4 * kDecThreads) {  // one pass when g * d <= 1024
      const int col = e / D, d = e % D;
      float M, L;
      float4 acc;
      fold_pieces4(base, np, p.slot_floats, col, e, M, L, acc);
      const size_t row = (size_t)mb * p.Hq + mh * p.g + col;
      float* o = p.out + row * D + d;  // the caller's buffer: 4-byte alignment only
      o[0] = L > 0.f ? acc.x / L : 0.f;
      o[1] = L > 0.f ? acc.y / L : 0.f;
      o[2] = L > 0.f ? acc.z / L : 0.f;
      o[3] = L > 0.f ? acc.w / L : 0.f;
      if (d == 0) p.lse[row] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    if (tid == 0) p.arrivals[ms] = 0;
  }
}

// ----------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

cudaError_t encode_bf16_2d_swizzled(CUtensorMap* map, const void* base, unsigned long long inner,
                                    unsigned long long rows, unsigned box_inner, unsigned box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

// [rows = num_phys*Hkv*P, D] bf16 viewed as 2-D; box = [16 rows x 64 channels].
cudaError_t make_page_map(CUtensorMap* map, const void* base, long long rows, int D, int P) {
  return encode_bf16_2d_swizzled(map, base, (unsigned long long)D, (unsigned long long)rows, 64,
                                 16);
}

// Dynamic shared memory of decode_kernel: 1 KiB alignment slack, the ring,
// the warp-merge area, per-slot metadata and mbarriers, flags, prefix[S + 1].
template <int D, int P, bool Deep>
size_t decode_smem_bytes(int S) {
  using C = Cfg<D, P, Deep>;
  return 1024 + (size_t)C::kRingBytes + C::kMergeFloats * 4 +
         kDecWarps * C::kSlots * (sizeof(int4) + 8) + 48 * 4 + (size_t)(S + 1) * 4;
}

int max_optin_smem() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return 0;
  return v;
}

template <int D, int P, bool Deep>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t stream) {
  using C = Cfg<D, P, Deep>;
  const asp_paged_kv& kv = *a.kv;
  const int S = kv.batch * kv.num_kv_heads;
  const size_t smem = decode_smem_bytes<D, P, Deep>(S);
  cudaError_t e = set_max_dynamic_smem((const void*)decode_kernel<D, P, Deep>, (int)smem);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)kv.num_phys_pages * kv.num_kv_heads * P;
  CUtensorMap tk, tv;
  if ((e = make_page_map(&tk, kv.k_cache, rows, D, P)) != cudaSuccess) return e;
  if ((e = make_page_map(&tv, kv.v_cache, rows, D, P)) != cudaSuccess) return e;
  DecParams p{a.q, a.lists, a.lens, kv.block_table, kv.seq_lens, a.out, a.lse, a.partials,
              a.arrivals, a.err, kv.batch, kv.num_q_heads, kv.num_kv_heads,
              kv.num_q_heads / kv.num_kv_heads, kv.max_pages, kv.num_phys_pages, a.slot_floats,
              decode_piece_cost(D, P), a.sm_scale * 1.4426950408889634f};
  return launch_pdl(decode_kernel<D, P, Deep>, dim3(a.grid), dim3(kDecThreads), smem, stream, tk, tv,
                    p);
}

// The deeper ring when its shared memory (which grows with the segment
// count through the prefix of list lengths) fits the device's per-block limit.
template <int D, int P>
cudaError_t launch_decode_dp(const DecodeArgs& a, cudaStream_t stream) {
  const int S = a.kv->batch * a.kv->num_kv_heads;
  if (decode_smem_bytes<D, P, true>(S) <= (size_t)max_optin_smem())
    return launch_decode_t<D, P, true>(a, stream);
  return launch_decode_t<D, P, false>(a, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const int d = a.kv->head_dim, P = a.kv->page_size;
  if (d == 128 && P == 16) return launch_decode_dp<128, 16>(a, stream);
  if (d == 128 && P == 32) return launch_decode_dp<128, 32>(a, stream);
  if (d == 128 && P == 64) return launch_decode_dp<128, 64>(a, stream);
  if (d == 64 && P == 16) return launch_decode_dp<64, 16>(a, stream);
  if (d == 64 && P == 32) return launch_decode_dp<64, 32>(a, stream);
  if (d == 64 && P == 64) return launch_decode_dp<64, 64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace asp
