// select.cu - coverage selection (MOIRA abstract: per request, layer, KV
// head and step, keep the smallest page set whose estimated attention mass
// reaches gamma). Two kernels:
//
// score_kernel   HBM-bound stream over the page summaries. Persistent CTAs
//                split the concatenated (request, page) space evenly. One
//                producer warp stages each physical page's summaries (all KV
//                heads, contiguous) into a shared-memory ring with 1-D bulk
//                copies; eight consumer warps each own one (page slot, KV
//                head) of a stage. A lane holds 8 (d=128) or 4 (d=64)
//                channels of either the min row or the max row, together with
//                the matching sign part of the group's queries, so
//                sum_i max(q_i*mn_i, q_i*mx_i) = sum_i q-_i*mn_i + q+_i*mx_i
//                is one fp32 FMA per element (paired with fma.rn.f32x2). A
//                transpose-reduce leaves each head's sum on a lane group; the
//                group max times 1/sqrt(d) is the page score. Scores stay
//                fp32: bf16 queries would move them by ~1e-3 and change lists.
//
// select_kernel  One CTA per segment. Softmax weights exp(s - max) are turned
//                into 64-bit fixed point (2^40 = weight of the top page), so
//                every sum is exact and order-independent. A radix select over
//                order-preserving score keys, with histograms of count and
//                mass over the candidates' actual key range, finds the cutoff
//                score in at most four rounds; ties at the cutoff go to the
//                lower page ids; one block scan compacts the kept ids in
//                ascending order.
#include "asp_internal.cuh"

namespace asp {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ============================================================== score kernel
constexpr int kScoreConsumerWarps = 8;
constexpr int kScoreThreads = (kScoreConsumerWarps + 1) * 32;
constexpr int kScoreStages = 16;

struct ScoreParams {
  const uint16_t* summ;
  const float* q;
  const int32_t* bt;
  const int32_t* seq_lens;
  float* scores;
  uint32_t* err;
  int B, Hq, Hkv, P, max_pages, num_phys;
  float inv_sqrt_d;
};

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Sum of v[j] over the 32 lanes for each j < G, then the max over j. The
// halving steps leave lane l with head j(l); the final max is on all lanes.
template <int G>
__device__ __forceinline__ float group_bound_max(float (&v)[G], int lane) {
#pragma unroll
  for (int n = G, mask = 16; n > 1; n >>= 1, mask >>= 1) {
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
  for (int mask = 16 / G; mask >= 1; mask >>= 1) s += __shfl_xor_sync(kFull, s, mask);
#pragma unroll
  for (int mask = 32 / G; mask <= 16; mask <<= 1) s = fmaxf(s, __shfl_xor_sync(kFull, s, mask));
  return s;
}

// Segment of the concatenated page space holding position pos: the largest
// r with prefix[r] <= pos (prefix non-decreasing, prefix[0] = 0, pos < prefix[n]).
__device__ __forceinline__ int find_owner(const int* prefix, int n, int pos) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= pos) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int D, int G>
__global__ void __launch_bounds__(kScoreThreads, 2) score_kernel(ScoreParams p) {
  constexpr int kUnitBytes = 4 * D;            // min row + max row, bf16
  constexpr int kStageBytes = 8 * kUnitBytes;  // 8 (page, head) units
  constexpr int kCpl = D / 16;                 // channels per lane
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  int2* meta = reinterpret_cast<int2*>(ring + kScoreStages * kStageBytes);  // [stage][8 slots]
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + kScoreStages * 8);
  uint64_t* empty = full + kScoreStages;
  int* req_prefix = reinterpret_cast<int*>(empty + kScoreStages);  // [B + 1]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pps = 8 / p.Hkv;  // pages per stage
  if (tid == 0) {
    for (int i = 0; i < kScoreStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kScoreConsumerWarps);
    }
    mbar_fence_init();
  }
  // request prefix of page counts (clamped sequence lengths)
  if (warp == 0) {
    int carry = 0;
    if (lane == 0) req_prefix[0] = 0;
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
      if (b < p.B) req_prefix[b + 1] = carry + x;
      carry += __shfl_sync(kFull, x, 31);
    }
  }
  __syncthreads();
  const int total = req_prefix[p.B];
  const int beg = (int)((long long)blockIdx.x * total / gridDim.x);
  const int end = (int)((long long)(blockIdx.x + 1) * total / gridDim.x);
  const int nstages = ceil_div(end - beg, pps);

  if (warp == kScoreConsumerWarps) {
    // ------------------------------------------------------------ producer
    bool aborted = false;
    int issued = 0;
    for (int base = beg; base < end && !aborted; base += 32) {
      const int pos = base + lane;
      int b = -1, lp = -1, phys = -1;
      if (pos < end) {
        b = find_owner(req_prefix, p.B + 1, pos);
        lp = pos - req_prefix[b];
        phys = __ldg(p.bt + (size_t)b * p.max_pages + lp);
        if (phys < 0 || phys >= p.num_phys) {
          report(p.err, ASP_DEVERR_PAGE_RANGE);
          phys = -1;
        }
      }
      for (int j = 0; j < 32 && base + j < end; j += pps) {
        const int it = (base + j - beg) / pps;
        const int stage = it % kScoreStages;
        if (lane == 0 && !mbar_wait(&empty[stage], ((it / kScoreStages) & 1) ^ 1)) {
          report(p.err, ASP_DEVERR_TIMEOUT);
          aborted = true;
        }
        aborted = __shfl_sync(kFull, aborted ? 1 : 0, 0) != 0;
        if (aborted) break;
        uint32_t bytes = 0;
        for (int u = 0; u < pps; ++u) {
          const int src = j + u;
          const int ub = __shfl_sync(kFull, b, src & 31);
          const int ulp = __shfl_sync(kFull, lp, src & 31);
          const int uph = __shfl_sync(kFull, phys, src & 31);
          const bool in = (src < 32) && (base + src < end) && uph >= 0;
          if (lane == 0) meta[stage * 8 + u] = in ? make_int2(ub, ulp) : make_int2(-1, -1);
          if (in) bytes += p.Hkv * kUnitBytes;
        }
        if (lane == 0) {
          if (bytes) {
            mbar_arrive_expect_tx(&full[stage], bytes);
          } else {
            mbar_arrive(&full[stage]);
          }
        }
        for (int u = 0; u < pps; ++u) {
          const int src = j + u;
          const int uph = __shfl_sync(kFull, phys, src & 31);
          const bool in = (src < 32) && (base + src < end) && uph >= 0;
          if (lane == 0 && in)
            bulk_g2s(ring + stage * kStageBytes + u * p.Hkv * kUnitBytes,
                     p.summ + (size_t)uph * p.Hkv * 2 * D, p.Hkv * kUnitBytes, &full[stage]);
        }
        ++issued;
      }
    }
    // never leave the CTA with copies in flight
    if (lane == 0)
      for (int it = max(0, issued - kScoreStages); it < issued; ++it)
        mbar_wait(&full[it % kScoreStages], (it / kScoreStages) & 1);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int slot = warp / p.Hkv, head = warp % p.Hkv;
  const int part = lane >> 4;  // 0: min row, paired with q-; 1: max row, paired with q+
  const int c0 = (lane & 15) * kCpl;
  float qv[G][kCpl];
  int cur_b = -1;
  bool aborted = false;
  for (int it = 0; it < nstages; ++it) {
    const int stage = it % kScoreStages;
    if (!aborted && !mbar_wait(&full[stage], (it / kScoreStages) & 1)) {
      if (lane == 0) report(p.err, ASP_DEVERR_TIMEOUT);
      aborted = true;
    }
    const int2 mt = aborted ? make_int2(-1, -1) : meta[stage * 8 + slot];
    if (mt.x >= 0) {
      if (mt.x != cur_b) {
        cur_b = mt.x;
        const float* qb = p.q + ((size_t)cur_b * p.Hq + head * G) * D + c0;
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
          for (int i = 0; i < kCpl; i += 4) {
            const float4 x = *reinterpret_cast<const float4*>(qb + (size_t)j * D + i);
            qv[j][i + 0] = part ? fmaxf(x.x, 0.f) : fminf(x.x, 0.f);
            qv[j][i + 1] = part ? fmaxf(x.y, 0.f) : fminf(x.y, 0.f);
            qv[j][i + 2] = part ? fmaxf(x.z, 0.f) : fminf(x.z, 0.f);
            qv[j][i + 3] = part ? fmaxf(x.w, 0.f) : fminf(x.w, 0.f);
          }
      }
      const uint8_t* u = ring + stage * kStageBytes + (slot * p.Hkv + head) * kUnitBytes +
                         part * (2 * D) + c0 * 2;
      uint32_t w[kCpl / 2];
      if constexpr (kCpl == 8) {
        const uint4 x = *reinterpret_cast<const uint4*>(u);
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
      } else {
        const uint2 x = *reinterpret_cast<const uint2*>(u);
        w[0] = x.x; w[1] = x.y;
      }
      float acc[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < kCpl / 2; ++m)
          a2 = ffma2(make_float2(qv[j][2 * m], qv[j][2 * m + 1]), bf16x2_to_float2(w[m]), a2);
        acc[j] = a2.x + a2.y;
      }
      const float s = group_bound_max<G>(acc, lane) * p.inv_sqrt_d;
      if (lane == 0)
        p.scores[((size_t)mt.x * p.Hkv + head) * p.max_pages + mt.y] = s;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
}

// ============================================================= select kernel
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCache = 8192;  // scores cached in shared memory when N fits

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
// Softmax weight of a page relative to the top page, in 2^-40 units.
__device__ __forceinline__ unsigned long long mass_fixed(float s, float smax) {
  return __float2ull_rn(expf(s - smax) * 1099511627776.0f);
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
  __shared__ float cache[kSelCache];
  __shared__ uint32_t h_cnt[256];
  __shared__ unsigned long long h_mass[256];
  __shared__ unsigned long long red_u64[kSelWarps];
  __shared__ float red_f[kSelWarps];
  __shared__ uint32_t pick[4];             // bin, count above (low 32), spare
  __shared__ unsigned long long pick_m[1];  // mass above

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
  while (true) {
    const uint32_t range = hi - lo;
    const int bits = range ? 32 - __clz(range) : 0;
    const int shift = bits > 8 ? bits - 8 : 0;
    for (int i = tid; i < 256; i += kSelThreads) {
      h_cnt[i] = 0;
      h_mass[i] = 0;
    }
    __syncthreads();
    for (int i = tid; i < N; i += kSelThreads) {
      const float v = sc[i];
      const uint32_t k = score_key(v);
      if (k >= lo && k <= hi) {
        const uint32_t bin = (k - lo) >> shift;
        atomicAdd(&h_cnt[bin], 1u);
        if (mass_mode) atomicAdd(&h_mass[bin], mass_fixed(v, smax));
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane owns bins [8*lane, 8*lane+8); find the largest bin j with
      // above + (sum over bins >= j) >= target
      unsigned long long lm = 0;
      uint32_t lc = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        lm += h_mass[lane * 8 + i];
        lc += h_cnt[lane * 8 + i];
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
      const bool reach = mass_mode ? (above_m + sm >= target) : ((unsigned long long)above_c + scn >= target);
      const unsigned ballot = __ballot_sync(kFull, reach);
      const int lstar = 31 - __clz(ballot);  // ballot has lane 0 set by the invariant
      if (lane == lstar) {
        unsigned long long run_m = above_m + (sm - lm);
        uint32_t run_c = above_c + (scn - lc);
        int j = lane * 8;
        for (int i = 7; i >= 0; --i) {
          const int bin = lane * 8 + i;
          const unsigned long long nm = run_m + h_mass[bin];
          const uint32_t nc = run_c + h_cnt[bin];
          if (mass_mode ? (nm >= target) : ((unsigned long long)nc >= target)) {
            j = bin;
            break;
          }
          run_m = nm;
          run_c = nc;
        }
        pick[0] = (uint32_t)j;
        pick[1] = run_c;
        pick[2] = h_cnt[j];
        pick_m[0] = run_m;
      }
    }
    __syncthreads();
    const uint32_t j = pick[0];
    above_c = pick[1];
    cnt_eq = pick[2];
    above_m = pick_m[0];
    const unsigned long long nlo = (unsigned long long)lo + ((unsigned long long)j << shift);
    const unsigned long long nhi = nlo + ((1ull << shift) - 1ull);
    lo = (uint32_t)nlo;
    hi = nhi < hi ? (uint32_t)nhi : hi;
    __syncthreads();
    if (shift == 0) break;
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
  constexpr int kStageBytes = 8 * 4 * D;
  const size_t smem = (size_t)kScoreStages * kStageBytes + kScoreStages * 8 * sizeof(int2) +
                      2 * kScoreStages * sizeof(uint64_t) + (kv.batch + 1) * sizeof(int);
  cudaError_t e = set_max_dynamic_smem((const void*)score_kernel<D, G>, (int)smem);
  if (e != cudaSuccess) return e;
  ScoreParams p{kv.summaries, a.q, kv.block_table, kv.seq_lens, a.scores, a.err,
                kv.batch, kv.num_q_heads, kv.num_kv_heads, kv.page_size, kv.max_pages,
                kv.num_phys_pages, 1.0f / sqrtf((float)D)};
  score_kernel<D, G><<<a.num_sms * 2, kScoreThreads, smem, stream>>>(p);
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
  select_kernel<<<kv.batch * kv.num_kv_heads, kSelThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace asp
