// score_common.cuh - the page-score arithmetic and the fixed-point masses of
// the coverage selection (MOIRA abstract: the smallest page set whose
// estimated attention mass reaches gamma; the estimate is the Quest bound
// named in the HiSparse abstract), shared by the two selection paths of
// libasp.so: the score pass + per-segment select kernels (select.cu) and the
// cluster kernel that scores and selects a segment in one pass
// (select_cluster.cu). Both compute every score with the same instructions,
// so they rank pages identically.
#pragma once

#include "asp_internal.cuh"

namespace asp {
namespace score {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kPieceBytes = 4096;  // summaries one warp copies per ring slot

// Three bf16 terms whose sum is x to fp32 precision: s0 = rn(x),
// s1 = rn(x - s0), s2 = rn(x - s0 - s1). Each residual is exact in fp32, and
// bf16 x bf16 products are exact in fp32, so the tensor-core dot products
// carry the full fp32 query.
__device__ __forceinline__ void split3_bf16(float x, float (&s)[3]) {
  s[0] = __bfloat162float(__float2bfloat16_rn(x));
  const float r1 = x - s[0];
  s[1] = __bfloat162float(__float2bfloat16_rn(r1));
  s[2] = __bfloat162float(__float2bfloat16_rn(r1 - s[1]));
}

// Page geometry of the summary stream and the shape of the score mma.
// Summaries of one page (min row, then max row: 4d bytes) sit in shared
// memory at a stride of 4d + 16 bytes, which keeps the ldmatrix rows of 8
// consecutive pages on distinct banks.
template <int D, int G>
struct Cfg {
  static constexpr int kPageBytes = 4 * D;                      // min and max rows
  static constexpr int kPiecePages = kPieceBytes / kPageBytes;  // 8 (d 128) or 16 (d 64)
  static constexpr int kStride = kPageBytes + 16;               // padded page stride in smem
  static constexpr int kSlotBytes = kPiecePages * kStride;
  static constexpr int kKs = 2 * D / 16;                        // k-steps of one page
  static constexpr int kBlocks = (3 * G + 7) / 8;               // 8-row A blocks holding data
  static constexpr int kMt = (kBlocks + 1) / 2;                 // m16 tiles
};

// The group's queries as the A operand of the score mma, and the score of 8
// pages per call. The bound sum_i max(q_i mn_i, q_i mx_i) = sum_i q-_i mn_i +
// q+_i mx_i is one row.col mma chain: A = the group's queries, one row per
// (split term, head), K = 2d with q- against the min row and q+ against the
// max row; B = the 8 pages' summaries (N = pages). Rows past 3 G are zero.
// Row r's head is r % G, and since G divides 8 a lane's rows all share head
// (lane / 4) % G: the lane sums its rows, a butterfly over the lanes of the
// other split terms completes each head's sum, and one over the heads takes
// the max.
template <int D, int G>
struct GroupQuery {
  using C = Cfg<D, G>;
  // block bi holds rows 8 bi + lane / 4; qa[bi][ks] = the two registers of
  // that row at k-step ks (k = 16 ks + 2 (lane % 4) + {0, 1} and the same + 8)
  uint32_t qa[C::kBlocks][C::kKs][2];

  // qp: the group's first query row, fp32 [G, D]
  __device__ __forceinline__ void load(const float* qp_group, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const float* qp = qp_group + (g % G) * D;
#pragma unroll
    for (int ks = 0; ks < C::kKs; ++ks)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int k = 16 * ks + 2 * t + 8 * e;  // k < D: q- with the min row, else q+ with max
        const float2 x = *reinterpret_cast<const float2*>(qp + (k < D ? k : k - D));
        float s0[3], s1[3];
        split3_bf16(k < D ? fminf(x.x, 0.f) : fmaxf(x.x, 0.f), s0);
        split3_bf16(k < D ? fminf(x.y, 0.f) : fmaxf(x.y, 0.f), s1);
#pragma unroll
        for (int bi = 0; bi < C::kBlocks; ++bi) {
          const int r = 8 * bi + g, sp = r / G;  // split term of row r (>= 3: zero row)
          const float lo = sp == 0 ? s0[0] : sp == 1 ? s0[1] : sp == 2 ? s0[2] : 0.f;
          const float hi = sp == 0 ? s1[0] : sp == 1 ? s1[1] : sp == 2 ? s1[2] : 0.f;
          qa[bi][ks][e] = pack_bf16(lo, hi);
        }
      }
  }

  // Byte offset, within a tile of 8 pages, of this lane's ldmatrix row.
  __device__ __forceinline__ static uint32_t lane_row(int lane) {
    return (uint32_t)((lane & 7) * C::kStride + (lane >> 3) * 16);
  }

  // Unscaled group bounds of 8 pages: lanes 0-3 receive pages 2 (lane % 4)
  // and 2 (lane % 4) + 1 in x0 and x1 (every lane takes part). addr(ks), for
  // even k-steps ks, is the shared address of this lane's ldmatrix row of
  // k-steps ks and ks + 1: page (lane % 8) of the tile, elements
  // 16 ks + 8 (lane / 8) .. + 8.
  template <class Addr>
  __device__ __forceinline__ void tile_at(Addr addr, float& x0, float& x1) const {
    float acc[C::kMt][2][4];  // [m tile][min half, max half][fragment]
#pragma unroll
    for (int mt = 0; mt < C::kMt; ++mt)
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[mt][c][j] = 0.f;
#pragma unroll
    for (int ks = 0; ks < C::kKs; ks += 2) {
      uint32_t bf[4];  // (b0, b1) of k-step ks, then of ks + 1
      ldsm_x4(addr(ks), bf);
      constexpr int kHalfKs = C::kKs / 2;
#pragma unroll
      for (int mt = 0; mt < C::kMt; ++mt) {
        const bool up = 2 * mt + 1 < C::kBlocks;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t a[4] = {qa[2 * mt][ks + u][0], up ? qa[2 * mt + up][ks + u][0] : 0u,
                                 qa[2 * mt][ks + u][1], up ? qa[2 * mt + up][ks + u][1] : 0u};
          mma16816(acc[mt][ks >= kHalfKs], a, bf[2 * u], bf[2 * u + 1]);
        }
      }
    }
    // this lane's rows share head (lane / 4) % G: columns 2t and 2t + 1
    x0 = 0.f;
    x1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < C::kMt; ++mt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        x0 += acc[mt][c][0] + acc[mt][c][2];
        x1 += acc[mt][c][1] + acc[mt][c][3];
      }
#pragma unroll
    for (int m = 4 * G; m <= 16; m <<= 1) {  // the other split terms of the head
      x0 += __shfl_xor_sync(kFull, x0, m);
      x1 += __shfl_xor_sync(kFull, x1, m);
    }
#pragma unroll
    for (int m = 4; m < 4 * G; m <<= 1) {  // max over the group's heads
      x0 = fmaxf(x0, __shfl_xor_sync(kFull, x0, m));
      x1 = fmaxf(x1, __shfl_xor_sync(kFull, x1, m));
    }
  }

  // Pages at a stride of kStride bytes, the tile's first page at `tile`
  // (+ lane_row(lane)).
  __device__ __forceinline__ void tile(uint32_t tile, float& x0, float& x1) const {
    tile_at([&](int ks) { return tile + (uint32_t)(ks * 32); }, x0, x1);
  }

  // Pages held as 2d / 64 tensor-copy sub-tiles of [rows pages x 128 B] with
  // the 128-byte swizzle: sub-tile t holds elements [64 t, 64 t + 64) of
  // every page, and 16-byte chunk c of page row r sits at chunk c ^ (r % 8).
  // The tile is pages [8 nt, 8 nt + 8) of the slot at `slot` (1 KiB aligned).
  __device__ __forceinline__ void tile_swz(uint32_t slot, int nt, int rows, int lane, float& x0,
                                           float& x1) const {
    const int r = lane & 7, j = lane >> 3;
    const uint32_t row = slot + (uint32_t)((nt * 8 + r) * 128);
    tile_at([&](int ks) {
      return row + (uint32_t)((ks >> 2) * rows * 128) + (uint32_t)(((((ks & 3) << 1) + j) ^ r) << 4);
    }, x0, x1);
  }
};

// ------------------------------------------------------- selection helpers
// Order-preserving key: a larger score gives a larger key; -0 maps like +0.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t f = __float_as_uint(s);
  if (f == 0x80000000u) f = 0u;
  return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Softmax weight of a page relative to the top page, in units of 1/unit of
// the top page's weight. Segments of up to 8192 pages use unit = 2^37: 8192
// weights sum below 2^50 (19-bit limbs of them below 2^32). Longer segments
// use 2^42, so that rounding 2^20 weights moves their total by at most 2^-23
// of the top page; their sums (below 2^62) are 64-bit, and radix rounds take
// them as three 14-bit limbs.
// Rounded to the nearest integer (ties to even) by IEEE bit arithmetic on
// the integer pipes, which have several times the throughput of the
// conversion unit: below 2^22, adding 2^23 leaves the rounded integer in the
// mantissa bits; from 2^23 on the float is an integer, its mantissa shifted
// by the exponent; the band between takes one conversion instruction.
constexpr float kUnitFast = 137438953472.0f;   // 2^37
constexpr float kUnitLong = 4398046511104.0f;  // 2^42
__device__ __forceinline__ unsigned long long mass_fixed(float s, float smax, float unit) {
  const float f = exp2f((s - smax) * 1.4426950408889634f) * unit;
  if (f < 4194304.0f) return __float_as_uint(f + 8388608.0f) & 0x7fffffu;
  if (f >= 8388608.0f) {
    const uint32_t u = __float_as_uint(f);
    return (unsigned long long)((u & 0x7fffffu) | 0x800000u) << (((u >> 23) & 0xffu) - 150u);
  }
  return __float2uint_rn(f);
}

// ceil(gamma * z) exactly, for 0 < gamma <= 1 and z < 2^64, in integers:
// gamma = m * 2^-k with a 24-bit m, so gamma * z = (m * z) >> k rounded up
// (the product needs up to 88 bits: high and low 64-bit words).
__device__ __forceinline__ unsigned long long ceil_gamma_times(float gamma, unsigned long long z) {
  const uint32_t u = __float_as_uint(gamma);
  const uint32_t e = (u >> 23) & 0xffu;  // gamma >= 2^-126 is normal for every gamma passed
  const unsigned long long m = (u & 0x7fffffu) | 0x800000u;
  const int k = 150 - (int)e;  // gamma = m * 2^-k, k >= 23 for gamma <= 1
  const unsigned long long lo = m * z, hi = __umul64hi(m, z);
  if (k >= 128) return (lo | hi) ? 1ull : 0ull;
  unsigned long long q;  // (hi:lo) >> k
  bool rem;
  if (k >= 64) {
    q = hi >> (k - 64);
    rem = lo != 0 || (k > 64 && (hi & ((1ull << (k - 64)) - 1ull)) != 0);
  } else {
    q = (lo >> k) | (k ? hi << (64 - k) : 0ull);
    rem = (lo & ((1ull << k) - 1ull)) != 0;
  }
  return q + (rem ? 1ull : 0ull);
}

// Ties at the cutoff key: how many pages of weight w (> 0) the remaining
// weight rem needs, ceil(rem / w), from a float estimate corrected exactly
// in integers. Results of 2^22 and more exceed every tie count (at most
// 2^20 pages) and are returned as 2^40.
__device__ __forceinline__ unsigned long long ceil_div_count(unsigned long long rem,
                                                             unsigned long long w) {
  const float est = ceilf((float)rem / (float)w);
  if (est >= 4194304.0f) return 1ull << 40;
  unsigned long long t = (unsigned long long)est;
  while (t * w < rem) ++t;
  while (t > 1 && (t - 1) * w >= rem) --t;
  return t;
}

}  // namespace score
}  // namespace asp
