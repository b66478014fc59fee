// Device helpers shared by the libtq kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "tq_internal.h"

namespace tq {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Warp-level coordinate mapping used by every warp-per-vector routine.
//
// A vector of D = 32*E coordinates is spread over the 32 lanes of a warp;
// lane l holds E values, element e being coordinate
//     coord(e, l) = 32 e + 2 (l & 15) + (l >> 4).
// Within each aligned 32-coordinate word this is the "even/odd split" order
// of the bit planes (coordinate 32w + 2j + s sits at bit 16 s + j), so one
// __ballot_sync over element e yields plane word e directly.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int coord_of(int e, int lane) { return 32 * e + 2 * (lane & 15) + (lane >> 4); }

// Alternate-layout page of 16 tokens: the key bytes (a kb-bit code stream per token and 16 x d/32
// fp16 (scale, minimum) pairs, or with kb = 16 the fp16 keys themselves and no pairs), a dense
// vb-bit stream of value indices per token, 16 fp16 value norms.
__host__ __device__ constexpr int alt_key_bytes(int d, int kb) { return kb == 16 ? 32 * d : (2 * kb + 2) * d; }
__host__ __device__ constexpr int alt_tile_bytes(int d, int kb, int vb) { return alt_key_bytes(d, kb) + 2 * vb * d + 32; }

// Sylvester Walsh-Hadamard transform (unnormalised) of a warp-distributed
// vector, y_i = sum_j (-1)^popcount(i & j) x_j.  Index bit 0 is lane bit 4,
// index bits 1..4 are lane bits 0..3, index bits >= 5 are the element index.
// Each butterfly maps (lo, hi) -> (lo + hi, lo - hi).
template <int E>
__device__ __forceinline__ void wht_warp(float (&x)[E], int lane) {
#pragma unroll
  for (int lb = 0; lb < 5; ++lb) {
    const int mask = lb == 0 ? 16 : (1 << (lb - 1));
    const float sgn = (lane & mask) ? -1.f : 1.f;  // upper half: p - x, lower half: x + p
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float p = __shfl_xor_sync(kFull, x[e], mask);
      x[e] = fmaf(sgn, x[e], p);
    }
  }
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (!(e & h)) {
        float a = x[e], b = x[e | h];
        x[e] = a + b;
        x[e | h] = a - b;
      }
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
  return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, m));
  return v;
}

// Minimum and maximum of each of the E groups of a warp-distributed vector (group e = element e
// of every lane): one warp-wide float reduction each (redux.sync, exact).
template <int E>
__device__ __forceinline__ void group_minmax(const float (&v)[E], float (&mn)[E], float (&mx)[E]) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(mx[e]) : "f"(v[e]));
    asm("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(mn[e]) : "f"(v[e]));
  }
}

// rint of the IEEE quotient num / s (round half to even), with rs an approximate 1 / s: the
// product num * rs decides, unless it lies within 2^-10 of a rounding boundary k + 1/2, where the
// correctly rounded quotient is formed and rounded instead.  Exact for quotients below 2^12 (the
// product's error is then far below 2^-10); the callers clamp larger ones to the top level.
__device__ __forceinline__ float rint_quot(float num, float s, float rs) {
  const float t = num * rs;
  if (fabsf(t - floorf(t) - 0.5f) < 0.0009765625f) return rintf(__fdiv_rn(num, s));
  return rintf(t);
}
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// Group quantisers of a warp-distributed vector (group e = element e of every lane), IEEE float32
// arithmetic without contraction, the (scale, minimum) of each group stored as fp16:
//   asymmetric min/max:      s = fp16((mx - mn) / levels),            mn = fp16(mn)
//   signed symmetric:        s = fp16(max |x| / (levels / 2)),         mn = fp16(-(levels / 2) s)
//   q = clamp(rint((v - mn) / s), 0, levels), q = 0 when s == 0 (v and mn are fp16 values, so the
//   asymmetric mn is exact in either precision).
// Each group's pair is formed once, by lane e for group e (one IEEE division per lane instead of
// E), and one shuffle per group hands it to the warp; `mine` is lane e's own pair (lanes >= E:
// group 0's), for the store.
template <int E, bool SIGNED>
__device__ __forceinline__ void group_pairs(const float (&mn)[E], const float (&mx)[E], float levels, int lane,
                                            __half2 (&sm)[E], __half2& mine) {
  static_assert(E <= 32, "one lane per group");
  float lo = mn[0], hi = mx[0];
#pragma unroll
  for (int e = 1; e < E; ++e)
    if (lane == e) {
      lo = mn[e];
      hi = mx[e];
    }
  __half s, m;
  if (SIGNED) {
    const float half = 0.5f * levels;
    s = __float2half_rn(__fdiv_rn(fmaxf(-lo, hi), half));
    m = __float2half_rn(__fmul_rn(-half, __half2float(s)));
  } else {
    s = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), levels));
    m = __float2half_rn(lo);
  }
  mine = __halves2half2(s, m);
#pragma unroll
  for (int e = 0; e < E; ++e) sm[e] = __shfl_sync(kFull, mine, e);
}
// The code of v in the group with the fp16 pair (s, mn).
__device__ __forceinline__ int group_code(float v, __half2 sm, float levels) {
  const float s = __low2float(sm), mn = __high2float(sm);
  int q = 0;
  if (s > 0.f) {
    float t = rint_quot(__fsub_rn(v, mn), s, rcp_approx(s));
    t = fminf(fmaxf(t, 0.f), levels);
    q = (int)t;
  }
  return q;
}

// c[idx] of a 2-, 4- or 8-entry codebook (kb - 1 = 1, 2 or 3 index bits) by a select tree on the
// index bits i0 (high) .. i2, without an indexed (local-memory) access.
__device__ __forceinline__ float sel_bits(const CodeTables& t, int kb, bool i0, bool i1, bool i2) {
  if (kb == 2) return i0 ? t.c[1] : t.c[0];
  if (kb == 3) return i0 ? (i1 ? t.c[3] : t.c[2]) : (i1 ? t.c[1] : t.c[0]);
  const float lo = i1 ? (i2 ? t.c[3] : t.c[2]) : (i2 ? t.c[1] : t.c[0]);
  const float hi = i1 ? (i2 ? t.c[7] : t.c[6]) : (i2 ? t.c[5] : t.c[4]);
  return i0 ? hi : lo;
}

__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t bit) { atomicOr(err, bit); }

}  // namespace tq
