// mma.sync building blocks of the main-layout decode kernels (decode_tc.cu, decode_hy.cu):
// fp16 m16n8k16 products with fp32 accumulation, the fp16 high/low split of fp32 operands,
// per-lane cp.async staging, the per-warp online-softmax state and the exact recent-buffer page.
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace tq {
namespace {

constexpr int kTcD = 128;  // head_dim of the tensor-core decoders

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// 2^x (log2-domain softmax weights, x <= kLazyLog2); -inf gives +0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// fp16 high/low split of a pair: high = fp16(v), low = fp16((v - high) * 2^11).
// The low part is stored scaled so that it has the magnitude of the high part
// (|v - high| <= 2^-11 |v|): it never becomes subnormal before the high part
// does, and the scale cannot overflow.  Rows of low parts accumulate into
// their own accumulator rows, which are multiplied by 2^-11 in the epilogue.
constexpr float kLoScale = 2048.f;
constexpr float kLoUnscale = 1.f / 2048.f;
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  hi = h2_bits(h);
  lo = h2_bits(__floats2half2_rn((a - hf.x) * kLoScale, (b - hf.y) * kLoScale));
}

__device__ __forceinline__ void cp16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ int tc_nc(const TcArgs& a, int b) {
  const int nc = a.n_compressed[b];
  if (nc < 0 || (nc & 15) || nc > a.max_blocks * kPage) {
    if (threadIdx.x == 0) flag_error(a.err, TQ_DEVERR_POSITION);
    return 0;
  }
  if (nc > a.max_ctx) {
    if (threadIdx.x == 0) flag_error(a.err, TQ_DEVERR_CHUNKS);
    return 0;
  }
  return nc;
}

__device__ __forceinline__ int tc_nb(const TcArgs& a, int b) {
  if (!a.n_buf) return 0;
  const int nb = a.n_buf[b];
  if (nb < 0 || nb > kRing) {
    if (threadIdx.x == 0) flag_error(a.err, TQ_DEVERR_RING);
    return 0;
  }
  return nb;
}

struct WarpState {
  float m, l;
  float o[16][4];
  float mn[4];
};

// Online softmax with a lazily updated reference maximum.  The running state (m, l, o, mn) is
// only rescaled when some head's page maximum exceeds its reference by more than 2^kLazyLog2 (or
// on the first page); otherwise the reference stays and weights p = 2^(s - m) may reach
// 2^kLazyLog2.  The result is exact either way (l and o share the reference, and so do the
// split-K partials).  A warp sees few pages, so an eager update rescaled the 68 accumulators on most
// of them.  Weights reach 2^kLazyLog2, so a value weight p * s (s an fp16 group scale, < 2^16) is
// entered into the fp16 value operands as p * s * kWeightScale, which stays below the fp16 maximum
// for every scale; the product's output is multiplied back by 2^kLazyLog2.  The high/low split keeps
// ~22 bits of the weight even where the high part falls into the fp16 subnormal range.
constexpr float kLazyLog2 = 8.f;
constexpr float kWeightScale = 1.f / 256.f;  // 2^-kLazyLog2
__device__ __forceinline__ void softmax_update(WarpState& st, float (&s)[4], float (&p)[4]) {
  float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
  if (__any_sync(kFull, mx > st.m + kLazyLog2)) {
    const float m_new = fmaxf(st.m, mx);
    const float alpha = fast_exp2(st.m - m_new);
    st.l *= alpha;
    st.m = m_new;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) st.o[nt][r] *= alpha;
#pragma unroll
    for (int g = 0; g < 4; ++g) st.mn[g] *= alpha;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) p[k] = fast_exp2(s[k] - st.m);
  st.l += (p[0] + p[1]) + (p[2] + p[3]);
}

// One ring page: tokens t0 .. t0+cnt-1 of the exact fp16 buffer.
__device__ __forceinline__ void page_ring(const TcArgs& a, const uint4 (&Aq)[8], const __half* rk, const __half* rv,
                                          int t0, int cnt, WarpState& st, int lane) {
  const int g = lane >> 2, t = lane & 3;
  float acc[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[n][r] = 0.f;
  const uint32_t* k0 = reinterpret_cast<const uint32_t*>(rk + (size_t)(t0 + g) * kTcD);
  const uint32_t* k1 = reinterpret_cast<const uint32_t*>(rk + (size_t)(t0 + g + 8) * kTcD);
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) {
    const int c = kb * 8 + t;  // uint32 index of dims kb*16 + 2t, +1
    mma_f16(acc[0], Aq[kb], k0[c], k0[c + 4]);
    mma_f16(acc[1], Aq[kb], k1[c], k1[c + 4]);
  }
  float s[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int tok = (k >> 1) * 8 + 2 * t + (k & 1);
    s[k] = tok < cnt ? acc[k >> 1][k & 1] * a.logit_scale : -INFINITY;
  }
  float p[4];
  softmax_update(st, s, p);
  uint4 Ap;
  split2(p[0], p[1], Ap.x, Ap.y);
  split2(p[2], p[3], Ap.z, Ap.w);
  const unsigned short* v16 = reinterpret_cast<const unsigned short*>(rv);
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int dim = nt * 8 + g;
    uint32_t e[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int tok = (k >> 1) * 8 + 2 * t + (k & 1);
      e[k] = tok < cnt ? (uint32_t)v16[(size_t)(t0 + tok) * kTcD + dim] : 0u;
    }
    mma_f16(st.o[nt], Ap, e[0] | (e[1] << 16), e[2] | (e[3] << 16));
  }
}

}  // namespace
}  // namespace tq
