// Main-layout decode attention on the tensor cores (head_dim 128, <= 8 query
// heads per KV head and CTA).
//
// The n_rep query heads that share a KV head turn one decode step into a
// small dense product per page of 16 tokens (the GQA grouping of the
// "TurboQuant-MLX overview", GPU kernel section: n_rep), so both halves run
// as mma.sync m16n8k16 (fp16 inputs, fp32 accumulation):
//
//   scores  S[16 x 16 tok] = Q'[16 x 384] . P[384 x 16 tok]
//     rows 0..7 = heads (fp16 high part), rows 8..15 = the same heads (fp16
//     low part, (value - high) * 2^11), so each product is good to ~22 bits;
//     K = three bit planes of 128 coordinates: the high and the low bit of
//     the 2-bit Lloyd-Max index and the QJL sign bit.  With a symmetric 2-bit
//     codebook, c[idx] = x a + y b for a, b = +-1 taken from the two index bits
//     (x = (c3+c2)/2, y = (c3-c2)/2), so the Lloyd-Max dot <q_r, c[idx]> and
//     the QJL dot <S q_r, 2 sigma - 1> are +-1 contractions, with -x q_r,
//     -y q_r and -S q_r as the rows.  Each bit enters the MMA at the position
//     it already has after one shift per word (an fp16 exponent or sign bit,
//     see enc12 .. enc15), the affine map from that value to +-1 being folded
//     into the query rows and the accumulators' start values.
//     logit = n_k (lm + sqrt(pi/2)/m n_r qjl) / sqrt(d)   (turboquant vLLM
//     guide, section 2 step 3, unbiased inner-product estimator).
//   values  O[16 x 128] += P'_g[16 x 16 tok] . C[16 tok x 128]
//     P'_g = p * s_g (fp16 high / low rows), C = the 2-bit codes taken from
//     the packed word as the exact fp16 values 1 + q/4 (one shift and one
//     bit-select per register); O = 4 (P'_g . C) + sum_t p_t (mn_g(t) - 4 s_g(t)),
//     i.e. the group minimum and the removal of the encoding offset enter once
//     per group and token through an fp32 accumulator (turboquant-bench:
//     asymmetric group quantisation).
//
// Work split: one CTA per (chunk of pages, KV-head group, sequence), four
// warps per CTA, each warp walking its own pages through a 4-deep cp.async
// pipeline with its own online-softmax state; warps combine at the end of the
// chunk, CTAs through a split-K partial that a small merge kernel combines
// (a sequence whose work fits one CTA is written directly).  The exact
// recent buffer is one more work item of the same kernel, scored from the raw
// fp16 keys and values with the same tensor-core path.
#include "tc_mma.cuh"

namespace tq {
namespace {

constexpr int D = 128;
constexpr int NWARP = 4;
constexpr int STAGES = 4;
// Score-side A planes for KB key bits: the Lloyd-Max planes (one per stored index bit, plus the
// XOR of the three bits for 4-bit keys) and the QJL plane; 8 k-steps of 16 coordinates each.
constexpr int a_planes(int kb) { return kb == 4 ? 5 : kb; }
constexpr int KSTEPS_MAX = 8 * a_planes(4);
// Query workspace per (sequence, head group): the A fragments, then the partial score offsets of
// each prep slice ([slice][Lloyd-Max / QJL][head] floats).
constexpr int kPrepSlices = 4;
constexpr int AFRAG_U4 = KSTEPS_MAX * 32 + kPrepSlices * 2 * kMaxRep / 4;
static_assert(AFRAG_U4 == kTcQueryU4, "query workspace layout");
static_assert(NWARP == kPrepSlices, "one prep slice per warp of the prep kernel");

// Tile of the main layout with KB key bits (KB bit planes of 2d bytes: the Lloyd-Max index
// bits, high first, then the QJL signs) and VB value bits (1600 bytes at KB = 3, VB = 2).
template <int KB, int VB>
struct TcLayout {
  static constexpr int NA = a_planes(KB);
  static constexpr size_t SMEM_A = (size_t)NA * 8 * 32 * sizeof(uint4);
  static constexpr int TILE = (2 * KB + 2 * VB + 2) * D + 64;
  static constexpr int O_VQ = 2 * KB * D;
  static constexpr int O_VSM = (2 * KB + 2 * VB) * D;
  static constexpr int O_NORM = (2 * KB + 2 * VB + 2) * D;
};
// ... and its staging in a CTA of NW warps (STAGES pages per warp, then the query fragments)
template <int KB, int VB, int NW = NWARP>
struct TcTile : TcLayout<KB, VB> {
  using TcLayout<KB, VB>::NA;
  using TcLayout<KB, VB>::SMEM_A;
  using TcLayout<KB, VB>::TILE;
  static constexpr size_t SMEM_STAGE = (size_t)NW * STAGES * TILE;
  static constexpr size_t SMEM_TOTAL = SMEM_A + SMEM_STAGE;
  static_assert((size_t)NW * kMaxRep * D * sizeof(float) <= SMEM_STAGE, "combine buffer fits the stages");
};


constexpr int kPartStride = D + 4;  // floats per split-K partial: o[D], m, l, pad (16-byte rows)

// Key bits as fp16 operands without a shift per element.  Lane t of an MMA takes bit pairs
// j = 4t .. 4t+3 of a plane word (bits j and j + 16: coordinates 32w + 2j and 32w + 2j + 1).  One
// multiplication by 2^(12 - 4t) moves them to bits 12..15 (and 28..31), i.e. onto fp16 exponent
// bits 2, 3, 4 and the sign bit, and one bit select per register then gives an fp16 pair whose
// value is affine in the bit, B = beta0 + (beta1 - beta0) b:
//   bit 12: 1/16 or 1        bit 13: 1/256 or 1        bit 14: 0 or 2        bit 15: 1 or -1
// The query side carries A' = -2 A / (beta1 - beta0) and the accumulator starts at the offset
// sum_k A_k (1 + 2 beta0 / (beta1 - beta0)); then offset + sum_k A'_k B_k = sum_k A_k (1 - 2 b_k),
// the +-1 contraction of the method.  No product carries an offset larger than |A| beside a
// signal of 2 |A|, so the fp32 accumulation keeps the precision of the plain +-1 form.  The bit
// position of coordinate c is 12 + ((c >> 1) & 3); its scale and offset factor:
__device__ __forceinline__ float bitenc_scale(int q2) {
  return q2 == 0 ? -32.f / 15.f : q2 == 1 ? -512.f / 255.f : q2 == 2 ? -1.f : 1.f;
}
__device__ __forceinline__ float bitenc_offset(int q2) {
  return q2 == 0 ? 17.f / 15.f : q2 == 1 ? 257.f / 255.f : q2 == 2 ? 1.f : 0.f;
}
__device__ __forceinline__ uint32_t enc12(uint32_t x) { return (x & 0x10001000u) | 0x2C002C00u; }
__device__ __forceinline__ uint32_t enc13(uint32_t x) { return (x & 0x20002000u) | 0x1C001C00u; }
__device__ __forceinline__ uint32_t enc14(uint32_t x) { return x & 0x40004000u; }
__device__ __forceinline__ uint32_t enc15(uint32_t x) { return (x & 0x80008000u) | 0x3C003C00u; }
// The shift as an integer multiply (FMA pipe), leaving the ALU pipe to the bit selects.
__device__ __forceinline__ uint32_t mul_lo(uint32_t a, uint32_t b) {
  uint32_t x;
  asm("mul.lo.u32 %0, %1, %2;" : "=r"(x) : "r"(a), "r"(b));
  return x;
}
// Coordinate of A-fragment register pair rh (0: regs 0/1, 1: regs 2/3) of lane group t in k-step kb
// of a plane (first of two adjacent coordinates).
__device__ __forceinline__ int frag_dim(int kb, int t, int rh) { return 32 * (kb >> 1) + 8 * t + 4 * (kb & 1) + 2 * rh; }

// ------------------------------------------------------------------ query side
// Per CTA, before its pages are scored (the first pages are already in flight):
// q_r = H (D q) / sqrt(d) for the group's heads, t = S q_r on the tensor cores
// (rows 0..7 = heads as fp16 high parts, rows 8..15 = their low parts x 2^11;
// B = S^T as high and low x 2^11 fragments), and the score-side A fragments
// (-x q_r, -y q_r, -t as fp16 high/low rows) in the exact register order of
// mma.sync m16n8k16: fragment (k-step, lane) holds
//   reg0 = row g,   cols 2t..2t+1     reg1 = row g+8, cols 2t..2t+1
//   reg2 = row g,   cols 2t+8..2t+9   reg3 = row g+8, cols 2t+8..2t+9
// with g = lane / 4, t = lane % 4; row g is head g (high part), row g+8 the
// same head's low part.
// The query values this lane rotates (heads warp + NW i, coordinates coord_of(e, lane)), times the
// random signs: loaded at the top of the kernel, together with the sequence's counts and its first
// block ids, so that these round trips to memory overlap.
template <int NW>
struct QueryRegs {
  static constexpr int HPW = kMaxRep / NW;  // heads per warp
  float x[HPW][D / 32];
};
template <int NW>
__device__ __forceinline__ void load_query(const TcArgs& a, int b, int h0, int lane, int warp, QueryRegs<NW>& r) {
#pragma unroll
  for (int e = 0; e < D / 32; ++e) {
    const int c = coord_of(e, lane);
    const float sg = a.signs[c];
#pragma unroll
    for (int i = 0; i < QueryRegs<NW>::HPW; ++i) {
      const int h = warp + NW * i;
      r.x[i][e] = h < a.nrg ? __half2float(a.q[((size_t)b * a.hq + h0 + h) * D + c]) * sg : 0.f;
    }
  }
}

// Query side of one CTA of NW warps: rotation; t = S q_r with warp w computing sketch rows
// (D / NW) w .. (D / NW)(w + 1) - 1; score offsets (slot w: this warp's part of the QJL offset,
// slot 0 also the Lloyd-Max offset); the fragments.  Ends with __syncthreads.
template <int NA, int NW>
__device__ __forceinline__ void build_query_frags(const TcArgs& a, QueryRegs<NW>& qx, uint4* sA, float (*qr)[D],
                                                  float (*qt)[D], float (*soff)[2][kMaxRep], int tid, int lane,
                                                  int warp) {
  constexpr int NJ = D / (8 * NW);  // sketch-row n-tiles per warp
  const float rs = rsqrtf((float)D);
#pragma unroll
  for (int i = 0; i < QueryRegs<NW>::HPW; ++i) {
    wht_warp<D / 32>(qx.x[i], lane);
#pragma unroll
    for (int e = 0; e < D / 32; ++e) qr[warp + NW * i][coord_of(e, lane)] = qx.x[i][e] * rs;
  }
  __syncthreads();
  {
    // t[h][j] = sum_i S[j][i] q_r[h][i].  Every coordinate this lane touches (16 ks + 2t +
    // {0, 1, 8, 9} of q_r, sketch rows 8 (NJ w + j) + 2t + {0, 1} of t) has bit position 12 + t, so
    // the lane's share of the score offsets is one factor times plain sums.
    const int g = lane >> 2, t = lane & 3;
    float ch[NJ][4], cl[NJ][4];
#pragma unroll
    for (int j = 0; j < NJ; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) ch[j][r] = cl[j][r] = 0.f;
    float sl = 0.f;
#pragma unroll 4  // four k-steps of sketch fragments in flight
    for (int ks = 0; ks < D / 16; ++ks) {
      const int k0 = 16 * ks + 2 * t;
      uint4 A;
      const float q0 = qr[g][k0], q1 = qr[g][k0 + 1], q8 = qr[g][k0 + 8], q9 = qr[g][k0 + 9];
      sl += (q0 + q1) + (q8 + q9);
      split2(q0, q1, A.x, A.y);
      split2(q8, q9, A.z, A.w);
      const uint4* bf = a.sfrag_enc + ((size_t)ks * (D / 8) + NJ * warp) * 32 + lane;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const uint4 bv = __ldg(bf + j * 32);
        mma_f16(ch[j], A, bv.x, bv.y);
        mma_f16(cl[j], A, bv.z, bv.w);
      }
    }
    // high x high + 2^-11 (low x high + high x low); low x low (2^-22) is dropped
    float sq = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int col = 8 * (NJ * warp + j) + 2 * t;
      const float t0 = fmaf(ch[j][2] + cl[j][0], kLoUnscale, ch[j][0]);
      const float t1 = fmaf(ch[j][3] + cl[j][1], kLoUnscale, ch[j][1]);
      qt[g][col] = t0;
      qt[g][col + 1] = t1;
      sq += t0 + t1;
    }
    const float cf = bitenc_offset(t);
    sl *= cf;
    sq *= cf;
    sl += __shfl_xor_sync(kFull, sl, 1);
    sl += __shfl_xor_sync(kFull, sl, 2);
    sq += __shfl_xor_sync(kFull, sq, 1);
    sq += __shfl_xor_sync(kFull, sq, 2);
    if (t == 0) {
      soff[warp][1][g] = -sq;  // QJL: this warp's sketch rows
      soff[warp][0][g] = warp == 0 ? ((a.lm_w[0] + a.lm_w[1]) + (a.lm_w[2] + a.lm_w[3])) * sl : 0.f;
    }
  }
  __syncthreads();
  // NA planes x 8 k-steps x 32 lanes x 2 register pairs, NW * 32 items per pass: a pass covers
  // NW / 2 k-steps of one plane, so the plane of every pass is a compile-time constant
  constexpr int KPP = NW / 2;  // k-steps per pass
  static_assert(8 % KPP == 0, "whole passes per plane");
  uint32_t* dst = reinterpret_cast<uint32_t*>(sA);
  const int half = tid & 1, L = (tid >> 1) & 31, g = L >> 2, t = L & 3;
#pragma unroll
  for (int it = 0; it < NA * (8 / KPP); ++it) {
    const int ks = KPP * it + (tid >> 6);  // k-steps: 8 per A plane, QJL last
    const int plane = it / (8 / KPP), kb = ks & 7;
    const int dim = frag_dim(kb, t, half);
    const float sc = bitenc_scale(2 * (kb & 1) + half);
    float v0, v1;
    if (plane == NA - 1) {  // QJL plane
      v0 = -qt[g][dim];
      v1 = -qt[g][dim + 1];
    } else {
      const float wl = plane == 0 ? a.lm_w[0] : plane == 1 ? a.lm_w[1] : plane == 2 ? a.lm_w[2] : a.lm_w[3];
      v0 = wl * qr[g][dim];
      v1 = wl * qr[g][dim + 1];
    }
    uint32_t hi, lo;
    split2(v0 * sc, v1 * sc, hi, lo);
    dst[(ks * 32 + L) * 4 + 2 * half] = hi;
    dst[(ks * 32 + L) * 4 + 2 * half + 1] = lo;
  }
  __syncthreads();
}

// When the decode grid is too large for every CTA to build its own fragments they are built
// once per (KV-head group, sequence) into the workspace, split over kPrepSlices CTAs: slice s
// covers coordinates 32 s .. 32 s + 31, i.e. k-steps 2s and 2s + 1 of every plane and sketch rows
// 32 s .. 32 s + 31 of t (four MMA n-tiles, one per warp), and writes its part of the score offsets.
__global__ void __launch_bounds__(128) tc_prep_kernel(TcArgs a) {
  __shared__ __align__(16) float qr[kMaxRep][D];
  __shared__ float qt[kMaxRep][32];
  const int hg = blockIdx.x, b = blockIdx.y, slice = blockIdx.z;
  const int h0 = (hg / a.groups) * a.n_rep + (hg % a.groups) * a.nrg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const float rs = rsqrtf((float)D);
  for (int h = warp; h < kMaxRep; h += NWARP) {
    float x[D / 32];
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      const int c = coord_of(e, lane);
      x[e] = h < a.nrg ? __half2float(a.q[((size_t)b * a.hq + h0 + h) * D + c]) * a.signs[c] : 0.f;
    }
    wht_warp<D / 32>(x, lane);
#pragma unroll
    for (int e = 0; e < D / 32; ++e) qr[h][coord_of(e, lane)] = x[e] * rs;
  }
  __syncthreads();
  {
    float ch[4] = {0.f, 0.f, 0.f, 0.f}, cl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int ks = 0; ks < D / 16; ++ks) {
      const int k0 = 16 * ks + 2 * t;
      uint4 A;
      split2(qr[g][k0], qr[g][k0 + 1], A.x, A.y);
      split2(qr[g][k0 + 8], qr[g][k0 + 9], A.z, A.w);
      const uint4 bv = __ldg(a.sfrag_enc + ((size_t)ks * (D / 8) + 4 * slice + warp) * 32 + lane);
      mma_f16(ch, A, bv.x, bv.y);
      mma_f16(cl, A, bv.z, bv.w);
    }
    const int col = 8 * warp + 2 * t;
    qt[g][col] = fmaf(ch[2] + cl[0], kLoUnscale, ch[0]);
    qt[g][col + 1] = fmaf(ch[3] + cl[1], kLoUnscale, ch[1]);
  }
  __syncthreads();
  uint4* base = a.afrag + ((size_t)b * a.hkv * a.groups + hg) * AFRAG_U4;
  uint32_t* dst = reinterpret_cast<uint32_t*>(base);
  for (int idx = tid; idx < (a.n_lm + 1) * 2 * 32 * 2; idx += NWARP * 32) {
    const int half = idx & 1, L = (idx >> 1) & 31, r = idx >> 6;  // r = plane * 2 + k-step of the slice
    const int plane = r >> 1, kb = 2 * slice + (r & 1);
    const int ks = plane * 8 + kb;
    const int gg = L >> 2, tt = L & 3;
    const int dim = frag_dim(kb, tt, half), loc = dim - 32 * slice;
    const float sc = bitenc_scale(2 * (kb & 1) + half);
    float v0, v1;
    if (plane == a.n_lm) {  // QJL plane
      v0 = -qt[gg][loc];
      v1 = -qt[gg][loc + 1];
    } else {
      const float wl = plane == 0 ? a.lm_w[0] : plane == 1 ? a.lm_w[1] : plane == 2 ? a.lm_w[2] : a.lm_w[3];
      v0 = wl * qr[gg][dim];
      v1 = wl * qr[gg][dim + 1];
    }
    uint32_t hi, lo;
    split2(v0 * sc, v1 * sc, hi, lo);
    dst[(ks * 32 + L) * 4 + 2 * half] = hi;
    dst[(ks * 32 + L) * 4 + 2 * half + 1] = lo;
  }
  // this slice's part of the score offsets (coordinate 32 slice + lane)
  {
    const float cf = bitenc_offset((lane >> 1) & 3);
    const float lsum = (a.lm_w[0] + a.lm_w[1]) + (a.lm_w[2] + a.lm_w[3]);
    float* off = reinterpret_cast<float*>(base + KSTEPS_MAX * 32) + slice * 2 * kMaxRep;
    for (int h = warp; h < kMaxRep; h += NWARP) {
      const float sl = warp_sum(qr[h][32 * slice + lane] * cf);
      const float sq = warp_sum(qt[h][lane] * cf);
      if (lane == 0) {
        off[h] = lsum * sl;
        off[kMaxRep + h] = -sq;
      }
    }
  }
}

// One compressed page (16 tokens) of the warp's KV head.  off_lm / off_qj: this lane's head's score
// offsets (the accumulators' start values, see bitenc_scale).
template <int KB, int VB>
__device__ __forceinline__ void page_compressed(const TcArgs& a, const uint4* sA, const uint8_t* T, WarpState& st,
                                                float off_lm, float off_qj, int lane) {
  using L = TcTile<KB, VB>;
  const int g = lane >> 2, t = lane & 3;
  // accumulators: rows g (high parts) start at the offset, rows g + 8 (low parts) at 0
  float acc[2][2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    acc[0][n][0] = acc[0][n][1] = off_lm;
    acc[1][n][0] = acc[1][n][1] = off_qj;
    acc[0][n][2] = acc[0][n][3] = acc[1][n][2] = acc[1][n][3] = 0.f;
  }
  // bit pairs 4t .. 4t+3 of each plane word to bits 12..15 (see enc12 .. enc15)
  const uint32_t shm = 1u << (12 - 4 * t);
  constexpr int NA = L::NA;
  uint4 xr0 = make_uint4(0u, 0u, 0u, 0u), xr1 = xr0;  // 4-bit keys: XOR of the index planes so far
#pragma unroll
  for (int p = 0; p < NA; ++p) {
    // A plane p: stored plane p (tokens g and g + 8), except for 4-bit keys: plane 3 = XOR of the
    // three index planes (the odd parity product), plane 4 = the QJL plane (stored plane 3)
    uint4 r0, r1;
    if (KB == 4 && p == 3) {
      r0 = xr0;
      r1 = xr1;
    } else {
      const int sp = (KB == 4 && p == 4) ? 3 : p;
      r0 = *reinterpret_cast<const uint4*>(T + 256 * sp + g * 16);
      r1 = *reinterpret_cast<const uint4*>(T + 256 * sp + (g + 8) * 16);
      if (KB == 4 && p < 3) {
        xr0 = make_uint4(xr0.x ^ r0.x, xr0.y ^ r0.y, xr0.z ^ r0.z, xr0.w ^ r0.w);
        xr1 = make_uint4(xr1.x ^ r1.x, xr1.y ^ r1.y, xr1.z ^ r1.z, xr1.w ^ r1.w);
      }
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t w0 = word_of(r0, w), w1 = word_of(r1, w);
      const uint32_t x0 = mul_lo(w0, shm), x1 = mul_lo(w1, shm);
      // k-step 2w: bits 12 (b0) and 13 (b1); k-step 2w + 1: bits 14 and 15
      const uint4 A0 = sA[(p * 8 + 2 * w) * 32 + lane];
      const uint4 A1 = sA[(p * 8 + 2 * w + 1) * 32 + lane];
      mma_f16(acc[p == NA - 1][0], A0, enc12(x0), enc13(x0));
      mma_f16(acc[p == NA - 1][1], A0, enc12(x1), enc13(x1));
      mma_f16(acc[p == NA - 1][0], A1, enc14(x0), enc15(x0));
      mma_f16(acc[p == NA - 1][1], A1, enc14(x1), enc15(x1));
    }
  }
  // logits of tokens 2t, 2t+1 (n-tile 0) and 8+2t, 9+2t (n-tile 1), log2 domain
  const float coef = a.qjl_coef, scale = a.logit_scale;
  float s[4];
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    const float2 nk = __half22float2(*reinterpret_cast<const __half2*>(T + L::O_NORM + (8 * n + 2 * t) * 2));
    const float2 nr = __half22float2(*reinterpret_cast<const __half2*>(T + L::O_NORM + 32 + (8 * n + 2 * t) * 2));
    const float lm0 = fmaf(acc[0][n][2], kLoUnscale, acc[0][n][0]);
    const float lm1 = fmaf(acc[0][n][3], kLoUnscale, acc[0][n][1]);
    const float qj0 = fmaf(acc[1][n][2], kLoUnscale, acc[1][n][0]);
    const float qj1 = fmaf(acc[1][n][3], kLoUnscale, acc[1][n][1]);
    s[2 * n] = nk.x * fmaf(coef * nr.x, qj0, lm0) * scale;
    s[2 * n + 1] = nk.y * fmaf(coef * nr.y, qj1, lm1) * scale;
  }
  float p[4];
  softmax_update(st, s, p);
  // value weights p * s_g as fp16 high/low rows, minimum term per group
  uint4 sm[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int tok = (k >> 1) * 8 + 2 * t + (k & 1);
    sm[k] = *reinterpret_cast<const uint4*>(T + L::O_VSM + tok * 16);
  }
  uint4 Ap[4];
#pragma unroll
  for (int gg = 0; gg < 4; ++gg) {
    float sc[4], mn[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t wv = word_of(sm[k], gg);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv));
      sc[k] = f.x;
      mn[k] = f.y;
    }
    float w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = p[k] * sc[k];
    // operands p * s * 2^-kLazyLog2 (< 2^16, see kWeightScale); the output is scaled back by vscale
    split2(w[0] * kWeightScale, w[1] * kWeightScale, Ap[gg].x, Ap[gg].y);
    split2(w[2] * kWeightScale, w[3] * kWeightScale, Ap[gg].z, Ap[gg].w);
    // group minimum, minus the 1 of the code encoding below (2^VB w, as the codes are scaled by 2^VB)
    float acc_mn = st.mn[gg];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc_mn = fmaf(p[k], mn[k], fmaf(-(float)(1 << VB), w[k], acc_mn));
    st.mn[gg] = acc_mn;
  }
  // VB-bit code q of tokens 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1) as the normal fp16 value
  // 1 + q / 2^VB (bit pattern 0x3C00 | q << (10 - VB)): exact, and free of the reduced
  // accumulation precision that subnormal operands get when products are chained.
  const uint32_t* vq = reinterpret_cast<const uint32_t*>(T + L::O_VQ);
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    uint32_t b0, b1;
    if (VB == 2) {
      const uint32_t wv = vq[nt * 8 + g];
      b0 = ((wv << (8 - 2 * t)) & 0x03000300u) | 0x3C003C00u;
      b1 = ((wv >> (2 * t)) & 0x03000300u) | 0x3C003C00u;
    } else {
      // word 0 holds tokens 0..7, word 1 tokens 8..15; pair t at bits 4t and 16 + 4t
      const uint32_t w0 = vq[nt * 8 + g], w1 = vq[D + nt * 8 + g];
      b0 = (((w0 >> (4 * t)) << 6) & 0x03C003C0u) | 0x3C003C00u;
      b1 = (((w1 >> (4 * t)) << 6) & 0x03C003C0u) | 0x3C003C00u;
    }
    mma_f16(st.o[nt], Ap[nt >> 2], b0, b1);
  }
}

// NW warps per CTA; MINB: CTAs per SM the register allocation must allow.
//   NW 8, MINB 1: grids of at most one CTA per SM (the query side is built once per SM, by 8 warps);
//   NW 4, MINB 2: grids that fit in one wave at 2 CTAs per SM (the extra registers remove spills
//                 from the page loop);
//   NW 4, MINB 3: larger grids, with the query fragments from tc_prep_kernel.
template <int KB, int VB, int MINB, int NW>
__global__ void __launch_bounds__(32 * NW, MINB) tc_decode_kernel(TcArgs a) {
  using L = TcTile<KB, VB, NW>;
  constexpr int NSLOT = NW > kPrepSlices ? NW : kPrepSlices;  // score-offset slots
  extern __shared__ __align__(16) uint8_t smem[];
  uint4* sA = reinterpret_cast<uint4*>(smem);
  uint8_t* stage = smem + L::SMEM_A;
  __shared__ float wm[NW][kMaxRep], wl[NW][kMaxRep];
  __shared__ int sblk[NW][STAGES];
  __shared__ __align__(16) float qr[kMaxRep][D];
  __shared__ __align__(16) float qt[kMaxRep][D];
  __shared__ __align__(16) float soff[NSLOT][2][kMaxRep];  // score offsets (partial sums)

  const int part = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int kvh = hg / a.groups;
  const int h0 = kvh * a.n_rep + (hg % a.groups) * a.nrg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  // Requested before the sequence's counts arrive (they decide what is used): the block ids of
  // this warp's first STAGES pages of the chunk (any index inside the block-table row is a valid
  // read) and, when this CTA builds its own query fragments, the query.
  const int32_t* btb = a.block_table + (size_t)b * a.max_blocks;
  const int pbeg = part * a.chunk_pages;
  int blk_pre[STAGES];
#pragma unroll
  for (int k = 0; k < STAGES; ++k) {
    const int idx = pbeg + warp + NW * k;
    blk_pre[k] = (part < a.n_chunks && idx < a.max_blocks) ? __ldg(btb + idx) : -1;
  }
  QueryRegs<NW> qx;
  if (!a.afrag && part < a.n_chunks) load_query<NW>(a, b, h0, lane, warp, qx);
  const int nc = tc_nc(a, b), nb = tc_nb(a, b);
  const int npages = nc >> 4;
  const int nch = (npages + a.chunk_pages - 1) / a.chunk_pages;
  const int nparts = nch + (nb > 0 ? 1 : 0);
  if (nparts == 0) {
    if (part == 0)
      for (int i = tid; i < a.nrg * D; i += blockDim.x) a.out[((size_t)b * a.hq + h0) * D + i] = 0.f;
    return;
  }
  const bool ring = part == a.n_chunks;
  if (ring ? nb == 0 : part >= nch) return;

  WarpState st;
  st.m = -INFINITY;
  st.l = 0.f;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) st.o[nt][r] = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) st.mn[k] = 0.f;
  // value codes entered as 1 + q/2^VB (the offset is removed through st.mn), weights scaled by kWeightScale
  float vscale = (float)(1 << VB) / kWeightScale;

  if (!ring) {
    if (a.afrag) {
      const uint4* af = a.afrag + ((size_t)b * a.hkv * a.groups + hg) * AFRAG_U4;
      for (int i = tid; i < L::NA * 8 * 32; i += blockDim.x) cp16(&sA[i], &af[i]);
      if (tid < kPrepSlices * 2 * kMaxRep / 4) cp16(reinterpret_cast<uint4*>(&soff[0][0][0]) + tid, &af[KSTEPS_MAX * 32 + tid]);
      cp_commit();
    }
    const int npg = min(npages, pbeg + a.chunk_pages) - pbeg;
    const int nw = npg > warp ? (npg - warp + NW - 1) / NW : 0;
    uint8_t* wst = stage + (size_t)warp * STAGES * L::TILE;
    // Block ids: the id of the next page to copy is read one page ahead, so the table read
    // never holds up a copy (or the compute queued behind it); the ids of the pages in flight
    // are kept per warp in shared memory.
    auto blk_of = [&](int k) { return k < nw ? __ldg(btb + pbeg + warp + NW * k) : -1; };
    auto issue = [&](int k, int blk) {
      if (k < nw) {
        if (lane == 0) sblk[warp][k % STAGES] = blk;
        if (blk >= 0 && blk < a.num_blocks) {
          const uint8_t* gsrc = a.pool + ((size_t)blk * a.hkv + kvh) * L::TILE;
          uint8_t* sdst = wst + (k % STAGES) * L::TILE;
          for (int c = lane; c < L::TILE / 16; c += 32) cp16(sdst + c * 16, gsrc + c * 16);
        }
      }
      cp_commit();
    };
#pragma unroll
    for (int k = 0; k < STAGES - 1; ++k) issue(k, k < nw ? blk_pre[k] : -1);
    int nxt = STAGES - 1 < nw ? blk_pre[STAGES - 1] : -1;
    if (a.afrag) {
      cp_wait<STAGES - 1>();
      __syncthreads();  // every thread's share of the fragments has landed
    } else {
      build_query_frags<L::NA, NW>(a, qx, sA, qr, qt, soff, tid, lane, warp);  // ends with __syncthreads
    }
    // score offsets of this lane's head: the partial sums (prep slices, or the warps of this CTA's
    // query side) added once, outside the page loop
    const int nslot = a.afrag ? kPrepSlices : NW;
    float off_lm = 0.f, off_qj = 0.f;
#pragma unroll
    for (int sl = 0; sl < NSLOT; ++sl) {
      if (sl < nslot) {
        off_lm += soff[sl][0][g];
        off_qj += soff[sl][1][g];
      }
    }
    for (int k = 0; k < nw; ++k) {
      __syncwarp();  // every lane is done with the slot and stage that are refilled next
      const int cur = nxt;
      nxt = blk_of(k + STAGES);
      issue(k + STAGES - 1, cur);
      cp_wait<STAGES - 1>();
      __syncwarp();
      const int blk = sblk[warp][k % STAGES];
      if (blk < 0 || blk >= a.num_blocks) {
        if (lane == 0) flag_error(a.err, TQ_DEVERR_BLOCK_ID);
        continue;
      }
      page_compressed<KB, VB>(a, sA, wst + (k % STAGES) * L::TILE, st, off_lm, off_qj, lane);
      __syncwarp();
    }
    cp_wait<0>();
  } else {
    vscale = 1.f;
    uint4 Aq[8];
    const __half* qh = a.q + ((size_t)b * a.hq + h0 + g) * D;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qh);
      Aq[kb].x = g < a.nrg ? q32[kb * 8 + t] : 0u;
      Aq[kb].y = 0u;
      Aq[kb].z = g < a.nrg ? q32[kb * 8 + t + 4] : 0u;
      Aq[kb].w = 0u;
    }
    const __half* rk = a.ring_k + ((size_t)b * a.hkv + kvh) * kRing * D;
    const __half* rv = a.ring_v + ((size_t)b * a.hkv + kvh) * kRing * D;
    for (int t0 = warp * 16; t0 < nb; t0 += NW * 16) page_ring(a, Aq, rk, rv, t0, min(16, nb - t0), st, lane);
  }

  // ---- per-warp results: head g, dims nt*8 + 2t + {0,1}
  float l = st.l;
  l += __shfl_xor_sync(kFull, l, 1);
  l += __shfl_xor_sync(kFull, l, 2);
  float mn[4];
#pragma unroll
  for (int gg = 0; gg < 4; ++gg) {
    mn[gg] = st.mn[gg];
    mn[gg] += __shfl_xor_sync(kFull, mn[gg], 1);
    mn[gg] += __shfl_xor_sync(kFull, mn[gg], 2);
  }
  __syncthreads();  // stage buffers are free: reuse them for the combine
  float* wo = reinterpret_cast<float*>(stage);  // [NW][kMaxRep][D]
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int dim = nt * 8 + 2 * t + e;
      wo[((size_t)warp * kMaxRep + g) * D + dim] = fmaf(st.o[nt][2 + e], kLoUnscale, st.o[nt][e]) * vscale + mn[nt >> 2];
    }
  }
  if (t == 0) {
    wm[warp][g] = st.m;
    wl[warp][g] = l;
  }
  __syncthreads();
  // per head: the CTA maximum, each warp's weight 2^(m_w - M) (in place of m_w) and the normaliser
  __shared__ float hM[kMaxRep], hden[kMaxRep];
  if (tid < kMaxRep) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w][tid]);
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = M == -INFINITY ? 0.f : exp2f(wm[w][tid] - M);
      wm[w][tid] = f;
      den = fmaf(f, wl[w][tid], den);
    }
    hM[tid] = M;
    hden[tid] = den;
  }
  __syncthreads();
  const bool direct = nparts == 1;  // sole contributor: write the output itself
  for (int i = tid; i < a.nrg * D; i += blockDim.x) {
    const int h = i / D, dim = i % D;
    const float M = hM[h], den = hden[h];
    float num = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) num = fmaf(wm[w][h], wo[((size_t)w * kMaxRep + h) * D + dim], num);
    if (direct) {
      a.out[((size_t)b * a.hq + h0 + h) * D + dim] = den > 0.f ? num / den : 0.f;
    } else {
      float* dst = a.parts + (((size_t)b * a.hq + h0 + h) * a.n_parts + part) * kPartStride;
      dst[dim] = num;
      if (dim == 0) {
        dst[D] = M;
        dst[D + 1] = den;
      }
    }
  }
}

// ------------------------------------------------------------------ merge
// o = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i over the split-K partials
// of one query head (sequences with a single partial were written directly).
// One CTA per (query head, sequence, quarter of the dimensions): the maxima
// and weighted sums are reduced over all partials by the whole CTA, then 16
// slices of partials x 8 lanes of 16-byte loads cover the 32 dimensions.
constexpr int kMergeSplit = 4;  // dimension quarters per head
constexpr int kMergeBatch = 8;  // chunk slots per thread on the one-round-trip path (<= 128 chunks)
__global__ void __launch_bounds__(128) tc_merge_kernel(TcArgs a) {
  extern __shared__ float sw[];  // [n_parts] weights
  __shared__ float4 red[16][8];
  __shared__ float s_m[NWARP], s_l[NWARP];
  const int h = blockIdx.x, b = blockIdx.y, quarter = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* base = a.parts + ((size_t)b * a.hq + h) * a.n_parts * kPartStride;
  const int slice = tid >> 3, q4 = tid & 7;  // 16 partial slices, 8 float4 of this quarter
  const int col4 = quarter * 8 + q4;
  if (a.n_chunks <= 16 * kMergeBatch) {
    // Up to 16 x kMergeBatch chunk slots (and the ring slot): every slot this thread may need is
    // requested at once, together with the sequence's counts, and the slots past the sequence's
    // chunk count are dropped afterwards, so the whole merge costs one round trip to L2.
    float m[kMergeBatch], l[kMergeBatch];
    float4 v[kMergeBatch];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      const int i = slice + 16 * j;
      if (i < a.n_chunks) {
        const float* pp = base + (size_t)i * kPartStride;
        m[j] = __ldcg(pp + D);
        l[j] = __ldcg(pp + D + 1);
        v[j] = __ldcg(reinterpret_cast<const float4*>(pp) + col4);
      }
    }
    const float* pr = base + (size_t)a.n_chunks * kPartStride;  // ring slot
    const float mr = __ldcg(pr + D), lr = __ldcg(pr + D + 1);
    const float4 vr = __ldcg(reinterpret_cast<const float4*>(pr) + col4);
    const int nc = tc_nc(a, b), nb = tc_nb(a, b);
    const int nch = ((nc >> 4) + a.chunk_pages - 1) / a.chunk_pages;
    if (nch + (nb > 0 ? 1 : 0) <= 1) return;  // written by the decode kernel itself
    float M = nb > 0 ? mr : -INFINITY;
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j)
      if (slice + 16 * j < nch) M = fmaxf(M, m[j]);
    M = warp_max(M);
    if (lane == 0) s_m[warp] = M;
    __syncthreads();
    M = fmaxf(fmaxf(s_m[0], s_m[1]), fmaxf(s_m[2], s_m[3]));
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float mi, float li, const float4& vi) {
      const float w = exp2f(mi - M);
      den = fmaf(w, li, den);
      acc.x = fmaf(w, vi.x, acc.x);
      acc.y = fmaf(w, vi.y, acc.y);
      acc.z = fmaf(w, vi.z, acc.z);
      acc.w = fmaf(w, vi.w, acc.w);
    };
    if (M != -INFINITY) {
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j)
        if (slice + 16 * j < nch) add(m[j], l[j], v[j]);
      if (nb > 0 && slice == 0) add(mr, lr, vr);
    }
    red[slice][q4] = acc;
    den = q4 == 0 ? den : 0.f;  // each slice's normaliser counted once
    den = warp_sum(den);
    if (lane == 0) s_l[warp] = den;
    __syncthreads();
    if (tid < 32) {
      den = (s_l[0] + s_l[1]) + (s_l[2] + s_l[3]);
      const int c = tid >> 2, comp = tid & 3;  // 8 float4 x 4 components = 32 dimensions
      float o = 0.f;
#pragma unroll
      for (int sl = 0; sl < 16; ++sl) {
        const float4 r = red[sl][c];
        o += comp == 0 ? r.x : comp == 1 ? r.y : comp == 2 ? r.z : r.w;
      }
      a.out[((size_t)b * a.hq + h) * D + quarter * 32 + tid] = den > 0.f ? o / den : 0.f;
    }
    return;
  }
  const int nc = tc_nc(a, b), nb = tc_nb(a, b);
  const int nch = ((nc >> 4) + a.chunk_pages - 1) / a.chunk_pages;
  const int nparts = nch + (nb > 0 ? 1 : 0);
  if (nparts <= 1) return;
  auto part = [&](int i) { return base + (size_t)(i < nch ? i : a.n_chunks) * kPartStride; };
  float M = -INFINITY;
  for (int i = tid; i < nparts; i += 128) {
    const float m = __ldcg(part(i) + D);
    sw[i] = m;
    M = fmaxf(M, m);
  }
  M = warp_max(M);
  if (lane == 0) s_m[warp] = M;
  __syncthreads();
  M = fmaxf(fmaxf(s_m[0], s_m[1]), fmaxf(s_m[2], s_m[3]));
  float den = 0.f;
  for (int i = tid; i < nparts; i += 128) {
    const float w = M == -INFINITY ? 0.f : exp2f(sw[i] - M);
    sw[i] = w;
    den = fmaf(w, __ldcg(part(i) + D + 1), den);
  }
  den = warp_sum(den);
  __syncthreads();  // all weights written; s_m reads done
  if (lane == 0) s_l[warp] = den;
  __syncthreads();
  den = (s_l[0] + s_l[1]) + (s_l[2] + s_l[3]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int i = slice; i < nparts; i += 16) {
    const float w = sw[i];
    const float4 v = __ldcg(reinterpret_cast<const float4*>(part(i)) + col4);
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  red[slice][q4] = acc;
  __syncthreads();
  if (tid < 32) {
    const int c = tid >> 2, comp = tid & 3;  // 8 float4 x 4 components = 32 dimensions
    float o = 0.f;
#pragma unroll
    for (int sl = 0; sl < 16; ++sl) {
      const float4 v = red[sl][c];
      o += comp == 0 ? v.x : comp == 1 ? v.y : comp == 2 ? v.z : v.w;
    }
    a.out[((size_t)b * a.hq + h) * D + quarter * 32 + tid] = den > 0.f ? o / den : 0.f;
  }
}

}  // namespace

bool tc_supported(const tq_ctx* ctx) {
  return ctx->cfg.layout == TQ_LAYOUT_MAIN && ctx->cfg.head_dim == D;
}

void tc_set_score_constants(const tq_ctx* ctx, TcArgs& a) {
  // Lloyd-Max row weights.  A bit enters the products as P = 1 - 2 bit = +-1, and a symmetric
  // codebook (c[K-1-i] = -c[i]) is odd under flipping every index bit, so c[idx] is a combination
  // of the odd parity products of the P's: one term per index bit, plus P0 P1 P2 for a 3-bit
  // index (whose plane is the XOR of the three stored planes).  Each weight is a Walsh
  // coefficient: (1/K) sum_idx c[idx] chi(idx).
  const int nb = ctx->cfg.key_bits - 1, K = 1 << nb;
  a.n_lm = nb == 3 ? 4 : nb;
  for (int p = 0; p < a.n_lm; ++p) {
    double w = 0.0;
    for (int idx = 0; idx < K; ++idx) {
      int par = 0;  // parity of the bits in the product
      if (p < nb)
        par = (idx >> (nb - 1 - p)) & 1;  // plane p = index bit nb-1-p (high bit first)
      else
        par = ((idx >> 2) ^ (idx >> 1) ^ idx) & 1;
      w += (double)ctx->h_centroids[idx] * (par ? -1.0 : 1.0);
    }
    a.lm_w[p] = (float)(w / K);
  }
  for (int p = a.n_lm; p < 4; ++p) a.lm_w[p] = 0.f;
  a.qjl_coef = 1.2533141373155003f / (float)ctx->cfg.qjl_m;
  a.logit_scale = (float)(1.4426950408889634 / 11.313708498984761);  // log2(e) / sqrt(128)
}

cudaError_t launch_tc_merge(tq_ctx* ctx, TcArgs& a, int batch, cudaStream_t s) {
  prof_start(ctx, kProfMerge, s);
  tc_merge_kernel<<<dim3(a.hq, batch, kMergeSplit), 128, sizeof(float) * a.n_parts, s>>>(a);
  prof_stop(ctx, kProfMerge, s);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) ctx->launches++;
  return e;
}

cudaError_t launch_decode_tc(tq_ctx* ctx, TcArgs& a, int batch, cudaStream_t s) {
  const int hgroups = a.hkv * a.groups;
  tc_set_score_constants(ctx, a);
  cudaError_t e = cudaSuccess;
  if (a.afrag) {
    tc_prep_kernel<<<dim3(hgroups, batch, kPrepSlices), 128, 0, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ctx->launches++;
  }
  const int kb = ctx->cfg.key_bits;
  const bool v4 = ctx->cfg.value_bits == 4;
  // 8-warp CTAs when the plan gives at most one CTA per SM (a.cta_warps == 8); otherwise 4-warp CTAs,
  // with the 2-CTA-per-SM register budget when the grid fits one wave at 2 per SM
  const bool w8 = a.cta_warps == 8;
  const bool wide = (int64_t)a.n_parts * hgroups * batch <= 2 * (int64_t)ctx->sm_count;
  using KernFn = void (*)(TcArgs);
  KernFn kern;
  size_t smem;
  if (w8) {
    kern = kb == 4 ? (v4 ? tc_decode_kernel<4, 4, 1, 8> : tc_decode_kernel<4, 2, 1, 8>)
         : kb == 3 ? (v4 ? tc_decode_kernel<3, 4, 1, 8> : tc_decode_kernel<3, 2, 1, 8>)
                   : (v4 ? tc_decode_kernel<2, 4, 1, 8> : tc_decode_kernel<2, 2, 1, 8>);
    smem = kb == 4 ? (v4 ? TcTile<4, 4, 8>::SMEM_TOTAL : TcTile<4, 2, 8>::SMEM_TOTAL)
         : kb == 3 ? (v4 ? TcTile<3, 4, 8>::SMEM_TOTAL : TcTile<3, 2, 8>::SMEM_TOTAL)
                   : (v4 ? TcTile<2, 4, 8>::SMEM_TOTAL : TcTile<2, 2, 8>::SMEM_TOTAL);
  } else {
    kern = wide ? (kb == 4 ? (v4 ? tc_decode_kernel<4, 4, 2, 4> : tc_decode_kernel<4, 2, 2, 4>)
                 : kb == 3 ? (v4 ? tc_decode_kernel<3, 4, 2, 4> : tc_decode_kernel<3, 2, 2, 4>)
                           : (v4 ? tc_decode_kernel<2, 4, 2, 4> : tc_decode_kernel<2, 2, 2, 4>))
                : (kb == 4 ? (v4 ? tc_decode_kernel<4, 4, 3, 4> : tc_decode_kernel<4, 2, 3, 4>)
                 : kb == 3 ? (v4 ? tc_decode_kernel<3, 4, 3, 4> : tc_decode_kernel<3, 2, 3, 4>)
                           : (v4 ? tc_decode_kernel<2, 4, 3, 4> : tc_decode_kernel<2, 2, 3, 4>));
    smem = kb == 4 ? (v4 ? TcTile<4, 4>::SMEM_TOTAL : TcTile<4, 2>::SMEM_TOTAL)
         : kb == 3 ? (v4 ? TcTile<3, 4>::SMEM_TOTAL : TcTile<3, 2>::SMEM_TOTAL)
                   : (v4 ? TcTile<2, 4>::SMEM_TOTAL : TcTile<2, 2>::SMEM_TOTAL);
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ctx->decode_kernel = "tc_decode_kernel";
  prof_start(ctx, kProfDecode, s);
  kern<<<dim3(a.n_parts, hgroups, batch), w8 ? 256 : 128, smem, s>>>(a);
  prof_stop(ctx, kProfDecode, s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ctx->launches++;
  return launch_tc_merge(ctx, a, batch, s);
}

}  // namespace tq
