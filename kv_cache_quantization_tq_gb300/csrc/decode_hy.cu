// Main-layout decode attention with the score on the 5th-generation tensor cores (tcgen05) and the
// value product on mma.sync: default widths (3-bit keys = 2-bit Lloyd-Max index + QJL sign, 2-bit
// values), head_dim 128, at most 8 query heads per KV head and CTA.
//
// Score (turboquant vLLM guide, section 2 step 3, unbiased inner-product estimator; the GQA
// grouping of the "TurboQuant-MLX overview", GPU kernel section):
//   logit = n_k (lm + sqrt(pi/2)/m n_r qjl) / sqrt(d),  lm = x <q_r, P_h> + y <q_r, P_l>,
//   qjl = <S q_r, P_s>,  P = 2 bit - 1 (+-1), x = (c3 + c2)/2, y = (c3 - c2)/2.
// A tile of 128 tokens (8 pages) is one tcgen05.mma M = 128 problem: each token's 384 key bits
// are spread into e4m3 bytes in tensor memory (row = token, lane = thread), one bit per byte at an
// exponent or sign bit position P of the byte (a bit select per four bytes: byte = base_P |
// bit << P, an e4m3 value beta0_P + delta_P bit), and multiplied by the query operand in shared
// memory: the three query vectors (x q_r, y q_r, S q_r) rescaled by 2 / delta_P and split into six e4m3
// pieces of ~4 bits each (N = 8 heads x 6 pieces = 48 columns).  The Lloyd-Max and QJL sums land
// in two fp32 accumulators in tensor memory; the epilogue (thread = token) adds the pieces with
// their power-of-two scales and the offset sum_k A_k (1 + 2 beta0/delta) that turns the byte values
// back into +-1.  Six pieces keep ~24 bits of every query coefficient.
// Measured on GB300: a tcgen05.mma with M = 128 costs ~44 cycles whatever N is up to 64, so K = 32
// per instruction (e4m3) halves the score's tensor time against fp16 operands (K = 16).
//
// Values (turboquant-bench: asymmetric group quantisation): as in decode_tc.cu, on mma.sync
// with the softmax weights p of the tile read back from shared memory.
//
// Softmax: one reference maximum per head for the whole CTA, updated lazily per tile (only when
// a logit exceeds it by more than 2^kLazyLog2); every warp's value accumulators share it, so the
// warps' results add without reweighting.
//
// Work split and merge: the chunks / ring item / split-K partials of decode_tc.cu; the ring item
// runs the mma.sync path of decode_tc.cu.  Every wait on an mbarrier is bounded (about a second):
// on expiry the CTA flags TQ_DEVERR_TIMEOUT, drains its copies, frees its tensor memory and leaves.
#include <cuda_fp8.h>

#include "tc_mma.cuh"

namespace tq {
namespace {

constexpr int D = kTcD;
constexpr int NW = 4;                  // warps per CTA
constexpr int TILE_PAGES = 8;          // pages per score tile: 128 tokens = M of the MMA
constexpr int TILE_TOK = TILE_PAGES * kPage;
constexpr int STAGES = 4;              // tiles of pages in shared memory
constexpr int PAGE_BYTES = 12 * D + 64;  // main tile, 3-bit keys and 2-bit values: 1600
constexpr int O_VQ = 6 * D, O_VSM = 10 * D, O_NORM = 12 * D;
constexpr int NPIECE = 6;
constexpr int QN = kMaxRep * NPIECE;   // columns of each score accumulator
constexpr int SLICE_BYTES = QN * 32;   // one K = 32 slice of the query operand
constexpr int NSLICE = 12;             // 3 planes x 4 words of 32 bits per token
constexpr int QOP_BYTES = NSLICE * SLICE_BYTES;
// Query record per (sequence, head group): the operand, then scale[2][8] (2^-e0 of piece 0 of
// the Lloyd-Max and QJL sets) and off[2][8] (their offsets), floats.
constexpr int QREC_BYTES = QOP_BYTES + 4 * 4 * kMaxRep;
static_assert(QREC_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");
static_assert(QREC_BYTES == kHyQueryBytes, "query record size");
// Tensor-memory columns: key bytes (96), Lloyd-Max and QJL accumulators (48 each).
constexpr int TM_A = 0, TM_LM = 96, TM_QJ = 144, TM_COLS = 256;
// tcgen05 instruction descriptor: kind::f8f6f4, A = B = E4M3, D = F32, K-major, N = 48, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(QN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

// Dynamic shared memory (offsets from a 1024-byte aligned base).
constexpr int OFF_Q = 0;
constexpr int OFF_STAGE = QREC_BYTES;
constexpr int STAGE_BYTES = TILE_PAGES * PAGE_BYTES;
constexpr int OFF_PBUF = OFF_STAGE + STAGES * STAGE_BYTES;
constexpr int PBUF_BYTES = kMaxRep * TILE_TOK * 4;
constexpr int OFF_MISC = OFF_PBUF + 2 * PBUF_BYTES;
constexpr int OFF_BAR_FULL = OFF_MISC;               // STAGES mbarriers
constexpr int OFF_BAR_MMA = OFF_MISC + 8 * STAGES;
constexpr int OFF_BAR_Q = OFF_BAR_MMA + 8;
constexpr int OFF_TMEM = OFF_BAR_Q + 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int OFF_VALID = OFF_ABORT + 4;             // [STAGES] valid-page masks
constexpr int OFF_WRED = OFF_VALID + 4 * STAGES;     // [NW][kMaxRep] floats
constexpr int OFF_WRED2 = OFF_WRED + 4 * NW * kMaxRep;
constexpr int MISC_BYTES = OFF_WRED2 + 4 * NW * kMaxRep - OFF_MISC;
constexpr int SMEM_USED = OFF_MISC + MISC_BYTES;
// With the alignment slack: above a third of the SM's shared memory, so at most two CTAs (2 x 256
// tensor-memory columns) share an SM and tcgen05.alloc never waits.
constexpr int HY_SMEM = SMEM_USED + 1024 > 80 * 1024 ? SMEM_USED + 1024 : 80 * 1024;
static_assert((size_t)NW * kMaxRep * D * sizeof(float) <= (size_t)STAGES * STAGE_BYTES, "combine buffer fits");
static_assert(OFF_STAGE % 16 == 0 && OFF_PBUF % 16 == 0 && OFF_MISC % 16 == 0, "alignment");

// A key bit lands at bit position P of its e4m3 byte, which then holds base_P when the bit is 0 and
// base_P | 1 << P when it is 1 (the e4m3 value beta0 + delta bit).  Only three positions are used:
//   P = 5 (exponent bit 2): 0.0625 or 1        P = 6 (exponent top bit): 1 or 256
//   P = 7 (sign): 1 or -1
// so that the offset sum_k A_k (1 + 2 beta0 / delta), which cancels against the product, is never
// more than 1.13 sum |A| (mantissa positions would reach 17 sum |A| and cost ~4 bits of the fp32
// result).  Bit j of each byte of a plane word goes to position pos_of(j): bits 5..7 stay, bits
// 2..4 move up by 3 and bits 0..1 by 5 (one shift per group).
__host__ __device__ constexpr int pos_of(int j) { return j >= 5 ? j : j >= 2 ? j + 3 : j + 5; }
__host__ __device__ constexpr uint32_t pos_base(int P) { return P == 5 ? 0x18u : 0x38u; }
__device__ __forceinline__ float pos_beta0(int P) { return P == 5 ? 0.0625f : 1.f; }
__device__ __forceinline__ float pos_delta(int P) { return P == 5 ? 0.9375f : P == 6 ? 255.f : -2.f; }
// Token-row bit (8 i + j) of plane word w (coordinate 32 w + 2 (b mod 16) + b / 16 of the stored
// even/odd order) becomes byte i of tensor-memory column 8 (4 p + w) + j, i.e. element k = 4 j + i
// of K-slice 4 p + w.
__device__ __forceinline__ uint32_t key_bytes(uint32_t x, int j) {
  const uint32_t y = j >= 5 ? x : j >= 2 ? x << 3 : x << 5;
  const int P = pos_of(j);
  return (y & (0x01010101u << P)) | (pos_base(P) * 0x01010101u);
}

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Bounded wait for phase `parity` (about a second of %globaltimer); false on expiry.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    if (ok) return true;
    if ((i & 63) == 0) {
      uint64_t now;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
      if (i == 0) t0 = now;
      else if (now - t0 > 1000000000ull) return false;
    }
  }
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
  // K-major, no swizzle: 8-row x 16-byte core matrices, 128 bytes apart along K (LBO) and 256
  // bytes apart along N (SBO); descriptor version 1.
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(256 >> 4) << 32) |
         ((uint64_t)1 << 46);
}
__device__ __forceinline__ void mma_f8(uint32_t d, uint32_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %3, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %4, p; }" ::"r"(d),
      "r"(a), "l"(b), "r"(acc), "n"(kIdesc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tm_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 48 columns of this warp's 32 lanes, loaded and waited for in one statement (the registers are
// defined only after tcgen05.wait::ld).
__device__ __forceinline__ void tm_ld48(uint32_t taddr, float (&v)[48]) {
  uint32_t r[48];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%48];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, "
      "[%49];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]),
        "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]),
        "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
      : "r"(taddr), "r"(taddr + 32)
      : "memory");
#pragma unroll
  for (int i = 0; i < 48; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- query record
// Per (sequence, head group), 4 warps: q_r = H (D q) / sqrt(d) of the group's heads, t = S q_r
// (mma.sync, fp16 high/low rows and S^T high/low fragments, as in decode_tc.cu), then the e4m3
// pieces of Q'_k = 2 A_k / delta_j (A = x q_r, y q_r on the two index planes, t on the QJL plane)
// in the canonical K-major layout of each K-slice, the per-(head, set) scale of piece 0 and the
// offsets -sum_k A_k (1 + 2 beta0_j / delta_j), so that offset + sum_k Q'_k byte_k = sum_k A_k (2 b_k - 1).
// With the Walsh weights of the codebook (c[idx] = sum_p lm_w[p] (1 - 2 b_p)), A = -lm_w[p] q_r on
// index plane p and A = t on the QJL plane.
__global__ void __launch_bounds__(128) hy_prep_kernel(TcArgs a, uint8_t* qrec) {
  __shared__ __align__(16) uint8_t rec[QREC_BYTES];
  __shared__ __align__(16) float qr[kMaxRep][D];
  __shared__ __align__(16) float qt[kMaxRep][D];
  __shared__ float red[2][kMaxRep][NW];
  const int hg = blockIdx.x, b = blockIdx.y;
  const int h0 = (hg / a.groups) * a.n_rep + (hg % a.groups) * a.nrg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float rs = rsqrtf((float)D);
  for (int h = warp; h < kMaxRep; h += NW) {
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
    // t[h][j] = sum_i S[j][i] q_r[h][i]: warp w covers sketch rows 32 w .. 32 w + 31 (4 n-tiles)
    const int g = lane >> 2, t = lane & 3;
    float ch[4][4], cl[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) ch[j][r] = cl[j][r] = 0.f;
#pragma unroll 2
    for (int ks = 0; ks < D / 16; ++ks) {
      const int k0 = 16 * ks + 2 * t;
      uint4 A;
      split2(qr[g][k0], qr[g][k0 + 1], A.x, A.y);
      split2(qr[g][k0 + 8], qr[g][k0 + 9], A.z, A.w);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 bv = __ldg(a.sfrag_enc + ((size_t)ks * (D / 8) + 4 * warp + j) * 32 + lane);
        mma_f16(ch[j], A, bv.x, bv.y);
        mma_f16(cl[j], A, bv.z, bv.w);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = 8 * (4 * warp + j) + 2 * t;
      qt[g][col] = fmaf(ch[j][2] + cl[j][0], kLoUnscale, ch[j][0]);
      qt[g][col + 1] = fmaf(ch[j][3] + cl[j][1], kLoUnscale, ch[j][1]);
    }
  }
  __syncthreads();
  // thread = coordinate c of every head and plane; A of (head h, plane p) at coordinate c
  const int c = tid;
  const int w = c >> 5, r = c & 31;
  const int bit = (r & 1) * 16 + (r >> 1);  // bit of plane word w that holds coordinate c
  const int j = bit & 7, i = bit >> 3;
  const float dl = pos_delta(pos_of(j)), cf = 1.f + 2.f * pos_beta0(pos_of(j)) / dl;
  float mx[2][kMaxRep], off[2][kMaxRep];
#pragma unroll
  for (int h = 0; h < kMaxRep; ++h) {
    const float a0 = -a.lm_w[0] * qr[h][c], a1 = -a.lm_w[1] * qr[h][c], a2 = qt[h][c];
    mx[0][h] = fmaxf(fabsf(a0), fabsf(a1)) * (2.f / fabsf(dl));
    mx[1][h] = fabsf(a2) * (2.f / fabsf(dl));
    off[0][h] = -(a0 + a1) * cf;
    off[1][h] = -a2 * cf;
  }
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) {
      const float m = warp_max(mx[s][h]);
      const float o = warp_sum(off[s][h]);
      if (lane == 0) red[s][h][warp] = m;
      mx[s][h] = m;
      off[s][h] = o;
    }
  __syncthreads();
  float* scale = reinterpret_cast<float*>(rec + QOP_BYTES);  // [2][8]
  float* offs = scale + 2 * kMaxRep;                         // [2][8]
  float e0[2][kMaxRep];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) {
      const float m = fmaxf(fmaxf(red[s][h][0], red[s][h][1]), fmaxf(red[s][h][2], red[s][h][3]));
      // piece 0 holds Q' * 2^e0 with 2^e0 * max |Q'| in (120, 240]: inside the e4m3 range
      e0[s][h] = m > 0.f ? floorf(log2f(240.f / m)) : 0.f;
    }
  __syncthreads();  // every thread has read red[][][]
  // offsets: reuse red[s][h][warp] for the per-warp partial sums
  if (lane == 0)
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) red[s][h][warp] = off[s][h];
  __syncthreads();
  if (tid < 2 * kMaxRep) {
    const int s = tid / kMaxRep, h = tid % kMaxRep;
    offs[s * kMaxRep + h] = (red[s][h][0] + red[s][h][1]) + (red[s][h][2] + red[s][h][3]);
    scale[s * kMaxRep + h] = exp2f(-e0[s][h]);
  }
  // the pieces: byte (n = 6 h + piece, k = 4 j + i) of slice 4 p + w
  const int k = 4 * j + i;
#pragma unroll
  for (int p = 0; p < 3; ++p) {
    uint8_t* slice = rec + (4 * p + w) * SLICE_BYTES + (k >> 4) * 128 + (k & 15);
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) {
      const float A = p == 0 ? -a.lm_w[0] * qr[h][c] : p == 1 ? -a.lm_w[1] * qr[h][c] : qt[h][c];
      float x = 2.f * A / dl * exp2f(e0[p == 2][h]);
#pragma unroll
      for (int pc = 0; pc < NPIECE; ++pc) {
        const __nv_fp8_e4m3 e(x);
        const int n = NPIECE * h + pc;
        slice[(n >> 3) * 256 + (n & 7) * 16] = e.__x;
        x = (x - static_cast<float>(e)) * 16.f;
      }
    }
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(qrec + ((size_t)b * a.hkv * a.groups + hg) * QREC_BYTES);
  const uint4* srcv = reinterpret_cast<const uint4*>(rec);
  for (int x = tid; x < QREC_BYTES / 16; x += 128) dst[x] = srcv[x];
}

// ---------------------------------------------------------------- decode
struct Smem {
  uint8_t* base;
  uint32_t base_s;
  __device__ uint8_t* ptr(int off) const { return base + off; }
  __device__ uint32_t addr(int off) const { return base_s + (uint32_t)off; }
};

// The ring item (exact fp16 buffer): the mma.sync path of decode_tc.cu, per-warp softmax states
// combined at the end.
__device__ void ring_item(const TcArgs& a, const Smem& sm, int b, int h0, int kvh, int nb, int nparts, int part) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  WarpState st;
  st.m = -INFINITY;
  st.l = 0.f;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) st.o[nt][r] = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) st.mn[k] = 0.f;
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
  float l = st.l;
  l += __shfl_xor_sync(kFull, l, 1);
  l += __shfl_xor_sync(kFull, l, 2);
  float* wo = reinterpret_cast<float*>(sm.ptr(OFF_STAGE));  // [NW][kMaxRep][D]
  float* wm = reinterpret_cast<float*>(sm.ptr(OFF_WRED));   // [NW][kMaxRep]
  float* wl = reinterpret_cast<float*>(sm.ptr(OFF_WRED2));
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e)
      wo[((size_t)warp * kMaxRep + g) * D + nt * 8 + 2 * t + e] = fmaf(st.o[nt][2 + e], kLoUnscale, st.o[nt][e]);
  if (t == 0) {
    wm[warp * kMaxRep + g] = st.m;
    wl[warp * kMaxRep + g] = l;
  }
  __syncthreads();
  for (int i = tid; i < a.nrg * D; i += NW * 32) {
    const int h = i / D, dim = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < NW; ++w2) M = fmaxf(M, wm[w2 * kMaxRep + h]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < NW; ++w2) {
      const float f = M == -INFINITY ? 0.f : exp2f(wm[w2 * kMaxRep + h] - M);
      num = fmaf(f, wo[((size_t)w2 * kMaxRep + h) * D + dim], num);
      den = fmaf(f, wl[w2 * kMaxRep + h], den);
    }
    if (nparts == 1) {
      a.out[((size_t)b * a.hq + h0 + h) * D + dim] = den > 0.f ? num / den : 0.f;
    } else {
      float* dst = a.parts + (((size_t)b * a.hq + h0 + h) * a.n_parts + part) * (D + 4);
      dst[dim] = num;
      if (dim == 0) {
        dst[D] = M;
        dst[D + 1] = den;
      }
    }
  }
}

// Value product of one page (16 tokens) of a tile for this warp: weights p of head g (lane
// g, t: tokens 2t, 2t+1, 8+2t, 9+2t) from the tile's p buffer, O += (p s_g) C as in decode_tc.cu.
__device__ __forceinline__ void page_values(const uint8_t* T, const float* pb, float (&o)[16][4], float (&mnacc)[4],
                                            int lane) {
  const int g = lane >> 2, t = lane & 3;
  const float2 p01 = *reinterpret_cast<const float2*>(pb + g * TILE_TOK + 2 * t);
  const float2 p89 = *reinterpret_cast<const float2*>(pb + g * TILE_TOK + 8 + 2 * t);
  const float p[4] = {p01.x, p01.y, p89.x, p89.y};
  uint4 smv[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int tok = (k >> 1) * 8 + 2 * t + (k & 1);
    smv[k] = *reinterpret_cast<const uint4*>(T + O_VSM + tok * 16);
  }
  uint4 Ap[4];
#pragma unroll
  for (int gg = 0; gg < 4; ++gg) {
    float sc[4], mn[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t wv = word_of(smv[k], gg);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv));
      sc[k] = f.x;
      mn[k] = f.y;
    }
    float w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = p[k] * sc[k];
    split2(w[0] * kWeightScale, w[1] * kWeightScale, Ap[gg].x, Ap[gg].y);
    split2(w[2] * kWeightScale, w[3] * kWeightScale, Ap[gg].z, Ap[gg].w);
    float acc = mnacc[gg];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc = fmaf(p[k], mn[k], fmaf(-4.f, w[k], acc));
    mnacc[gg] = acc;
  }
  const uint32_t* vq = reinterpret_cast<const uint32_t*>(T + O_VQ);
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const uint32_t wv = vq[nt * 8 + g];
    const uint32_t b0 = ((wv << (8 - 2 * t)) & 0x03000300u) | 0x3C003C00u;
    const uint32_t b1 = ((wv >> (2 * t)) & 0x03000300u) | 0x3C003C00u;
    mma_f16(o[nt], Ap[nt >> 2], b0, b1);
  }
}

__global__ void __launch_bounds__(NW * 32, 2) hy_decode_kernel(TcArgs a, const uint8_t* qrec) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  {
    const uint32_t s0 = smem_u32(smem_raw);
    const uint32_t al = (s0 + 1023u) & ~1023u;
    sm.base = smem_raw + (al - s0);
    sm.base_s = al;
  }
  const int part = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int kvh = hg / a.groups;
  const int h0 = kvh * a.n_rep + (hg % a.groups) * a.nrg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
  if (ring) {
    ring_item(a, sm, b, h0, kvh, nb, nparts, part);
    return;
  }

  // ---------------------------------------------------------------- compressed chunk
  const int pbeg = part * a.chunk_pages;
  const int npg = min(npages, pbeg + a.chunk_pages) - pbeg;
  const int ntiles = (npg + TILE_PAGES - 1) / TILE_PAGES;
  const int32_t* btb = a.block_table + (size_t)b * a.max_blocks + pbeg;
  uint32_t* abort_flag = reinterpret_cast<uint32_t*>(sm.ptr(OFF_ABORT));
  uint32_t* valid = reinterpret_cast<uint32_t*>(sm.ptr(OFF_VALID));
  const uint32_t bar_full = sm.addr(OFF_BAR_FULL), bar_mma = sm.addr(OFF_BAR_MMA), bar_q = sm.addr(OFF_BAR_Q);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sm.addr(OFF_TMEM)),
                 "n"(TM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Thread 0 issues every copy: the query record, then the first STAGES tiles of pages.
  int issued = 0;  // tiles whose copies thread 0 has issued
  // Block ids of a tile's pages (thread 0; -1 past the chunk), requested one tile before the copies
  // are issued so that the table read is off the path of the barrier that follows the issue.
  auto tile_blocks = [&](int ti, int (&blk)[TILE_PAGES]) {
    const int p0 = ti * TILE_PAGES, np = ti < ntiles ? min(TILE_PAGES, npg - p0) : 0;
#pragma unroll
    for (int q = 0; q < TILE_PAGES; ++q) blk[q] = q < np ? __ldg(btb + p0 + q) : -1;
  };
  auto issue_tile = [&](int ti, const int (&blk)[TILE_PAGES]) {
    issued = ti + 1;
    const int st = ti % STAGES;
    const int p0 = ti * TILE_PAGES, np = min(TILE_PAGES, npg - p0);
    uint32_t mask = 0, bytes = 0;
#pragma unroll
    for (int q = 0; q < TILE_PAGES; ++q) {
      if (q < np) {
        if (blk[q] >= 0 && blk[q] < a.num_blocks) {
          mask |= 1u << q;
          bytes += PAGE_BYTES;
        } else {
          flag_error(a.err, TQ_DEVERR_BLOCK_ID);
        }
      }
    }
    valid[st] = mask;
    mbar_expect_tx(bar_full + 8 * st, bytes);
#pragma unroll
    for (int q = 0; q < TILE_PAGES; ++q)
      if (mask >> q & 1)
        bulk_g2s(sm.addr(OFF_STAGE + st * STAGE_BYTES + q * PAGE_BYTES),
                 a.pool + ((size_t)blk[q] * a.hkv + kvh) * PAGE_BYTES, PAGE_BYTES, bar_full + 8 * st);
  };
  if (tid == 0) {
    *abort_flag = 0;
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(bar_full + 8 * s, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_q, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_expect_tx(bar_q, QREC_BYTES);
    bulk_g2s(sm.addr(OFF_Q), qrec + ((size_t)b * a.hkv * a.groups + hg) * QREC_BYTES, QREC_BYTES, bar_q);
    for (int ti = 0; ti < min(STAGES, ntiles); ++ti) {
      int blk[TILE_PAGES];
      tile_blocks(ti, blk);
      issue_tile(ti, blk);
    }
  }
  int nblk[TILE_PAGES];  // thread 0: block ids of the next tile to issue
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm.ptr(OFF_TMEM));
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  // per-thread state: the CTA's reference maxima (identical in every thread), this token's share of
  // the normalisers, the warp's value accumulators and group-minimum terms
  float mref[kMaxRep], lsum[kMaxRep];
#pragma unroll
  for (int h = 0; h < kMaxRep; ++h) {
    mref[h] = -INFINITY;
    lsum[h] = 0.f;
  }
  float o[16][4], mnacc[4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) o[nt][r] = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) mnacc[k] = 0.f;
  const float coef = a.qjl_coef, lscale = a.logit_scale;
  bool aborted = false;

  auto values_of = [&](int ti) {
    const int st = ti % STAGES;
    const uint32_t mask = valid[st];
    const float* pb = reinterpret_cast<const float*>(sm.ptr(OFF_PBUF + (ti & 1) * PBUF_BYTES));
#pragma unroll 1
    for (int q = warp; q < TILE_PAGES; q += NW)
      if (mask >> q & 1)
        page_values(sm.ptr(OFF_STAGE + st * STAGE_BYTES + q * PAGE_BYTES), pb + q * kPage, o, mnacc, lane);
  };

#pragma unroll 1
  for (int ti = 0; ti < ntiles; ++ti) {
    const int st = ti % STAGES;
    if (tid == 0 && ti > 0) tile_blocks(ti - 1 + STAGES, nblk);  // issued at the end of this iteration
    // ---- tile ti's pages in shared memory; key bits of token tid -> e4m3 bytes in tensor memory
    if (!mbar_wait(bar_full + 8 * st, (uint32_t)(ti / STAGES) & 1u)) atomicOr(abort_flag, 1u);
    {
      const uint8_t* T = sm.ptr(OFF_STAGE + st * STAGE_BYTES + (tid >> 4) * PAGE_BYTES);
      const int slot = tid & 15;
#pragma unroll
      for (int p = 0; p < 3; ++p) {
        const uint4 row = *reinterpret_cast<const uint4*>(T + 2 * D * p + slot * 16);
        uint32_t r[32];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t x = word_of(row, w);
#pragma unroll
          for (int j = 0; j < 8; ++j) r[8 * w + j] = key_bytes(x, j);
        }
        tm_st32(tmem + lane_base + TM_A + 32 * p, r);
      }
      tm_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    if (*reinterpret_cast<volatile uint32_t*>(abort_flag)) {
      aborted = true;
      break;
    }
    tc_fence_after();
    if (tid == 0) {
      if (ti == 0 && !mbar_wait(bar_q, 0)) atomicOr(abort_flag, 2u);
      const uint32_t qop = sm.addr(OFF_Q);
#pragma unroll
      for (int s = 0; s < NSLICE; ++s)
        mma_f8(tmem + (s < 8 ? TM_LM : TM_QJ), tmem + TM_A + 8 * s, sdesc(qop + s * SLICE_BYTES), s % 8 != 0);
      mma_commit(bar_mma);
    }
    // ---- meanwhile: the value product of the previous tile
    if (ti > 0) values_of(ti - 1);
    // ---- score epilogue of tile ti: thread = token
    if (ti == 0 && tid != 0 && !mbar_wait(bar_q, 0)) atomicOr(abort_flag, 2u);
    if (!mbar_wait(bar_mma, (uint32_t)ti & 1u)) atomicOr(abort_flag, 4u);
    tc_fence_after();
    float logit[kMaxRep];
    {
      const float* qs = reinterpret_cast<const float*>(sm.ptr(OFF_Q + QOP_BYTES));  // scale[2][8], off[2][8]
      float lm[kMaxRep], qj[kMaxRep];
#pragma unroll
      for (int set = 0; set < 2; ++set) {
        float v[QN];
        tm_ld48(tmem + lane_base + (set ? TM_QJ : TM_LM), v);
#pragma unroll
        for (int h = 0; h < kMaxRep; ++h) {
          float acc = v[NPIECE * h + NPIECE - 1];
#pragma unroll
          for (int pc = NPIECE - 2; pc >= 0; --pc) acc = fmaf(acc, 0.0625f, v[NPIECE * h + pc]);
          const float r = fmaf(acc, qs[set * kMaxRep + h], qs[2 * kMaxRep + set * kMaxRep + h]);
          if (set == 0)
            lm[h] = r;
          else
            qj[h] = r;
        }
      }
      const uint8_t* T = sm.ptr(OFF_STAGE + st * STAGE_BYTES + (tid >> 4) * PAGE_BYTES);
      const int slot = tid & 15;
      const float nk = __half2float(*reinterpret_cast<const __half*>(T + O_NORM + 2 * slot));
      const float nr = __half2float(*reinterpret_cast<const __half*>(T + O_NORM + 32 + 2 * slot));
      const bool ok = valid[st] >> (tid >> 4) & 1;
      const float cnr = coef * nr, nks = nk * lscale;
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) logit[h] = (ok && h < a.nrg) ? nks * fmaf(cnr, qj[h], lm[h]) : -INFINITY;
    }
    // lazy reference update: only when a logit passes its reference by more than 2^kLazyLog2
    int exceed = 0;
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) exceed |= logit[h] > mref[h] + kLazyLog2;
    tc_fence_before();
    if (__syncthreads_or(exceed)) {
      float* wred = reinterpret_cast<float*>(sm.ptr(OFF_WRED));
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) {
        const float m = warp_max(logit[h]);
        if (lane == 0) wred[warp * kMaxRep + h] = m;
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) {
        float m = mref[h];
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2) m = fmaxf(m, wred[w2 * kMaxRep + h]);
        // 0 on a head's first update (reference -inf); 1 while the head has no valid token
        const float alpha = m == -INFINITY ? 1.f : fast_exp2(mref[h] - m);
        mref[h] = m;
        lsum[h] *= alpha;
        // this warp's value state: lane (g, t) holds head g's rows
        if ((lane >> 2) == h) {
#pragma unroll
          for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) o[nt][r] *= alpha;
#pragma unroll
          for (int k = 0; k < 4; ++k) mnacc[k] *= alpha;
        }
      }
    }
    {
      float* pb = reinterpret_cast<float*>(sm.ptr(OFF_PBUF + (ti & 1) * PBUF_BYTES));
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) {
        const float p = logit[h] == -INFINITY ? 0.f : fast_exp2(logit[h] - mref[h]);
        lsum[h] += p;
        pb[h * TILE_TOK + tid] = p;
      }
    }
    __syncthreads();  // p of tile ti visible; tile ti-1's stage and values done by every warp
    if (*reinterpret_cast<volatile uint32_t*>(abort_flag)) {
      aborted = true;
      break;
    }
    if (tid == 0 && ti > 0 && ti - 1 + STAGES < ntiles) issue_tile(ti - 1 + STAGES, nblk);
  }
  if (!aborted && ntiles > 0) values_of(ntiles - 1);

  if (aborted) {
    if (tid == 0) {
      flag_error(a.err, TQ_DEVERR_TIMEOUT);
      // drain: the copies of the last tile issued into each stage complete (bounded) before the
      // shared memory is released
      for (int ti = max(0, issued - STAGES); ti < issued; ++ti)
        mbar_wait(bar_full + 8 * (ti % STAGES), (uint32_t)(ti / STAGES) & 1u);
    }
  }
  // the tensor memory is free once the last MMA has been waited for (or the wait gave up)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(TM_COLS) : "memory");
  if (aborted) return;

  // ---- combine: normalisers over the CTA's tokens, value accumulators over its warps
  float* wred = reinterpret_cast<float*>(sm.ptr(OFF_WRED));
#pragma unroll
  for (int h = 0; h < kMaxRep; ++h) {
    const float s = warp_sum(lsum[h]);
    if (lane == 0) wred[warp * kMaxRep + h] = s;
  }
  const int g = lane >> 2, t = lane & 3;
  float mn[4];
#pragma unroll
  for (int gg = 0; gg < 4; ++gg) {
    mn[gg] = mnacc[gg];
    mn[gg] += __shfl_xor_sync(kFull, mn[gg], 1);
    mn[gg] += __shfl_xor_sync(kFull, mn[gg], 2);
  }
  float* wo = reinterpret_cast<float*>(sm.ptr(OFF_STAGE));  // [NW][kMaxRep][D]; stages are idle
  constexpr float vscale = 4.f / kWeightScale;             // codes 1 + q/4, weights p s 2^-kLazyLog2
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e)
      wo[((size_t)warp * kMaxRep + g) * D + nt * 8 + 2 * t + e] =
          fmaf(o[nt][2 + e], kLoUnscale, o[nt][e]) * vscale + mn[nt >> 2];
  __syncthreads();
  const bool direct = nparts == 1;
  for (int i = tid; i < a.nrg * D; i += NW * 32) {
    const int h = i / D, dim = i % D;
    const float den = (wred[h] + wred[kMaxRep + h]) + (wred[2 * kMaxRep + h] + wred[3 * kMaxRep + h]);
    float num = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < NW; ++w2) num += wo[((size_t)w2 * kMaxRep + h) * D + dim];
    if (direct) {
      a.out[((size_t)b * a.hq + h0 + h) * D + dim] = den > 0.f ? num / den : 0.f;
    } else {
      float* dst = a.parts + (((size_t)b * a.hq + h0 + h) * a.n_parts + part) * (D + 4);
      dst[dim] = num;
      if (dim == 0) {
        dst[D] = mref[h];
        dst[D + 1] = den;
      }
    }
  }
}

}  // namespace

bool hy_supported(const tq_ctx* ctx) {
  return ctx->cfg.layout == TQ_LAYOUT_MAIN && ctx->cfg.head_dim == D && ctx->cfg.key_bits == 3 &&
         ctx->cfg.value_bits == 2 && ctx->cfg.qjl_m == D;
}

cudaError_t launch_decode_hy(tq_ctx* ctx, TcArgs& a, int batch, uint8_t* qrec, cudaStream_t s) {
  const int hgroups = a.hkv * a.groups;
  tc_set_score_constants(ctx, a);
  hy_prep_kernel<<<dim3(hgroups, batch), 128, 0, s>>>(a, qrec);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ctx->launches++;
  e = cudaFuncSetAttribute(hy_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, HY_SMEM);
  if (e != cudaSuccess) return e;
  ctx->decode_kernel = "hy_decode_kernel";
  prof_start(ctx, kProfDecode, s);
  hy_decode_kernel<<<dim3(a.n_parts, hgroups, batch), NW * 32, HY_SMEM, s>>>(a, qrec);
  prof_stop(ctx, kProfDecode, s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ctx->launches++;
  return launch_tc_merge(ctx, a, batch, s);
}

}  // namespace tq
