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
// CTA: one per SM with all 512 tensor-memory columns, its warps in roles joined by mbarriers (a
// page-copy lane, 4 score warps, an MMA-issue lane, 8 value warps; see hy_decode_kernel).
// Work split and merge: the chunks / ring item / split-K partials of decode_tc.cu, in a
// one-dimensional grid with the ring items last; the ring item runs the mma.sync path of
// decode_tc.cu on every warp.  Every wait on an mbarrier is bounded (about a second): on expiry the
// CTA flags TQ_DEVERR_TIMEOUT, waits for its own copies and MMAs, frees its tensor memory and
// leaves.
#include <cuda_fp8.h>

#include "tc_mma.cuh"

namespace tq {
namespace {

constexpr int D = kTcD;
// Warp roles of a CTA (one CTA per SM; it holds all 512 tensor-memory columns):
//   warps 0..3   score: token t = thread t of the tile; key bytes into tensor memory, epilogue
//   warp  4      producer: page copies into the stage ring
//   warp  5      MMA issue (one lane)
//   warps 6..13  value: warp 6 + v owns page v of every tile
constexpr int NSW = 4;                 // score warps
constexpr int NVW = 8;                 // value warps
constexpr int W_PROD = NSW, W_MMA = NSW + 1, W_VAL0 = NSW + 2;
constexpr int NWARPS = W_VAL0 + NVW;
constexpr int NTHREADS = 32 * NWARPS;
constexpr int NW = NSW;                // warps of the query-record kernel (hy_prep_kernel)
constexpr int TILE_PAGES = 8;          // pages per score tile: 128 tokens = M of the MMA
static_assert(TILE_PAGES == NVW, "one value warp per page of a tile");
constexpr int TILE_TOK = TILE_PAGES * kPage;
constexpr int STAGES = 8;              // tiles of pages in shared memory
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
// Tensor-memory columns, two buffers of each: key bytes (96), Lloyd-Max and QJL accumulators
// (48 each).
constexpr int TM_BUF = 192, TM_A = 0, TM_LM = 96, TM_QJ = 144, TM_COLS = 512;
// tcgen05 instruction descriptor: kind::f8f6f4, A = B = E4M3, D = F32, K-major, N = 48, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(QN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

// Dynamic shared memory (offsets from a 1024-byte aligned base).
constexpr int OFF_Q = 0;
constexpr int OFF_STAGE = QREC_BYTES;
constexpr int STAGE_BYTES = TILE_PAGES * PAGE_BYTES;
constexpr int OFF_PBUF = OFF_STAGE + STAGES * STAGE_BYTES;
constexpr int PBUF_BYTES = kMaxRep * TILE_TOK * 4;
constexpr int OFF_WO = OFF_PBUF + 2 * PBUF_BYTES;              // [NVW][kMaxRep][D] value results
constexpr int OFF_MISC = OFF_WO + NVW * kMaxRep * D * 4;
// mbarriers (8 bytes each)
constexpr int OFF_BAR_SFULL = OFF_MISC;                  // [STAGES] pages landed (producer, tx)
constexpr int OFF_BAR_SEMPTY = OFF_BAR_SFULL + 8 * STAGES;  // [STAGES] score + value warps done
constexpr int OFF_BAR_AFULL = OFF_BAR_SEMPTY + 8 * STAGES;  // [2] key bytes in tensor memory
constexpr int OFF_BAR_DFULL = OFF_BAR_AFULL + 16;           // [2] score MMAs complete
constexpr int OFF_BAR_PFULL = OFF_BAR_DFULL + 16;           // [2] p of a tile written
constexpr int OFF_BAR_PEMPTY = OFF_BAR_PFULL + 16;          // [2] value warps done with p
constexpr int OFF_BAR_Q = OFF_BAR_PEMPTY + 16;              // query record landed
constexpr int OFF_TMEM = OFF_BAR_Q + 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int OFF_VALID = OFF_ABORT + 4;                    // [STAGES] valid-page masks
constexpr int OFF_ALPHA = OFF_VALID + 4 * STAGES;           // [2][kMaxRep + 1] rescale factors, flag
constexpr int OFF_WRED = OFF_ALPHA + 4 * 2 * (kMaxRep + 1) + 8;  // [NWARPS][kMaxRep] floats
constexpr int OFF_WRED2 = OFF_WRED + 4 * NWARPS * kMaxRep;
constexpr int OFF_MFIN = OFF_WRED2 + 4 * NWARPS * kMaxRep;  // [kMaxRep] final reference maxima
constexpr int MISC_BYTES = OFF_MFIN + 4 * kMaxRep - OFF_MISC;
constexpr int SMEM_USED = OFF_MISC + MISC_BYTES;
constexpr int HY_SMEM = SMEM_USED + 1024;
// The ring item combines its warps' results in the (idle) stage ring.
static_assert((size_t)NWARPS * kMaxRep * D * sizeof(float) <= (size_t)STAGES * STAGE_BYTES, "combine buffer fits");
// More than half of an SM's shared memory: one CTA per SM, so that the CTA's 512 tensor-memory
// columns are always free when it allocates them.
static_assert(HY_SMEM > 116 * 1024 && HY_SMEM <= 227 * 1024, "one CTA per SM");
static_assert(OFF_STAGE % 16 == 0 && OFF_PBUF % 16 == 0 && OFF_MISC % 16 == 0, "alignment");
static_assert(OFF_BAR_SFULL % 8 == 0 && OFF_BAR_Q % 8 == 0, "mbarrier alignment");

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
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Named barrier 1 over the score warps: the OR of v over their threads (ordering their shared
// memory accesses like bar.sync).
__device__ __forceinline__ bool score_any(bool v) {
  uint32_t r;
  asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, 1, %2, p; selp.u32 %0, 1, 0, q; }"
               : "=r"(r)
               : "r"((uint32_t)v), "n"(NSW * 32)
               : "memory");
  return r != 0;
}
__device__ __forceinline__ void score_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NSW * 32) : "memory"); }

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

// The ring item (exact fp16 buffer): the mma.sync path of decode_tc.cu on every warp of the CTA,
// per-warp softmax states combined at the end.
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
  for (int t0 = warp * 16; t0 < nb; t0 += NWARPS * 16) page_ring(a, Aq, rk, rv, t0, min(16, nb - t0), st, lane);
  float l = st.l;
  l += __shfl_xor_sync(kFull, l, 1);
  l += __shfl_xor_sync(kFull, l, 2);
  float* wo = reinterpret_cast<float*>(sm.ptr(OFF_STAGE));  // [NWARPS][kMaxRep][D]
  float* wm = reinterpret_cast<float*>(sm.ptr(OFF_WRED));   // [NWARPS][kMaxRep]
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
  for (int i = tid; i < a.nrg * D; i += NTHREADS) {
    const int h = i / D, dim = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < NWARPS; ++w2) M = fmaxf(M, wm[w2 * kMaxRep + h]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < NWARPS; ++w2) {
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

// Pipeline of a compressed chunk, in tiles of 128 tokens (8 pages).  Producer: tile i's pages into
// stage i mod STAGES.  Score warps: tile i's key bits into key-byte buffer i mod 2 of tensor memory
// (a_full), then the epilogue of tile i - 1 (d_full): logits, the lazy reference update, p and the
// rescale factors into p buffer (i - 1) mod 2 (p_full).  MMA lane: the 12 score MMAs of tile i into
// accumulator buffer i mod 2 (d_full).  Value warps: page v of tile j once its p is written; they
// release the p buffer (p_empty) and, with the score warps, the stage (s_empty).
__global__ void __launch_bounds__(NTHREADS, 1) hy_decode_kernel(TcArgs a, const uint8_t* qrec, int batch) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  {
    const uint32_t s0 = smem_u32(smem_raw);
    const uint32_t al = (s0 + 1023u) & ~1023u;
    sm.base = smem_raw + (al - s0);
    sm.base_s = al;
  }
  // One-dimensional grid: every (sequence, head group)'s chunks first, then the ring items, so the
  // short ring CTAs take whatever SMs the chunks leave and never hold a chunk back a wave.
  const int hgroups = a.hkv * a.groups;
  const int nchunk_ctas = a.n_chunks * batch * hgroups;
  const int id = blockIdx.x;
  const int part = id < nchunk_ctas ? id % a.n_chunks : a.n_chunks;
  const int item = id < nchunk_ctas ? id / a.n_chunks : id - nchunk_ctas;  // (sequence, head group)
  const int hg = item % hgroups, b = item / hgroups;
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
  float* alpha_s = reinterpret_cast<float*>(sm.ptr(OFF_ALPHA));  // [2][kMaxRep + 1]: factors, flag
  float* wred = reinterpret_cast<float*>(sm.ptr(OFF_WRED));
  float* wl = reinterpret_cast<float*>(sm.ptr(OFF_WRED2));
  float* mfin = reinterpret_cast<float*>(sm.ptr(OFF_MFIN));
  float* wo = reinterpret_cast<float*>(sm.ptr(OFF_WO));
  const uint32_t bar_sfull = sm.addr(OFF_BAR_SFULL), bar_sempty = sm.addr(OFF_BAR_SEMPTY);
  const uint32_t bar_afull = sm.addr(OFF_BAR_AFULL), bar_dfull = sm.addr(OFF_BAR_DFULL);
  const uint32_t bar_pfull = sm.addr(OFF_BAR_PFULL), bar_pempty = sm.addr(OFF_BAR_PEMPTY);
  const uint32_t bar_q = sm.addr(OFF_BAR_Q);
  auto stage = [&](int st) { return sm.ptr(OFF_STAGE + st * STAGE_BYTES); };

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sm.addr(OFF_TMEM)),
                 "n"(TM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == W_PROD * 32) {
    *abort_flag = 0;
#pragma unroll
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(bar_sfull + 8 * st, 1);
      mbar_init(bar_sempty + 8 * st, NSW + NVW);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar_afull + 8 * k, NSW * 32);
      mbar_init(bar_dfull + 8 * k, 1);
      mbar_init(bar_pfull + 8 * k, NSW * 32);
      mbar_init(bar_pempty + 8 * k, NVW);
    }
    mbar_init(bar_q, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_expect_tx(bar_q, QREC_BYTES);
    bulk_g2s(sm.addr(OFF_Q), qrec + ((size_t)b * a.hkv * a.groups + hg) * QREC_BYTES, QREC_BYTES, bar_q);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm.ptr(OFF_TMEM));
  bool bad = false;  // a bounded wait of this thread expired

  if (warp < NSW) {
    // ================================================================ score warps: thread = token
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float* qs = reinterpret_cast<const float*>(sm.ptr(OFF_Q + QOP_BYTES));  // scale[2][8], off[2][8]
    const float coef = a.qjl_coef, lscale = a.logit_scale;
    float mref[kMaxRep], lsum[kMaxRep];
#pragma unroll
    for (int h = 0; h < kMaxRep; ++h) {
      mref[h] = -INFINITY;
      lsum[h] = 0.f;
    }
    bool stop = false;
#pragma unroll 1
    for (int i = 0; i <= ntiles; ++i) {
      if (i < ntiles) {
        // key bits of token tid of tile i -> e4m3 bytes in key-byte buffer i mod 2
        const int st = i % STAGES;
        bad |= !mbar_wait(bar_sfull + 8 * st, (uint32_t)(i / STAGES) & 1u);
        const uint8_t* T = stage(st) + (tid >> 4) * PAGE_BYTES;
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
          tm_st32(tmem + lane_base + (i & 1) * TM_BUF + TM_A + 32 * p, r);
        }
        tm_wait_st();
        tc_fence_before();
        mbar_arrive(bar_afull + 8 * (i & 1));
      }
      if (i == 0) continue;
      // ---- epilogue of tile j = i - 1
      const int j = i - 1, st = j % STAGES, buf = j & 1;
      if (j == 0) bad |= !mbar_wait(bar_q, 0);
      bad |= !mbar_wait(bar_dfull + 8 * buf, (uint32_t)(j >> 1) & 1u);
      tc_fence_after();
      float logit[kMaxRep];
      {
        float lm[kMaxRep], qj[kMaxRep];
#pragma unroll
        for (int set = 0; set < 2; ++set) {
          float v[QN];
          tm_ld48(tmem + lane_base + buf * TM_BUF + (set ? TM_QJ : TM_LM), v);
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
        const uint8_t* T = stage(st) + (tid >> 4) * PAGE_BYTES;
        const int slot = tid & 15;
        const float nk = __half2float(*reinterpret_cast<const __half*>(T + O_NORM + 2 * slot));
        const float nr = __half2float(*reinterpret_cast<const __half*>(T + O_NORM + 32 + 2 * slot));
        const bool ok = valid[st] >> (tid >> 4) & 1;
        const float cnr = coef * nr, nks = nk * lscale;
#pragma unroll
        for (int h = 0; h < kMaxRep; ++h) logit[h] = (ok && h < a.nrg) ? nks * fmaf(cnr, qj[h], lm[h]) : -INFINITY;
      }
      // p buffer j mod 2 and its rescale factors are free once the value warps are done with tile j - 2
      if (j >= 2) bad |= !mbar_wait(bar_pempty + 8 * buf, (uint32_t)((j >> 1) - 1) & 1u);
      bad |= *reinterpret_cast<volatile uint32_t*>(abort_flag) != 0;
      // lazy reference update: only when a logit passes its reference by more than 2^kLazyLog2;
      // the same vote carries the abort decision, so the four warps always leave together
      int exceed = 0;
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) exceed |= logit[h] > mref[h] + kLazyLog2;
      float* al = alpha_s + buf * (kMaxRep + 1);
      if (score_any(exceed || bad)) {
        if (score_any(bad)) {
          stop = true;
          break;
        }
#pragma unroll
        for (int h = 0; h < kMaxRep; ++h) {
          const float m = warp_max(logit[h]);
          if (lane == 0) wred[warp * kMaxRep + h] = m;
        }
        score_sync();
#pragma unroll
        for (int h = 0; h < kMaxRep; ++h) {
          float m = mref[h];
#pragma unroll
          for (int w2 = 0; w2 < NSW; ++w2) m = fmaxf(m, wred[w2 * kMaxRep + h]);
          // 0 on a head's first update (reference -inf); 1 while the head has no valid token
          const float alpha = m == -INFINITY ? 1.f : fast_exp2(mref[h] - m);
          mref[h] = m;
          lsum[h] *= alpha;
          if (tid == 0) al[h] = alpha;
        }
        if (tid == 0) al[kMaxRep] = 1.f;
      } else if (tid == 0) {
        al[kMaxRep] = 0.f;
      }
      float* pb = reinterpret_cast<float*>(sm.ptr(OFF_PBUF + buf * PBUF_BYTES));
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) {
        const float p = logit[h] == -INFINITY ? 0.f : fast_exp2(logit[h] - mref[h]);
        lsum[h] += p;
        pb[h * TILE_TOK + tid] = p;
      }
      mbar_arrive(bar_pfull + 8 * buf);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sempty + 8 * st);
    }
    if (stop) {
      if (tid == 0) atomicOr(abort_flag, 1u);
    } else {
      // this CTA's normalisers (in their own array: another score warp may still read the maxima
      // of the last update) and reference maxima
#pragma unroll
      for (int h = 0; h < kMaxRep; ++h) {
        const float s = warp_sum(lsum[h]);
        if (lane == 0) wl[warp * kMaxRep + h] = s;
        if (tid == 0) mfin[h] = mref[h];
      }
    }
  } else if (warp == W_PROD) {
    // ================================================================ producer
    if (lane == 0) {
      int issued = 0;
      int blk[TILE_PAGES];  // block ids of the next tile (-1 past the chunk), read one tile ahead
      auto tile_blocks = [&](int ti) {
        const int p0 = ti * TILE_PAGES, np = min(TILE_PAGES, npg - p0);
#pragma unroll
        for (int q = 0; q < TILE_PAGES; ++q) blk[q] = q < np ? __ldg(btb + p0 + q) : -1;
      };
      tile_blocks(0);
#pragma unroll 1
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % STAGES;
        if (i >= STAGES && !mbar_wait(bar_sempty + 8 * st, (uint32_t)(i / STAGES - 1) & 1u)) {
          bad = true;
          break;
        }
        uint32_t mask = 0, bytes = 0;
#pragma unroll
        for (int q = 0; q < TILE_PAGES; ++q) {
          if (blk[q] >= 0 && blk[q] < a.num_blocks) {
            mask |= 1u << q;
            bytes += PAGE_BYTES;
          } else if (q < min(TILE_PAGES, npg - i * TILE_PAGES)) {
            flag_error(a.err, TQ_DEVERR_BLOCK_ID);
          }
        }
        valid[st] = mask;
        mbar_expect_tx(bar_sfull + 8 * st, bytes);
#pragma unroll
        for (int q = 0; q < TILE_PAGES; ++q)
          if (mask >> q & 1)
            bulk_g2s(sm.addr(OFF_STAGE + st * STAGE_BYTES + q * PAGE_BYTES),
                     a.pool + ((size_t)blk[q] * a.hkv + kvh) * PAGE_BYTES, PAGE_BYTES, bar_sfull + 8 * st);
        issued = i + 1;
        if (i + 1 < ntiles) tile_blocks(i + 1);
        if (*reinterpret_cast<volatile uint32_t*>(abort_flag)) break;
      }
      if (bad) atomicOr(abort_flag, 1u);
      // the copies of the last tile issued into each stage land before the CTA leaves (every earlier
      // tile was consumed, which needed its copies)
      for (int i = max(0, issued - STAGES); i < issued; ++i)
        mbar_wait(bar_sfull + 8 * (i % STAGES), (uint32_t)(i / STAGES) & 1u);
    }
  } else if (warp == W_MMA) {
    // ================================================================ MMA issue
    if (lane == 0) {
      int last = -1;
      bad = !mbar_wait(bar_q, 0);
      const uint32_t qop = sm.addr(OFF_Q);
#pragma unroll 1
      for (int i = 0; i < ntiles && !bad; ++i) {
        const int buf = i & 1;
        if (!mbar_wait(bar_afull + 8 * buf, (uint32_t)(i >> 1) & 1u)) {
          bad = true;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * TM_BUF;
#pragma unroll
        for (int s = 0; s < NSLICE; ++s)
          mma_f8(d + (s < 8 ? TM_LM : TM_QJ), d + TM_A + 8 * s, sdesc(qop + s * SLICE_BYTES), s % 8 != 0);
        mma_commit(bar_dfull + 8 * buf);
        last = i;
      }
      if (bad) atomicOr(abort_flag, 1u);
      // the tensor memory is released only after the last MMA has completed
      if (last >= 0) mbar_wait(bar_dfull + 8 * (last & 1), (uint32_t)(last >> 1) & 1u);
    }
  } else {
    // ================================================================ value warps: page v of each tile
    const int v = warp - W_VAL0;
    const int g = lane >> 2, t = lane & 3;
    float o[16][4], mnacc[4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) o[nt][r] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) mnacc[k] = 0.f;
#pragma unroll 1
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % STAGES, buf = j & 1;
      bool ok = mbar_wait(bar_sfull + 8 * st, (uint32_t)(j / STAGES) & 1u);
      ok = ok && mbar_wait(bar_pfull + 8 * buf, (uint32_t)(j >> 1) & 1u);
      if (!__all_sync(kFull, ok)) {
        bad = true;
        break;
      }
      const float* al = alpha_s + buf * (kMaxRep + 1);
      if (al[kMaxRep] != 0.f) {
        const float f = al[g];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) o[nt][r] *= f;
#pragma unroll
        for (int k = 0; k < 4; ++k) mnacc[k] *= f;
      }
      if (valid[st] >> v & 1)
        page_values(stage(st) + v * PAGE_BYTES, reinterpret_cast<const float*>(sm.ptr(OFF_PBUF + buf * PBUF_BYTES)) +
                                                    v * kPage,
                    o, mnacc, lane);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_pempty + 8 * buf);
        mbar_arrive(bar_sempty + 8 * st);
      }
    }
    if (bad && lane == 0) atomicOr(abort_flag, 1u);
    float mn[4];
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) {
      mn[gg] = mnacc[gg];
      mn[gg] += __shfl_xor_sync(kFull, mn[gg], 1);
      mn[gg] += __shfl_xor_sync(kFull, mn[gg], 2);
    }
    constexpr float vscale = 4.f / kWeightScale;  // codes 1 + q/4, weights p s 2^-kLazyLog2
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        wo[((size_t)v * kMaxRep + g) * D + nt * 8 + 2 * t + e] =
            fmaf(o[nt][2 + e], kLoUnscale, o[nt][e]) * vscale + mn[nt >> 2];
  }

  // every role is done: MMAs complete, copies landed, tensor memory read
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(TM_COLS) : "memory");
  if (*reinterpret_cast<volatile uint32_t*>(abort_flag)) {
    if (tid == 0) flag_error(a.err, TQ_DEVERR_TIMEOUT);
    return;
  }

  // ---- combine: normalisers over the score warps, value results over the value warps
  const bool direct = nparts == 1;
  for (int i = tid; i < a.nrg * D; i += NTHREADS) {
    const int h = i / D, dim = i % D;
    const float den = (wl[h] + wl[kMaxRep + h]) + (wl[2 * kMaxRep + h] + wl[3 * kMaxRep + h]);
    float num = 0.f;
#pragma unroll
    for (int v = 0; v < NVW; ++v) num += wo[((size_t)v * kMaxRep + h) * D + dim];
    if (direct) {
      a.out[((size_t)b * a.hq + h0 + h) * D + dim] = den > 0.f ? num / den : 0.f;
    } else {
      float* dst = a.parts + (((size_t)b * a.hq + h0 + h) * a.n_parts + part) * (D + 4);
      dst[dim] = num;
      if (dim == 0) {
        dst[D] = mfin[h];
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
  hy_decode_kernel<<<a.n_parts * hgroups * batch, NTHREADS, HY_SMEM, s>>>(a, qrec, batch);
  prof_stop(ctx, kProfDecode, s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ctx->launches++;
  return launch_tc_merge(ctx, a, batch, s);
}

}  // namespace tq
