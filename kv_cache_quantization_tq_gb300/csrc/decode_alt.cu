// Alternate-layout decode attention, one warp per page (block dots on the tensor cores).
//
// Keys are 8-, 5-, 4- or 2-bit affine codes per block of 32 (no rotation; the vllm-metal
// TurboQuant guide's q8_0 / q5_0 / q4_0 / uint2 key formats) or the fp16 keys themselves (the
// V-only cache of the "TurboQuant-MLX overview", usage paths), values are
// VB-bit (2, 3 or 4) Lloyd-Max indices of the rotated unit value with an fp16
// norm (vllm-metal TurboQuant guide, quantisation table: q2_0 .. q4_0 values).  With one query head per
// KV head the work per byte is small, so the kernel is written to stream the
// pages: each warp walks its own pages through a cp.async pipeline, lane l
// owns the E = d/32 consecutive dimensions [l E, l E + E):
//
//   logit_t = sum_b s_b <q_b, code_b> + mn_b sum(q_b)
//   The block dots <q_b, code_b> of a page are one small dense product on the
//   tensor cores (mma.sync m16n8k16): rows = the 16 tokens, k = coordinates,
//   columns = (query head, block of 32) with B holding q restricted to the
//   block.  8- and 4-bit codes enter as the exact fp16 value 1024 + code (one
//   byte-permute or two bit selects per pair), the 1024 sum(q_b) offset is
//   removed per block in fp32; 5- and 2-bit codes enter as 1 + code 2^-kb (the
//   code in the top mantissa bits), so only sum(q_b) is removed and the product
//   is scaled by 2^kb: with few levels, a 1024 offset would cancel most of the
//   fp32 accumulator's bits.  fp16 keys are the A operand as they are.  The key
//   rows are XOR-swizzled by 16-byte chunk as they are copied in, so the
//   fragment loads are free of bank conflicts.  Scores then move to lane
//   l = token l/2 for the softmax and value steps;
//   online softmax per head; v_rot += p_t n_v,t c[idx_t] in the rotated domain;
//   one inverse rotation per chunk ("TurboQuant-MLX overview", GPU kernel
//   section: butterfly pulled out of the value sum).
//
// Split-K partials use the same layout as the main-layout kernels
// ([d] values, max, sum; stride d + 2) and the same merge kernel.
#include "common.cuh"

namespace tq {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarps = 4;

struct AltArgs {
  const __half* q;
  const uint8_t* pool;
  int num_blocks;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* n_compressed;
  const __half* ring_k;
  const __half* ring_v;
  const int32_t* n_buf;
  int max_ctx;
  float* parts;
  int chunk_tokens, n_chunks, n_parts;
  int hq, hkv, n_rep, nrg, groups;
  const float* signs;
  CodeTables tab;
  int vb;              // value bits (read by the 5- to 8-bit instance)
  const float* vcent;  // the 2^vb value centroids (device)
  uint32_t* err;
};

__device__ __forceinline__ void cp16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

template <int D, int VB, int KB>
struct AltCfg {
  static constexpr int E = D / 32;      // dimensions per lane
  static constexpr int KEYB = alt_key_bytes(D, KB);  // KB-bit key codes and (scale, minimum), or fp16 keys
  static constexpr int TILE = alt_tile_bytes(D, KB, VB);
  static constexpr int STAGES = TILE <= 3200 ? 4 : (TILE <= 6400 ? 3 : 2);
  static constexpr size_t SMEM = (size_t)kWarps * STAGES * TILE;
};

// Whether n-tile j of the score product (columns 8j .. 8j+7 of NRG = heads x blocks) has a
// column of block blk (G blocks per head).
template <int G, int NRG>
__device__ constexpr bool tile_has_block(int j, int blk) {
  for (int c = 0; c < 8; ++c) {
    const int n = 8 * j + c;
    if (n < NRG && n % G == blk) return true;
  }
  return false;
}

// KB-bit key rows (KB = 8, 4, 2; KB D / 8 bytes, NCH = KB D / 128 chunks of 16 bytes): chunk c of
// row r sits at chunk c ^ kq_swizzle(r).  Rows whose starts share a 128-byte bank window get
// different XORs, so the fragment loads of rows g = 0..7 at one k-step fall in distinct banks
// (without it, nibble rows of 64 bytes are 4-way and 2-bit rows of 32 bytes 2-way conflicted).
template <int D, int KB>
__device__ __forceinline__ int kq_swizzle(int row) {
  constexpr int NCH = KB * D / 128;
  if (NCH <= 1) return 0;
  return NCH >= 8 ? (row & 7) : ((row * NCH) >> 3) & (NCH - 1);
}
// fp16 key rows (D/8 >= 8 chunks each): chunk c of row r sits at chunk c ^ 2 (r & 3).  A half-warp's
// 8-byte fragment loads (rows g..g+3, chunks 2 ks and 2 ks + 1) then land in 8 distinct chunk slots.
__device__ __forceinline__ int kh_swizzle(int row) { return 2 * (row & 3); }

// 4-bit key codes: the nibbles n0..n3 of w (coordinates 4t .. 4t+3) as the fp16 pairs
// (1024 + n0, 1024 + n1) and (1024 + n2, 1024 + n3).
__device__ __forceinline__ uint32_t nib_pair_lo(uint32_t w) { return (w & 0xFu) | ((w << 12) & 0xF0000u) | 0x64006400u; }
__device__ __forceinline__ uint32_t nib_pair_hi(uint32_t w) {
  return ((w >> 8) & 0xFu) | ((w << 4) & 0xF0000u) | 0x64006400u;
}

// 2-bit key codes: the four codes of w's low byte (coordinates 4t .. 4t+3) as the fp16 pairs
// (1 + c0/4, 1 + c1/4) and (1 + c2/4, 1 + c3/4).
__device__ __forceinline__ uint32_t q2_pair_lo(uint32_t w) {
  return ((w << 8) & 0x300u) | ((w << 22) & 0x3000000u) | 0x3C003C00u;
}
__device__ __forceinline__ uint32_t q2_pair_hi(uint32_t w) {
  return ((w << 4) & 0x300u) | ((w << 18) & 0x3000000u) | 0x3C003C00u;
}
// 5-bit key codes: the four codes in bits 0..19 of x as (1 + c0/32, 1 + c1/32) and
// (1 + c2/32, 1 + c3/32).
__device__ __forceinline__ uint32_t q5_pair_lo(uint32_t x) {
  return ((x << 5) & 0x3E0u) | ((x << 16) & 0x3E00000u) | 0x3C003C00u;
}
__device__ __forceinline__ uint32_t q5_pair_hi(uint32_t x) {
  return ((x >> 5) & 0x3E0u) | ((x << 6) & 0x3E00000u) | 0x3C003C00u;
}

// How KB-bit codes enter the score product: as offset + code / scale, so that
// sum(code q) = scale (dot - offset sum(q)).
template <int KB>
struct KeyEntry {
  static constexpr bool kBiased = KB == 8 || KB == 4;  // 1024 + code
  static constexpr float kOffset = kBiased ? 1024.f : 1.f;
  static constexpr float kScale = kBiased ? 1.f : (float)(1 << KB);
};

// VBT: the value bits (2, 3 or 4), or 0 for 5- to 8-bit values read from the arguments (one
// instance for the four widths: the stages are sized for 8 bits, the centroid table holds 256).
template <int D, int NR, int VBT, int KB>
__global__ void __launch_bounds__(128) decode_alt_v2_kernel(AltArgs a) {
  static_assert(KB == 16 || KB == 8 || KB == 5 || KB == 4 || KB == 2, "key widths");
  using C = AltCfg<D, VBT ? VBT : 8, KB>;  // staging for the widest values of the instance
  constexpr int NCMAX = 1 << (VBT ? VBT : 8);
  const int VB = VBT ? VBT : a.vb;
  const int tile = VBT ? C::TILE : alt_tile_bytes(D, KB, VB);  // bytes of a page in the pool
  const uint32_t vmask = (1u << VB) - 1u;
  constexpr int E = C::E;
  constexpr int G = D / 32;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float lut[NCMAX];
  __shared__ float wm[kWarps][NR], wl[kWarps][NR];
  __shared__ float wo[kWarps][NR][D];
  __shared__ int sblk[kWarps][C::STAGES];
  __shared__ float qsum_s[NR * G];
  __shared__ __align__(16) float wbuf[kWarps][16];  // this warp's token weights of the current head

  const int part = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int kvh = hg / a.groups;
  const int h0 = kvh * a.n_rep + (hg % a.groups) * a.nrg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int nc = a.n_compressed[b];
  if (nc < 0 || (nc & 15) || nc > a.max_blocks * kPage || nc > a.max_ctx) {
    if (tid == 0) flag_error(a.err, nc > a.max_ctx ? TQ_DEVERR_CHUNKS : TQ_DEVERR_POSITION);
    nc = 0;
  }
  const int tbeg = part * a.chunk_tokens;
  const int tend = min(nc, tbeg + a.chunk_tokens);
  if (tbeg >= tend) return;
  if (VBT == 0) {
    for (int i = tid; i < (1 << VB); i += blockDim.x) lut[i] = __ldg(a.vcent + i);
  } else if (tid < NCMAX) {
    float c = a.tab.c[0];
#pragma unroll
    for (int j = 1; j < NCMAX; ++j) c = tid == j ? a.tab.c[j] : c;
    lut[tid] = c;
  }

  // Score product: columns n = (head n / G, block n % G), NT n-tiles of 8.  Lane (g, t) holds
  // the B fragment of column 8j + g for the two k-steps of its block (k-step ks covers block
  // ks / 2; within a k-step, k = 2t + u is coordinate 4t + u and k = 2t + 8 + u is 4t + 2 + u).
  constexpr int NT = (NR * G + 7) / 8;
  const int g = lane >> 2, t = lane & 3;
  uint32_t bq[NT][2][2];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int n = 8 * j + g, hh = n / G, blk = n % G;
    const bool valid = n < NR * G && hh < a.nrg;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t* qw = reinterpret_cast<const uint32_t*>(a.q + ((size_t)b * a.hq + h0 + (valid ? hh : 0)) * D +
                                                             16 * (2 * blk + u) + 4 * t);
      bq[j][u][0] = valid ? qw[0] : 0u;
      bq[j][u][1] = valid ? qw[1] : 0u;
    }
  }
  // sum of q over each (head, block), for the C columns 8j + 2t + u this lane holds
  for (int idx = warp; idx < NR * G; idx += kWarps) {
    const int hh = idx / G, blk = idx % G;
    float v = hh < a.nrg ? __half2float(a.q[((size_t)b * a.hq + h0 + hh) * D + 32 * blk + lane]) : 0.f;
    v = warp_sum(v);
    if (lane == 0) qsum_s[idx] = v;
  }
  float m_run[NR], l_run[NR], acc[NR][E];
#pragma unroll
  for (int h = 0; h < NR; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[h][e] = 0.f;
  }
  __syncthreads();  // lut, qsum_s
  float qsc[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int n = 8 * j + 2 * t + u;
      qsc[j][u] = n < NR * G ? qsum_s[n] : 0.f;
    }

  const float scale = kLog2e / sqrtf((float)D);
  const int pbeg = tbeg >> 4;
  const int npg = (tend >> 4) - pbeg;
  const int nw = npg > warp ? (npg - warp + kWarps - 1) / kWarps : 0;
  uint8_t* wst = smem + (size_t)warp * C::STAGES * C::TILE;
  const int32_t* btb = a.block_table + (size_t)b * a.max_blocks;
  // block id of the next page to copy read one page ahead; ids of pages in flight per warp
  auto blk_of = [&](int k) { return k < nw ? __ldg(btb + pbeg + warp + kWarps * k) : -1; };
  auto issue = [&](int k, int blk) {
    if (k < nw) {
      if (lane == 0) sblk[warp][k % C::STAGES] = blk;
      if (blk >= 0 && blk < a.num_blocks) {
        const uint8_t* src = a.pool + ((size_t)blk * a.hkv + kvh) * tile;
        uint8_t* dst = wst + (k % C::STAGES) * C::TILE;
        for (int c = lane; c < tile / 16; c += 32) {
          int cd = c;
          if ((KB == 8 || KB == 4 || KB == 2) && c < KB * D / 8) {  // key rows: 16 x KB D / 128 chunks
            constexpr int NCH = KB * D / 128 > 0 ? KB * D / 128 : 1;
            const int row = c / NCH, ch = c % NCH;
            cd = row * NCH + (ch ^ kq_swizzle<D, KB>(row));
          } else if (KB == 16 && c < 2 * D) {  // fp16 key rows: 16 rows x D/8 chunks, swizzled
            const int row = c / (D / 8), ch = c % (D / 8);
            cd = row * (D / 8) + (ch ^ kh_swizzle(row));
          }
          cp16(dst + cd * 16, src + c * 16);
        }
      }
    }
    cp_commit();
  };
#pragma unroll
  for (int k = 0; k < C::STAGES - 1; ++k) issue(k, blk_of(k));
  int nxt = blk_of(C::STAGES - 1);
  for (int k = 0; k < nw; ++k) {
    __syncwarp();  // every lane is done with the slot and stage that are refilled next
    const int cur = nxt;
    nxt = blk_of(k + C::STAGES);
    issue(k + C::STAGES - 1, cur);
    cp_wait<C::STAGES - 1>();
    __syncwarp();
    const int blk = sblk[warp][k % C::STAGES];
    if (blk < 0 || blk >= a.num_blocks) {
      if (lane == 0) flag_error(a.err, TQ_DEVERR_BLOCK_ID);
      continue;
    }
    const uint8_t* T = wst + (k % C::STAGES) * C::TILE;
    const __half2* ksm2 = reinterpret_cast<const __half2*>(T + 2 * KB * D);  // not read for fp16 keys
    const uint32_t* vi = reinterpret_cast<const uint32_t*>(T + C::KEYB);
    const __half* vn = reinterpret_cast<const __half*>(T + C::KEYB + 2 * VB * D);
    // C[token][column] = sum over the column's block of (1024 + code) q_head
    float cacc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) cacc[j][r] = 0.f;
    {
      const uint32_t* w0r = reinterpret_cast<const uint32_t*>(T + g * (KB * D / 8));  // 5-bit rows
      const uint32_t* w1r = reinterpret_cast<const uint32_t*>(T + (g + 8) * (KB * D / 8));
      const uint8_t* rb0 = T + g * (KB * D / 8);  // row starts (chunks swizzled for KB = 8, 4, 2)
      const uint8_t* rb1 = T + (g + 8) * (KB * D / 8);
      const int sw0 = kq_swizzle<D, KB>(g), sw1 = kq_swizzle<D, KB>(g + 8);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint4 A;
        if (KB == 16) {  // coordinates 16 ks + 4t .. + 3: 8 bytes of chunk 2 ks + t/2 (swizzled)
          const int ch = 2 * ks + (t >> 1);
          const uint2 k0 = *reinterpret_cast<const uint2*>(T + g * (2 * D) + 16 * (ch ^ kh_swizzle(g)) + 8 * (t & 1));
          const uint2 k1 =
              *reinterpret_cast<const uint2*>(T + (g + 8) * (2 * D) + 16 * (ch ^ kh_swizzle(g + 8)) + 8 * (t & 1));
          A.x = k0.x;
          A.y = k1.x;
          A.z = k0.y;
          A.w = k1.y;
        } else if (KB == 8) {
          // byte 16 ks + 4t of the row: chunk ks, byte 4t within it
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(rb0 + 16 * (ks ^ sw0) + 4 * t);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(rb1 + 16 * (ks ^ sw1) + 4 * t);
          A.x = __byte_perm(w0, 0x64646464u, 0x4140u);  // row g: coordinates 4t, 4t+1 as 1024 + code
          A.y = __byte_perm(w1, 0x64646464u, 0x4140u);  // row g + 8
          A.z = __byte_perm(w0, 0x64646464u, 0x4342u);  // row g: coordinates 4t+2, 4t+3
          A.w = __byte_perm(w1, 0x64646464u, 0x4342u);
        } else if (KB == 4) {  // the four codes of coordinates 16 ks + 4t .. + 3 are 16 bits of the row
          // byte 8 ks + 2t of the row: chunk ks / 2, byte 8 (ks & 1) + 2t within it
          const uint32_t w0 = *reinterpret_cast<const uint16_t*>(rb0 + 16 * ((ks >> 1) ^ sw0) + 8 * (ks & 1) + 2 * t);
          const uint32_t w1 = *reinterpret_cast<const uint16_t*>(rb1 + 16 * ((ks >> 1) ^ sw1) + 8 * (ks & 1) + 2 * t);
          A.x = nib_pair_lo(w0);
          A.y = nib_pair_lo(w1);
          A.z = nib_pair_hi(w0);
          A.w = nib_pair_hi(w1);
        } else if (KB == 2) {  // ... 8 bits of the row
          // byte 4 ks + t of the row: chunk ks / 4, byte 4 (ks & 3) + t within it
          const uint32_t w0 = rb0[16 * ((ks >> 2) ^ sw0) + 4 * (ks & 3) + t];
          const uint32_t w1 = rb1[16 * ((ks >> 2) ^ sw1) + 4 * (ks & 3) + t];
          A.x = q2_pair_lo(w0);
          A.y = q2_pair_lo(w1);
          A.z = q2_pair_hi(w0);
          A.w = q2_pair_hi(w1);
        } else {  // 5 bits: 20 bits of the row from bit 80 ks + 20 t, across at most two words
          const int bit = 80 * ks + 20 * t, wi = bit >> 5, sh = bit & 31;
          const bool two = sh + 20 > 32;
          const uint32_t x0 = __funnelshift_r(w0r[wi], two ? w0r[wi + 1] : 0u, sh);
          const uint32_t x1 = __funnelshift_r(w1r[wi], two ? w1r[wi + 1] : 0u, sh);
          A.x = q5_pair_lo(x0);
          A.y = q5_pair_lo(x1);
          A.z = q5_pair_hi(x0);
          A.w = q5_pair_hi(x1);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if (tile_has_block<G, NR * G>(j, ks / 2)) {
            const bool mine = (8 * j + g) % G == ks / 2;
            mma_f16(cacc[j], A, mine ? bq[j][ks & 1][0] : 0u, mine ? bq[j][ks & 1][1] : 0u);
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < NR; ++h) {
      if (h >= a.nrg) break;
      float p0 = 0.f, p1 = 0.f;  // tokens g and g + 8
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int n = 8 * j + 2 * t + u;
          if (n < NR * G && n / G == h && KB == 16) {  // the block dots of fp16 keys are the score
            p0 += cacc[j][u];
            p1 += cacc[j][2 + u];
          } else if (n < NR * G && n / G == h) {
            const int blk = n % G;
            const float2 s0 = __half22float2(ksm2[g * G + blk]);
            const float2 s1 = __half22float2(ksm2[(g + 8) * G + blk]);
            const float qb = qsc[j][u];
            using KE = KeyEntry<KB>;
            const float sc0 = KE::kBiased ? s0.x : s0.x * KE::kScale;
            const float sc1 = KE::kBiased ? s1.x : s1.x * KE::kScale;
            p0 = fmaf(sc0, fmaf(-KE::kOffset, qb, cacc[j][u]), fmaf(s0.y, qb, p0));
            p1 = fmaf(sc1, fmaf(-KE::kOffset, qb, cacc[j][2 + u]), fmaf(s1.y, qb, p1));
          }
        }
      p0 += __shfl_xor_sync(kFull, p0, 1);
      p0 += __shfl_xor_sync(kFull, p0, 2);
      p1 += __shfl_xor_sync(kFull, p1, 1);
      p1 += __shfl_xor_sync(kFull, p1, 2);
      const int src = 4 * ((lane >> 1) & 7);
      const float a0 = __shfl_sync(kFull, p0, src), a1 = __shfl_sync(kFull, p1, src);
      const float s_tok = (lane < 16 ? a0 : a1) * scale;  // token lane/2
      float mx = s_tok;
#pragma unroll
      for (int o = 16; o >= 2; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      const float m_new = fmaxf(m_run[h], mx);
      const float alpha = fast_exp2(m_run[h] - m_new);
      const float p = fast_exp2(s_tok - m_new);
      float ps = (lane & 1) ? 0.f : p;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) ps += __shfl_xor_sync(kFull, ps, o);
      l_run[h] = l_run[h] * alpha + ps;
      m_run[h] = m_new;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[h][e] *= alpha;
      const float w = p * __half2float(vn[lane >> 1]);
      // the 16 token weights to every lane: at d <= 128 stored once (even lanes) and read back as
      // four broadcast 16-byte loads (measured: +3% at d = 64, no change at 128); at larger d by
      // one shuffle per token (the staged form measured 2% slower at d = 512)
      constexpr bool kStagedW = E <= 4;
      float wts[16];
      if constexpr (kStagedW) {
        if ((lane & 1) == 0) wbuf[warp][lane >> 1] = w;
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 w4 = reinterpret_cast<const float4*>(wbuf[warp])[k];
          wts[4 * k] = w4.x;
          wts[4 * k + 1] = w4.y;
          wts[4 * k + 2] = w4.z;
          wts[4 * k + 3] = w4.w;
        }
        __syncwarp();  // every lane has the weights before the next head overwrites them
      }
      // v_rot += w_t c[idx_t] for the lane's E dimensions: VB E bits at bit VB E lane of the token's
      // index stream, read in pieces of up to 8 indices of up to 4 bits or 4 wider ones (at most 32
      // bits, one funnel shift each)
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float wt = kStagedW ? wts[t] : __shfl_sync(kFull, w, 2 * t);
        const uint32_t* row = vi + t * (VB * D / 32);
        constexpr int PMAX = VBT != 0 ? 8 : 4;
        constexpr int PIECE = E < PMAX ? E : PMAX;
#pragma unroll
        for (int c0 = 0; c0 < E; c0 += PIECE) {
          const int bitc = VB * (E * lane + c0);
          const uint32_t lo = row[bitc >> 5];
          const uint32_t hi = ((bitc & 31) + VB * PIECE > 32) ? row[(bitc >> 5) + 1] : 0u;
          const uint32_t bits = __funnelshift_r(lo, hi, bitc & 31);
#pragma unroll
          for (int e = 0; e < PIECE; ++e)
            acc[h][c0 + e] = fmaf(wt, lut[(bits >> (VB * e)) & vmask], acc[h][c0 + e]);
        }
      }
    }
    __syncwarp();
  }
  cp_wait<0>();

  // per-warp results (rotated domain) -> shared memory, combine, inverse rotation, partial
#pragma unroll
  for (int h = 0; h < NR; ++h) {
#pragma unroll
    for (int e = 0; e < E; ++e) wo[warp][h][lane * E + e] = acc[h][e];
    if (lane == 0) {
      wm[warp][h] = m_run[h];
      wl[warp][h] = l_run[h];
    }
  }
  __syncthreads();
  for (int h = warp; h < a.nrg; h += kWarps) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w][h]);
    float f[kWarps], den = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      f[w] = M == -INFINITY ? 0.f : fast_exp2(wm[w][h] - M);
      den = fmaf(f[w], wl[w][h], den);
    }
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = coord_of(e, lane);
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s = fmaf(f[w], wo[w][h][c], s);
      x[e] = s;
    }
    wht_warp<E>(x, lane);
    float* dst = a.parts + (((size_t)b * a.hq + h0 + h) * a.n_parts + part) * (D + 2);
    const float rs = rsqrtf((float)D);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = coord_of(e, lane);
      dst[c] = x[e] * rs * a.signs[c];
    }
    if (lane == 0) {
      dst[D] = M;
      dst[D + 1] = den;
    }
  }
}

template <int D, int NR, int VB, int KB>
cudaError_t launch_alt_vb(const AltArgs& a, dim3 grid, cudaStream_t s) {
  auto kern = decode_alt_v2_kernel<D, NR, VB, KB>;
  constexpr size_t SMEM = AltCfg<D, VB ? VB : 8, KB>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, SMEM, s>>>(a);
  return cudaGetLastError();
}

// 5- to 8-bit values (q5_0 .. q8_0) only with 8-bit or fp16 keys; other pairs take the CUDA-core
// decoder.
template <int D, int NR, int KB>
cudaError_t launch_alt_kb(const AltArgs& a, int vb, dim3 grid, cudaStream_t s) {
  if (vb > 4) {
    if constexpr (KB == 8 || KB == 16) return launch_alt_vb<D, NR, 0, KB>(a, grid, s);
    return cudaErrorNotSupported;
  }
  return vb == 2 ? launch_alt_vb<D, NR, 2, KB>(a, grid, s)
       : vb == 4 ? launch_alt_vb<D, NR, 4, KB>(a, grid, s)
                 : launch_alt_vb<D, NR, 3, KB>(a, grid, s);
}

template <int D, int NR>
cudaError_t launch_alt(const AltArgs& a, int vb, int kb, dim3 grid, cudaStream_t s) {
  switch (kb) {
    case 16: return launch_alt_kb<D, NR, 16>(a, vb, grid, s);
    case 2: return launch_alt_kb<D, NR, 2>(a, vb, grid, s);
    case 4: return launch_alt_kb<D, NR, 4>(a, vb, grid, s);
    case 5: return launch_alt_kb<D, NR, 5>(a, vb, grid, s);
    default: return launch_alt_kb<D, NR, 8>(a, vb, grid, s);
  }
}

}  // namespace

// Whether the warp-per-page kernel has an instance for the context: up to 4 query heads per KV-head
// group (4 at d <= 128, 2 at d <= 256, 1 at d = 512), value bits 2..4, or 5..8 beside 8-bit or
// fp16 keys.
bool alt_v2_supported(const tq_ctx* ctx) {
  const int d = ctx->cfg.head_dim, vb = ctx->cfg.value_bits, kb = ctx->cfg.key_bits;
  const int groups = (ctx->n_rep + kMaxRep - 1) / kMaxRep, nr = ctx->n_rep / groups;
  const bool heads = nr == 1 ? (d == 64 || d == 128 || d == 256 || d == 512)
                   : nr == 2 ? (d == 64 || d == 128 || d == 256)
                   : nr <= 4 && (d == 64 || d == 128);
  const bool widths = vb <= 4 || ((kb == 8 || kb == 16) && ctx->d_vcent);
  return heads && widths;
}

// Compressed parts of the alternate layout with the warp-per-page kernel, when it
// supports (d, heads per group); returns cudaErrorNotSupported otherwise.
cudaError_t launch_decode_alt_v2(tq_ctx* ctx, const void* q, const void* pool, int num_blocks,
                                 const int32_t* block_table, int max_blocks, const int32_t* n_compressed, int max_ctx,
                                 float* parts, int chunk_tokens, int n_chunks, int n_parts, int batch, cudaStream_t s) {
  AltArgs a{};
  a.q = static_cast<const __half*>(q);
  a.pool = static_cast<const uint8_t*>(pool);
  a.num_blocks = num_blocks;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.n_compressed = n_compressed;
  a.max_ctx = max_ctx;
  a.parts = parts;
  a.chunk_tokens = chunk_tokens;
  a.n_chunks = n_chunks;
  a.n_parts = n_parts;
  a.hq = ctx->cfg.num_q_heads;
  a.hkv = ctx->cfg.num_kv_heads;
  a.n_rep = ctx->n_rep;
  a.groups = (ctx->n_rep + kMaxRep - 1) / kMaxRep;
  a.nrg = ctx->n_rep / a.groups;
  a.signs = ctx->d_signs;
  a.tab = ctx->tab;
  a.vb = ctx->cfg.value_bits;
  a.vcent = ctx->d_vcent;
  a.err = ctx->d_err;
  dim3 grid(n_chunks, a.hkv * a.groups, batch);
  const int d = ctx->cfg.head_dim, nr = a.nrg, vb = ctx->cfg.value_bits, kb = ctx->cfg.key_bits;
  if (!alt_v2_supported(ctx)) return cudaErrorNotSupported;
  if (nr == 1) {
    switch (d) {
      case 64: return launch_alt<64, 1>(a, vb, kb, grid, s);
      case 128: return launch_alt<128, 1>(a, vb, kb, grid, s);
      case 256: return launch_alt<256, 1>(a, vb, kb, grid, s);
      case 512: return launch_alt<512, 1>(a, vb, kb, grid, s);
    }
  } else if (nr == 2) {
    switch (d) {
      case 64: return launch_alt<64, 2>(a, vb, kb, grid, s);
      case 128: return launch_alt<128, 2>(a, vb, kb, grid, s);
      case 256: return launch_alt<256, 2>(a, vb, kb, grid, s);
    }
  } else if (nr <= 4) {
    if (d == 64) return launch_alt<64, 4>(a, vb, kb, grid, s);
    if (d == 128) return launch_alt<128, 4>(a, vb, kb, grid, s);
  }
  return cudaErrorNotSupported;
}

}  // namespace tq
