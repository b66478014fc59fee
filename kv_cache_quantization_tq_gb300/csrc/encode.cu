// Write path of the compressed KV cache: the encode/flush kernels and the
// ring-buffer append with flush-on-overflow.
//
// Main layout, per (token, KV head) (turboquant vLLM guide, section 2 steps
// 1-5; turboquant-bench, compression algorithm details):
//   n_k = ||k||; y = H (D k) / (sqrt(d) n_k); idx_i = #{boundaries <= y_i};
//   r = y - c[idx]; n_r = ||r||; sigma_j = [(S r)_j >= 0];
//   values: asymmetric 2-bit min/max quantisation in groups of 32.
// Alternate layout (vllm-metal TurboQuant guide, quantisation table):
//   keys: 8-, 5-, 4- or 2-bit affine codes per block of 32, or the fp16 keys unchanged (the
//   V-only cache of the "TurboQuant-MLX overview"); values: n_v = ||v||, the 2-, 3- or 4-bit
//   Lloyd-Max index of H (D v) / (sqrt(d) n_v).
//
// One CTA encodes up to TB tokens of one (sequence, KV head): a warp per
// token computes norms, the rotation (registers + shuffles), the Lloyd-Max
// indices (bit planes straight from __ballot_sync) and the value codes; the
// QJL projection z = S r of all TB tokens is then a dense product on the
// tensor cores (mma.sync m16n8k16): the residuals are staged in shared memory
// as fp16 high parts and low parts scaled by 2^11, S comes as precomputed
// fragments of the same split, and z = hi*hi + 2^-11 (hi*lo + lo*hi) keeps
// ~22 bits, far inside the margin at which a sign may legitimately differ;
// finished tiles leave through 16-byte stores to the pages named by the block
// table.
#include "common.cuh"

namespace tq {
namespace {

struct EncArgs {
  const __half* k;
  const __half* v;
  int src_tokens;
  int n_tokens;
  const int32_t* start_pos;
  const int32_t* block_table;
  int max_blocks;
  uint8_t* pool;
  int num_blocks;
  int hkv;
  const float* signs;
  const uint4* sfrag;     // S^T as mma.sync B fragments (k = coordinate, n = sketch row), hi / lo
  int kb;                 // main layout: key bits, 3 (2-bit Lloyd-Max index) or 2 (1-bit index)
  int avb;                // alternate layout: value index bits, 2, 3 or 4
  int key_signed;         // alternate layout, 2-bit keys: signed symmetric codes (int2)
  const float* vbound;    // alternate layout: value decision boundaries (device, 2^vb - 1)
  CodeTables tab;
  uint32_t* err;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}

__device__ __forceinline__ void mma_f16_acc(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// S^T as B fragments of mma.sync m16n8k16 for z = r S^T with k = coordinate i and n = sketch
// row j: entry (ks, nt, lane) holds, for i0 = 16 ks + 2 (lane % 4) and j = 8 nt + lane / 4, the
// fp16 pairs (S[j][i0], S[j][i0+1]), (S[j][i0+8], S[j][i0+9]) — high parts, then the low parts
// (S - high) * 2^11.
__global__ void sketch_frag_enc_kernel(const float* __restrict__ s, int d, uint4* __restrict__ frag) {
  const int total = (d / 16) * (d / 8) * 32;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int lane = idx & 31, unit = idx >> 5;
  const int nt = unit % (d / 8), ks = unit / (d / 8);
  const int i0 = 16 * ks + 2 * (lane & 3), j = 8 * nt + (lane >> 2);
  const int cols[4] = {i0, i0 + 1, i0 + 8, i0 + 9};
  unsigned short hi[4], lo[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float v = s[(size_t)j * d + cols[r]];
    const __half h = __float2half_rn(v);
    hi[r] = __half_as_ushort(h);
    lo[r] = __half_as_ushort(__float2half_rn((v - __half2float(h)) * 2048.f));
  }
  frag[idx] = make_uint4(hi[0] | (uint32_t)hi[1] << 16, hi[2] | (uint32_t)hi[3] << 16, lo[0] | (uint32_t)lo[1] << 16,
                         lo[2] | (uint32_t)lo[3] << 16);
}

// ------------------------------------------------------------------ main layout
// Main tile: key bit planes (kb - 1 Lloyd-Max index planes, high bit first, then the QJL plane;
// turboquant vLLM guide, --key-bits 2, 3 or 4), VB-bit value codes (--value-bits 2 or 4), the
// group scale / minimum, the two norm rows.  Staging in shared memory is sized for kb = 4.
// Tokens per CTA for long encodes: 64 at d <= 256 (about 50 KB of shared memory at d = 128, 4 CTAs
// per SM; 128 tokens per CTA fit only 2 per SM and encoded 21% fewer tokens per second), 32 at d = 512.
// Short encodes (a 128-token flush) use 16 tokens per CTA: 8 times the CTAs, a quarter of the
// tokens per warp, for latency.
template <int D>
constexpr int main_tb_long() { return D <= 256 ? 64 : 32; }
constexpr int kMainTbShort = 16;

template <int D, int VB, int TB_ = main_tb_long<D>()>
struct MainEnc {
  static constexpr int E = D / 32;
  static constexpr int TB = TB_;
  static constexpr int TILE = (10 + 2 * VB) * D + 64;  // largest tile (kb = 4): staging stride
  static constexpr int THREADS = 256;
  static constexpr int RS = D + 8;                     // residual row stride (halves): conflict-free fragments
  static constexpr size_t SMEM_R = 2 * sizeof(__half) * TB * RS;  // high and low parts
  static constexpr size_t SMEM_TILES = (size_t)(TB / 16) * TILE;
  static constexpr size_t SMEM = SMEM_R + SMEM_TILES;
};

// Copy `npages` staged tiles (staging stride `stride`, `tile` bytes each) to the pool pages of (b, h)
// starting at token `start`.
__device__ void store_tiles(const EncArgs& a, const uint8_t* tiles, int stride, int tile, int npages, int b, int h,
                            int first_page) {
  for (int p = 0; p < npages; ++p) {
    const int page = first_page + p;
    int blk = -1;
    if (page < a.max_blocks) blk = a.block_table[(size_t)b * a.max_blocks + page];
    if (page >= a.max_blocks || blk < 0 || blk >= a.num_blocks) {
      if (threadIdx.x == 0) flag_error(a.err, page >= a.max_blocks ? TQ_DEVERR_POSITION : TQ_DEVERR_BLOCK_ID);
      continue;
    }
    uint4* dst = reinterpret_cast<uint4*>(a.pool + ((size_t)blk * a.hkv + h) * tile);
    const uint4* src = reinterpret_cast<const uint4*>(tiles + (size_t)p * stride);
    for (int i = threadIdx.x; i < tile / 16; i += blockDim.x) dst[i] = src[i];
  }
}

template <int D, int VB, int KB, int TB_>
__device__ void encode_main_block(const EncArgs& a, int b, int h, int tok0, int ntok, int start, uint8_t* smem) {
  using C = MainEnc<D, VB, TB_>;
  constexpr int E = C::E;
  constexpr int TB = C::TB;
  __half* rh = reinterpret_cast<__half*>(smem);                 // [TB][RS] residual, fp16 high part
  __half* rl = rh + TB * C::RS;                                 // [TB][RS] (r - high) * 2^11
  uint8_t* tiles = smem + C::SMEM_R;                            // [TB/16][TILE]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t base = ((size_t)b * a.hkv + h) * a.src_tokens;

  // ---- phase 0: the block's k and v rows (contiguous in [B][Hkv][src_tokens][d]) staged with
  // 16-byte cp.async into the residual buffers, row stride RS: token tt's k row sits where its
  // residual's high part goes and its v row where the low part goes.  Each token's rows are read
  // and then overwritten by the one warp that encodes it, so no other warp ever sees them change.
  {
    constexpr int CH = D / 8;  // 16-byte chunks per row
    const __half* kb = a.k + (base + tok0) * D;
    const __half* vb = a.v + (base + tok0) * D;
    for (int i = threadIdx.x; i < ntok * CH; i += C::THREADS) {
      const int tt = i / CH, c = i % CH;
      cp_async16(rh + tt * C::RS + 8 * c, kb + (size_t)tt * D + 8 * c);
      cp_async16(rl + tt * C::RS + 8 * c, vb + (size_t)tt * D + 8 * c);
    }
    asm volatile("cp.async.commit_group;\n" ::);
  }
  // value-code words of the block's pages (2 VB d bytes each) start at zero: phase 1 ORs every
  // code into them
  {
    constexpr int WPP = 2 * VB * D / 4;  // words per page
    for (int i = threadIdx.x; i < (TB / 16) * WPP; i += C::THREADS)
      reinterpret_cast<uint32_t*>(tiles + (size_t)(i / WPP) * C::TILE + 2 * KB * D)[i % WPP] = 0u;
  }
  float sg[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sg[e] = a.signs[coord_of(e, lane)];
  const float sqrt_d = sqrtf((float)D);
  asm volatile("cp.async.wait_group 0;\n" ::);
  __syncthreads();

  // ---- phase 1: one warp per token
  constexpr int o_ks = 2 * (KB - 1) * D, o_vq = 2 * KB * D;      // QJL plane, value codes
  constexpr int o_vsm = o_vq + 2 * VB * D, o_norm = o_vsm + 2 * D; // scale / minimum, norms
  for (int tt = warp; tt < ntok; tt += C::THREADS / 32) {
    const __half* kp = rh + tt * C::RS;  // staged k and v rows of this token
    const __half* vp = rl + tt * C::RS;
    float x[E], vv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      x[e] = __half2float(kp[coord_of(e, lane)]);
      vv[e] = __half2float(vp[coord_of(e, lane)]);
    }
    __syncwarp();  // every lane has its k and v values before any lane overwrites the rows
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
    const float nk = sqrtf(warp_sum(ss));
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] *= sg[e];
    wht_warp<E>(x, lane);
    const float inv = nk > 0.f ? __fdiv_rn(1.f, sqrt_d * nk) : 0.f;
    uint8_t* tile = tiles + (size_t)(tt >> 4) * C::TILE;
    const int slot = tt & 15;
    float rr = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float y = x[e] * inv;
      // #{boundaries <= y} over the 2^(kb-1) - 1 boundaries (straight-line code per key width)
      // #{boundaries <= y}: the comparisons with the ascending boundaries form a thermometer code
      // n_0 >= n_1 >= ..., so the index bits are XORs of comparisons (bit 1 of a 2-bit index is
      // n_1, bit 0 the parity of all three) and the centroid is a chain of selects (a NaN y
      // compares false everywhere: index 0, as with the count)
      bool ib0, ib1 = false, ib2 = false;  // index bits
      float cy;
      if (KB == 3) {
        const bool n0 = y >= a.tab.b[0], n1 = y >= a.tab.b[1], n2 = y >= a.tab.b[2];
        ib1 = n1;
        ib0 = n0 ^ n1 ^ n2;
        cy = n2 ? a.tab.c[3] : n1 ? a.tab.c[2] : n0 ? a.tab.c[1] : a.tab.c[0];
      } else if (KB == 2) {
        ib0 = y >= a.tab.b[0];
        cy = ib0 ? a.tab.c[1] : a.tab.c[0];
      } else {
        bool n[7];
#pragma unroll
        for (int j = 0; j < 7; ++j) n[j] = y >= a.tab.b[j];
        ib2 = n[3];
        ib1 = n[1] ^ n[3] ^ n[5];
        ib0 = n[0] ^ n[1] ^ n[2] ^ n[3] ^ n[4] ^ n[5] ^ n[6];
        cy = a.tab.c[0];
#pragma unroll
        for (int j = 0; j < 7; ++j) cy = n[j] ? a.tab.c[j + 1] : cy;
      }
      const float r = y - cy;
      rr = fmaf(r, r, rr);
      const __half r_hi = __float2half_rn(r);
      rh[tt * C::RS + coord_of(e, lane)] = r_hi;
      rl[tt * C::RS + coord_of(e, lane)] = __float2half_rn((r - __half2float(r_hi)) * 2048.f);
      // index planes, high bit first
      uint32_t* kp0 = reinterpret_cast<uint32_t*>(tile + slot * (D / 8)) + e;
      if (KB == 3) {
        const unsigned hi = __ballot_sync(kFull, ib1);
        const unsigned lo = __ballot_sync(kFull, ib0);
        if (lane == 0) {
          kp0[0] = hi;
          kp0[2 * D / 4] = lo;
        }
      } else if (KB == 2) {
        const unsigned bits = __ballot_sync(kFull, ib0);
        if (lane == 0) kp0[0] = bits;
      } else {
        const unsigned b2 = __ballot_sync(kFull, ib2);
        const unsigned b1 = __ballot_sync(kFull, ib1);
        const unsigned b0 = __ballot_sync(kFull, ib0);
        if (lane == 0) {
          kp0[0] = b2;
          kp0[2 * D / 4] = b1;
          kp0[4 * D / 4] = b0;
        }
      }
    }
    const float nr = sqrtf(warp_sum(rr));
    if (lane == 0) {
      reinterpret_cast<__half*>(tile + o_norm)[slot] = __float2half_rn(nk);
      reinterpret_cast<__half*>(tile + o_norm + 32)[slot] = __float2half_rn(nr);
    }
    // values: group e = coordinates 32e..32e+31, one per lane
    float vmn[E], vmx[E];
    group_minmax<E>(vv, vmn, vmx);
    constexpr float vlevels = (float)((1 << VB) - 1);
    __half2 vsm[E], vmine;
    group_pairs<E, false>(vmn, vmx, vlevels, lane, vsm, vmine);
    if (lane < E) *reinterpret_cast<__half2*>(tile + o_vsm + (slot * (D / 32) + lane) * 4) = vmine;
    // dimension-major code words: 2-bit: one word per dimension, token 2j+e at bits 16e+2j; 4-bit:
    // two words per dimension (all first words, then all second words), word w holding tokens
    // 8w+2j+e at bits 16e+4j.  Tokens of a page come from different warps: OR into the words.
    uint32_t* vqw = reinterpret_cast<uint32_t*>(tile + o_vq) + (VB == 4 ? (slot >> 3) * D : 0);
    const int vsh = VB == 2 ? 16 * (slot & 1) + 2 * (slot >> 1) : 16 * (slot & 1) + 4 * ((slot & 7) >> 1);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int q = group_code(vv[e], vsm[e], vlevels);
      if (q) atomicOr(vqw + coord_of(e, lane), (uint32_t)q << vsh);
    }
  }
  __syncthreads();

  // ---- phase 2: QJL sketch z = S r on the tensor cores; one unit = 16 tokens x one plane word
  // (32 sketch rows = 4 n-tiles); sign bits gathered into the word by two shuffles
  {
    constexpr int NG = 4;
    constexpr int UNITS = (TB / 16) * (D / 32);
    const int g = lane >> 2, t = lane & 3;
    for (int u = warp; u < UNITS; u += C::THREADS / 32) {
      const int tile16 = u / (D / 32), wd = u % (D / 32);
      const int row0 = (tile16 * 16 + g) * C::RS, row1 = row0 + 8 * C::RS;
      float acc[NG][4], cor[NG][4];
#pragma unroll
      for (int j = 0; j < NG; ++j)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[j][r] = cor[j][r] = 0.f;
#pragma unroll 4  // measured: 4 k-steps of fragment loads in flight (+9% encode), 8 is slower
      for (int ks = 0; ks < D / 16; ++ks) {
        const int k0 = 16 * ks + 2 * t;
        uint4 ah, al;
        ah.x = *reinterpret_cast<const uint32_t*>(rh + row0 + k0);
        ah.y = *reinterpret_cast<const uint32_t*>(rh + row1 + k0);
        ah.z = *reinterpret_cast<const uint32_t*>(rh + row0 + k0 + 8);
        ah.w = *reinterpret_cast<const uint32_t*>(rh + row1 + k0 + 8);
        al.x = *reinterpret_cast<const uint32_t*>(rl + row0 + k0);
        al.y = *reinterpret_cast<const uint32_t*>(rl + row1 + k0);
        al.z = *reinterpret_cast<const uint32_t*>(rl + row0 + k0 + 8);
        al.w = *reinterpret_cast<const uint32_t*>(rl + row1 + k0 + 8);
        const uint4* bf = a.sfrag + ((size_t)ks * (D / 8) + NG * wd) * 32 + lane;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
          const uint4 bv = __ldg(bf + j * 32);
          mma_f16_acc(acc[j], ah, bv.x, bv.y);
          mma_f16_acc(cor[j], ah, bv.z, bv.w);
          mma_f16_acc(cor[j], al, bv.x, bv.y);
        }
      }
      // sketch row 32 wd + 8 j + 2 t + e sits at bit 16 e + 4 j + t of plane word wd
      uint32_t w0 = 0u, w1 = 0u;  // tokens g and g + 8
#pragma unroll
      for (int j = 0; j < NG; ++j) {
        const int jj = 4 * j + t;
        w0 |= (fmaf(cor[j][0], 1.f / 2048.f, acc[j][0]) >= 0.f ? 1u : 0u) << jj;
        w0 |= (fmaf(cor[j][1], 1.f / 2048.f, acc[j][1]) >= 0.f ? 1u : 0u) << (16 + jj);
        w1 |= (fmaf(cor[j][2], 1.f / 2048.f, acc[j][2]) >= 0.f ? 1u : 0u) << jj;
        w1 |= (fmaf(cor[j][3], 1.f / 2048.f, acc[j][3]) >= 0.f ? 1u : 0u) << (16 + jj);
      }
      w0 |= __shfl_xor_sync(kFull, w0, 1);
      w0 |= __shfl_xor_sync(kFull, w0, 2);
      w1 |= __shfl_xor_sync(kFull, w1, 1);
      w1 |= __shfl_xor_sync(kFull, w1, 2);
      if (t == 0) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int tt = tile16 * 16 + g + 8 * hh;
          if (tt < ntok) {
            uint8_t* tile = tiles + (size_t)(tt >> 4) * C::TILE;
            reinterpret_cast<uint32_t*>(tile + o_ks + (tt & 15) * (D / 8))[wd] = hh ? w1 : w0;
          }
        }
      }
    }
  }
  __syncthreads();
  store_tiles(a, tiles, C::TILE, o_norm + 64, ntok >> 4, b, h, (start + tok0) >> 4);
}

// ------------------------------------------------------------------ alternate layout
// Alternate-layout page (alt_tile_bytes): a dense kb-bit stream of key codes per token (kb = 8, 5,
// 4 or 2; 8 bits: one byte per coordinate) and 16 x d/32 (scale, minimum) fp16 pairs, or the fp16
// keys (kb = 16); a dense vb-bit stream of value indices per token (index i at bit vb i); 16 fp16
// value norms.  The function attribute allows the largest staging (kb = 16, vb = 8).
template <int D>
struct AltEnc {
  static constexpr int E = D / 32;
  static constexpr int TB = 32;
  static constexpr int THREADS = 256;
  // staged tiles, value codes, and (keys below 8 bits) key codes before packing
  static constexpr size_t smem(int kb, int vb) {
    return (size_t)(TB / 16) * alt_tile_bytes(D, kb, vb) + (size_t)TB * D + (kb == 8 || kb == 16 ? 0 : (size_t)TB * D);
  }
  static constexpr size_t SMEM = smem(16, 8);  // the largest
  static_assert(smem(16, 8) >= smem(8, 8) && smem(16, 8) >= smem(5, 8) && smem(16, 8) >= smem(4, 8) &&
                    smem(16, 8) >= smem(2, 8),
                "fp16 keys and 8-bit values bound the staging");
};

// Codes of every staged token as a dense little-endian VB-bit stream at byte `offset` of its page
// (VB d / 8 bytes per token): index kk of a chunk of 32 at bit VB kk of the chunk's VB words.
template <int D, int VB>
__device__ __forceinline__ void pack_value_stream(const uint8_t* vcodes, uint8_t* tiles, int tile_bytes, int ntok,
                                                  int offset) {
  for (int w = threadIdx.x; w < ntok * (D / 32); w += AltEnc<D>::THREADS) {
    const int tt = w / (D / 32), chunk = w % (D / 32);
    uint32_t o[VB];
#pragma unroll
    for (int i = 0; i < VB; ++i) o[i] = 0u;
#pragma unroll
    for (int kk = 0; kk < 32; ++kk) {
      const uint32_t code = vcodes[tt * D + chunk * 32 + kk];
      const int bit = VB * kk;
      o[bit >> 5] |= code << (bit & 31);
      if ((bit & 31) + VB > 32) o[(bit >> 5) + 1] |= code >> (32 - (bit & 31));
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(tiles + (size_t)(tt >> 4) * tile_bytes + offset +
                                                (tt & 15) * (VB * D / 8) + chunk * 4 * VB);
#pragma unroll
    for (int i = 0; i < VB; ++i) dst[i] = o[i];
  }
}

template <int D, int VB>
__device__ void encode_alt_block_vb(const EncArgs& a, int b, int h, int tok0, int ntok, int start, uint8_t* smem) {
  using C = AltEnc<D>;
  constexpr int E = C::E;
  constexpr int vb = VB, nbound = (1 << VB) - 1;
  const int kb = a.kb, tile_bytes = alt_tile_bytes(D, kb, vb);
  const int o_ksm = 2 * kb * D, o_vi = alt_key_bytes(D, kb), o_vn = o_vi + 2 * vb * D;
  uint8_t* tiles = smem;
  uint8_t* vcodes = smem + (size_t)(C::TB / 16) * tile_bytes;
  uint8_t* kcodes = vcodes + C::TB * D;  // keys below 8 bits: staged, then packed
  // 5- to 8-bit values: the boundaries in shared memory for a binary search (the narrower codebooks
  // compare against the kernel-parameter table)
  __shared__ float sbound[VB >= 5 ? (1 << VB) : 1];
  if (VB >= 5) {
    for (int i = threadIdx.x; i < nbound; i += C::THREADS) sbound[i] = a.vbound[i];
    __syncthreads();
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t base = ((size_t)b * a.hkv + h) * a.src_tokens;
  float sg[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sg[e] = a.signs[coord_of(e, lane)];
  const float sqrt_d = sqrtf((float)D);

  for (int tt = warp; tt < ntok; tt += C::THREADS / 32) {
    const __half* kp = a.k + (base + tok0 + tt) * D;
    const __half* vp = a.v + (base + tok0 + tt) * D;
    uint8_t* tile = tiles + (size_t)(tt >> 4) * tile_bytes;
    const int slot = tt & 15;
    float vv[E], kx[E], kmn[E], kmx[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = coord_of(e, lane);
      kx[e] = __half2float(kp[c]);
      vv[e] = __half2float(vp[c]);
    }
    if (kb == 16) {  // keys kept as they are: the fp16 inputs (exact through fp32)
      __half* kh = reinterpret_cast<__half*>(tile) + slot * D;
#pragma unroll
      for (int e = 0; e < E; ++e) kh[coord_of(e, lane)] = __float2half_rn(kx[e]);
    } else {
      group_minmax<E>(kx, kmn, kmx);
      const float klevels = (float)((1 << kb) - 1);
      __half2 ksm[E], kmine;
      if (a.key_signed)
        group_pairs<E, true>(kmn, kmx, klevels, lane, ksm, kmine);
      else
        group_pairs<E, false>(kmn, kmx, klevels, lane, ksm, kmine);
      if (lane < E) *reinterpret_cast<__half2*>(tile + o_ksm + (slot * (D / 32) + lane) * 4) = kmine;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int c = coord_of(e, lane);
        const int q = group_code(kx[e], ksm[e], klevels);
        if (kb == 8)
          tile[slot * D + c] = (uint8_t)q;
        else
          kcodes[tt * D + c] = (uint8_t)q;
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(vv[e], vv[e], ss);
    const float nv = sqrtf(warp_sum(ss));
#pragma unroll
    for (int e = 0; e < E; ++e) vv[e] *= sg[e];
    wht_warp<E>(vv, lane);
    const float inv = nv > 0.f ? __fdiv_rn(1.f, sqrt_d * nv) : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float y = vv[e] * inv;
      // #{boundaries <= y} over the 2^vb - 1 ascending boundaries (ties go up)
      int idx = 0;
      if (VB >= 5) {
        // binary lifting: idx + step - 1 <= 2^VB - 2 at every step, inside the table
#pragma unroll
        for (int step = 1 << (VB - 1); step; step >>= 1) idx += (y >= sbound[idx + step - 1]) ? step : 0;
      } else {
#pragma unroll
        for (int j = 0; j < nbound; ++j) idx += y >= a.tab.b[j];
      }
      vcodes[tt * D + coord_of(e, lane)] = (uint8_t)idx;
    }
    if (lane == 0) reinterpret_cast<__half*>(tile + o_vn)[slot] = __float2half_rn(nv);
  }
  __syncthreads();
  // dense vb-bit stream per token: 32 indices -> vb words; keys below 8 bits likewise (kb words)
  pack_value_stream<D, VB>(vcodes, tiles, tile_bytes, ntok, o_vi);
  if (kb == 4)
    pack_value_stream<D, 4>(kcodes, tiles, tile_bytes, ntok, 0);
  else if (kb == 5)
    pack_value_stream<D, 5>(kcodes, tiles, tile_bytes, ntok, 0);
  else if (kb == 2)
    pack_value_stream<D, 2>(kcodes, tiles, tile_bytes, ntok, 0);
  __syncthreads();
  store_tiles(a, tiles, tile_bytes, tile_bytes, ntok >> 4, b, h, (start + tok0) >> 4);
}

template <int D>
__device__ void encode_alt_block(const EncArgs& a, int b, int h, int tok0, int ntok, int start, uint8_t* smem) {
  switch (a.avb) {
    case 2: encode_alt_block_vb<D, 2>(a, b, h, tok0, ntok, start, smem); break;
    case 4: encode_alt_block_vb<D, 4>(a, b, h, tok0, ntok, start, smem); break;
    case 5: encode_alt_block_vb<D, 5>(a, b, h, tok0, ntok, start, smem); break;
    case 6: encode_alt_block_vb<D, 6>(a, b, h, tok0, ntok, start, smem); break;
    case 7: encode_alt_block_vb<D, 7>(a, b, h, tok0, ntok, start, smem); break;
    case 8: encode_alt_block_vb<D, 8>(a, b, h, tok0, ntok, start, smem); break;
    default: encode_alt_block_vb<D, 3>(a, b, h, tok0, ntok, start, smem); break;
  }
}

// ------------------------------------------------------------------ kernels
// VB: value bits of the main layout (2 or 4), 0 for the alternate layout; TB: tokens per CTA of
// the main layout (the alternate layout's are fixed).
template <int D, int VB>
constexpr int enc_tb(bool short_run) {
  return VB ? (short_run ? kMainTbShort : main_tb_long<D>()) : AltEnc<D>::TB;
}

template <int D, int VB, int TB>
__device__ __forceinline__ void encode_block(const EncArgs& a, int b, int h, int tok0, int ntok, int start,
                                             uint8_t* smem) {
  if constexpr (VB == 0) {
    encode_alt_block<D>(a, b, h, tok0, ntok, start, smem);
  } else {
    if (a.kb == 3)
      encode_main_block<D, VB, 3, TB>(a, b, h, tok0, ntok, start, smem);
    else if (a.kb == 2)
      encode_main_block<D, VB, 2, TB>(a, b, h, tok0, ntok, start, smem);
    else
      encode_main_block<D, VB, 4, TB>(a, b, h, tok0, ntok, start, smem);
  }
}

template <int D, int VB, int TB>
__global__ void __launch_bounds__(256) encode_kernel(EncArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int b = blockIdx.z, h = blockIdx.y;
  const int tok0 = blockIdx.x * TB;
  const int ntok = min(TB, a.n_tokens - tok0);
  const int start = a.start_pos[b];
  if (start < 0 || (start & 15)) {
    if (threadIdx.x == 0) flag_error(a.err, TQ_DEVERR_POSITION);
    return;
  }
  encode_block<D, VB, TB>(a, b, h, tok0, ntok, start, smem);
}

struct AppendArgs {
  EncArgs enc;          // k/v point at the rings, src_tokens = 128
  const __half* k_new;
  const __half* v_new;
  const int32_t* pos;
  __half* ring_k;
  __half* ring_v;
};

// One CTA per (KV head, sequence, TB-token slice of the ring).  When the ring is full (pos a
// nonzero multiple of 128) each slice compresses its tokens; the new token then goes to ring
// slot pos mod 128, written by the slice that holds that slot, after its own tokens were read.
template <int D, int VB, int TB>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int b = blockIdx.y, h = blockIdx.x, t0 = blockIdx.z * TB;
  static_assert(kRing % TB == 0, "ring flush is a whole number of encode batches");
  const int pos = a.pos[b];
  if (pos < 0) {
    if (threadIdx.x == 0 && blockIdx.z == 0) flag_error(a.enc.err, TQ_DEVERR_POSITION);
    return;
  }
  const int slot = pos % kRing;
  if (pos > 0 && slot == 0) encode_block<D, VB, TB>(a.enc, b, h, t0, TB, pos - kRing, smem);
  if (slot < t0 || slot >= t0 + TB) return;
  const size_t src = ((size_t)b * a.enc.hkv + h) * D;
  const size_t dst = (((size_t)b * a.enc.hkv + h) * kRing + slot) * D;
  for (int i = threadIdx.x; i < D / 8; i += blockDim.x) {
    reinterpret_cast<uint4*>(a.ring_k + dst)[i] = reinterpret_cast<const uint4*>(a.k_new + src)[i];
    reinterpret_cast<uint4*>(a.ring_v + dst)[i] = reinterpret_cast<const uint4*>(a.v_new + src)[i];
  }
}

// Dynamic shared memory of one launch: the main layout's fixed staging, or the alternate layout's
// for its key and value widths (the function attribute allows the largest).
template <int D, int VB, int TB>
size_t enc_smem(const EncArgs& a) {
  if constexpr (VB == 0) return AltEnc<D>::smem(a.kb, a.avb);
  else return MainEnc<D, VB, TB>::SMEM;
}
template <int D, int VB, int TB>
constexpr size_t enc_smem_max() {
  if constexpr (VB == 0) return AltEnc<D>::SMEM;
  else return MainEnc<D, VB, TB>::SMEM;
}

template <int D, int VB, int TB>
cudaError_t launch_encode_tb(const EncArgs& a, int batch, cudaStream_t s) {
  auto kern = encode_kernel<D, VB, TB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)enc_smem_max<D, VB, TB>());
  if (e != cudaSuccess) return e;
  dim3 grid((a.n_tokens + TB - 1) / TB, a.hkv, batch);
  kern<<<grid, 256, enc_smem<D, VB, TB>(a), s>>>(a);
  return cudaGetLastError();
}

// Short encodes (fewer CTAs of the long size than two per SM) take the short CTAs.
template <int D, int VB>
cudaError_t launch_encode_t(const EncArgs& a, int batch, int sm_count, cudaStream_t s) {
  constexpr int TL = enc_tb<D, VB>(false);
  const int64_t ctas = (int64_t)((a.n_tokens + TL - 1) / TL) * a.hkv * batch;
  if (VB && ctas < 2 * (int64_t)sm_count) return launch_encode_tb<D, VB, enc_tb<D, VB>(true)>(a, batch, s);
  return launch_encode_tb<D, VB, TL>(a, batch, s);
}

template <int D, int VB>
cudaError_t launch_append_t(const AppendArgs& a, int batch, cudaStream_t s) {
  constexpr int TB = enc_tb<D, VB>(true);
  auto kern = append_kernel<D, VB, TB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)enc_smem_max<D, VB, TB>());
  if (e != cudaSuccess) return e;
  dim3 grid(a.enc.hkv, batch, kRing / TB);
  kern<<<grid, 256, enc_smem<D, VB, TB>(a.enc), s>>>(a);
  return cudaGetLastError();
}

EncArgs make_args(tq_ctx* ctx, const void* k, const void* v, int src_tokens, int n_tokens, const int32_t* start_pos,
                  const int32_t* block_table, int max_blocks, void* pool, int num_blocks) {
  EncArgs a;
  a.k = static_cast<const __half*>(k);
  a.v = static_cast<const __half*>(v);
  a.src_tokens = src_tokens;
  a.n_tokens = n_tokens;
  a.start_pos = start_pos;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.pool = static_cast<uint8_t*>(pool);
  a.num_blocks = num_blocks;
  a.hkv = ctx->cfg.num_kv_heads;
  a.signs = ctx->d_signs;
  a.sfrag = ctx->d_sfrag_enc;
  a.kb = ctx->cfg.key_bits;
  a.avb = ctx->cfg.value_bits;
  a.key_signed = ctx->cfg.layout == TQ_LAYOUT_ALT && ctx->cfg.key_format == TQ_KEY_SIGNED;
  a.vbound = ctx->d_vbound;
  a.tab = ctx->tab;
  a.err = ctx->d_err;
  return a;
}

}  // namespace

cudaError_t launch_encode(tq_ctx* ctx, const void* k, const void* v, int batch, int src_tokens, int n_tokens,
                          const int32_t* start_pos, const int32_t* block_table, int max_blocks, void* pool,
                          int num_blocks, cudaStream_t s) {
  EncArgs a = make_args(ctx, k, v, src_tokens, n_tokens, start_pos, block_table, max_blocks, pool, num_blocks);
  const int vb = ctx->cfg.layout == TQ_LAYOUT_MAIN ? ctx->cfg.value_bits : 0;
  cudaError_t e = cudaErrorInvalidValue;
  prof_start(ctx, kProfEncode, s);
  switch (ctx->cfg.head_dim) {
    case 64: e = vb == 4 ? launch_encode_t<64, 4>(a, batch, ctx->sm_count, s) : vb == 2 ? launch_encode_t<64, 2>(a, batch, ctx->sm_count, s) : launch_encode_t<64, 0>(a, batch, ctx->sm_count, s); break;
    case 128: e = vb == 4 ? launch_encode_t<128, 4>(a, batch, ctx->sm_count, s) : vb == 2 ? launch_encode_t<128, 2>(a, batch, ctx->sm_count, s) : launch_encode_t<128, 0>(a, batch, ctx->sm_count, s); break;
    case 256: e = vb == 4 ? launch_encode_t<256, 4>(a, batch, ctx->sm_count, s) : vb == 2 ? launch_encode_t<256, 2>(a, batch, ctx->sm_count, s) : launch_encode_t<256, 0>(a, batch, ctx->sm_count, s); break;
    case 512: e = vb == 4 ? launch_encode_t<512, 4>(a, batch, ctx->sm_count, s) : vb == 2 ? launch_encode_t<512, 2>(a, batch, ctx->sm_count, s) : launch_encode_t<512, 0>(a, batch, ctx->sm_count, s); break;
  }
  prof_stop(ctx, kProfEncode, s);
  if (e == cudaSuccess) ctx->launches++;
  return e;
}

cudaError_t launch_append(tq_ctx* ctx, const void* k_new, const void* v_new, const int32_t* pos, int batch,
                          void* ring_k, void* ring_v, const int32_t* block_table, int max_blocks, void* pool,
                          int num_blocks, cudaStream_t s) {
  AppendArgs a;
  a.enc = make_args(ctx, ring_k, ring_v, kRing, kRing, nullptr, block_table, max_blocks, pool, num_blocks);
  a.k_new = static_cast<const __half*>(k_new);
  a.v_new = static_cast<const __half*>(v_new);
  a.pos = pos;
  a.ring_k = static_cast<__half*>(ring_k);
  a.ring_v = static_cast<__half*>(ring_v);
  const int vb = ctx->cfg.layout == TQ_LAYOUT_MAIN ? ctx->cfg.value_bits : 0;
  cudaError_t e = cudaErrorInvalidValue;
  switch (ctx->cfg.head_dim) {
    case 64: e = vb == 4 ? launch_append_t<64, 4>(a, batch, s) : vb == 2 ? launch_append_t<64, 2>(a, batch, s) : launch_append_t<64, 0>(a, batch, s); break;
    case 128: e = vb == 4 ? launch_append_t<128, 4>(a, batch, s) : vb == 2 ? launch_append_t<128, 2>(a, batch, s) : launch_append_t<128, 0>(a, batch, s); break;
    case 256: e = vb == 4 ? launch_append_t<256, 4>(a, batch, s) : vb == 2 ? launch_append_t<256, 2>(a, batch, s) : launch_append_t<256, 0>(a, batch, s); break;
    case 512: e = vb == 4 ? launch_append_t<512, 4>(a, batch, s) : vb == 2 ? launch_append_t<512, 2>(a, batch, s) : launch_append_t<512, 0>(a, batch, s); break;
  }
  if (e == cudaSuccess) ctx->launches++;
  return e;
}

cudaError_t build_sketch_frags_enc(const float* sketch, int d, void* frag) {
  const int total = (d / 16) * (d / 8) * 32;
  sketch_frag_enc_kernel<<<(total + 255) / 256, 256>>>(sketch, d, static_cast<uint4*>(frag));
  cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : cudaDeviceSynchronize();
}

}  // namespace tq
