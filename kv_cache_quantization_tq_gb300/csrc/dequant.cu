// Prefill materialisation: the compressed history of every sequence read back
// as dense fp16 keys and values (vllm-metal TurboQuant guide, advanced
// settings: with a long history and a long prefill the history pages are
// dequantised to fp16 once and ordinary attention runs on them).
//
// Main layout, per (token, KV head) — the reconstruction the score estimator
// stands for (turboquant vLLM guide, section 2 steps 2-3):
//   x   = c[idx] + sqrt(pi/2)/m * n_r * S^T (2 sigma - 1)
//   k^  = n_k * D (H x) / sqrt(d)                     (inverse rotation)
//   v^  = mn_g + s_g q                                 (turboquant-bench: asymmetric groups)
// Alternate layout (vllm-metal TurboQuant guide, quantisation table):
//   k^  = mn_b + s_b q (or the stored fp16 key) ;  v^ = n_v * D (H c[idx]) / sqrt(d).
//
// One CTA handles TB tokens (whole pages) of one (sequence, KV head).  The
// QJL back-projection Z = (2 sigma - 1) S of a page (16 tokens x m sketch
// rows -> 16 x d) is a dense product and runs as mma.sync m16n8k16: the sign
// bits enter as exact fp16 +-1 (A), S as an fp16 high part plus a low part
// scaled by 2^11 (B, precomputed per context in fragment order), the low pass
// with A = +-2^-11 so both passes share one fp32 accumulator (~22-bit S).
// The rest is warp-per-token work: codes from the bit planes, the butterfly in
// registers and shuffles, coalesced fp16 stores.  The exact recent buffer is
// appended after the compressed tokens by a copy kernel.
#include <cuda_bf16.h>

#include <type_traits>

#include "common.cuh"

namespace tq {
namespace {

struct DqArgs {
  const uint8_t* pool;
  int num_blocks;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* n_tokens;
  const __half* ring_k;
  const __half* ring_v;
  const int32_t* n_buf;
  int max_tokens;
  void* k_out;   // fp16 or bf16 [batch][Hkv][max_tokens][d] (the kernels' OUT type)
  void* v_out;
  int hkv;
  const float* signs;
  const uint4* sfrag;   // S as mma.sync B fragments (back-projection order), fp16 high / low
  int kb;               // main layout key bits (3 or 2)
  int avb;              // alternate layout value index bits (2 .. 8)
  CodeTables tab;
  const float* vcent;   // alternate layout: value centroids in device memory (2^avb of them)
  float qjl_coef;       // sqrt(pi/2) / m
  uint32_t* err;
};

// Output element types of the materialisation: fp16 or bf16, rounded to nearest even from fp32.
__device__ __forceinline__ void store_out(__half* p, float v) { *p = __float2half_rn(v); }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ void mma_f16_acc(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// S (m = d rows) as B fragments of mma.sync m16n8k16 for Z = A S with k = sketch row j and
// n = coordinate i: entry (ks, nt, lane) holds, for j0 = 16 ks + 2 (lane % 4) and
// i = 8 nt + lane / 4, the fp16 pairs (S[j0][i], S[j0+1][i]), (S[j0+8][i], S[j0+9][i]) — high
// parts, then the low parts (S - high) * 2^11.
__global__ void sketch_frag_kernel(const float* __restrict__ s, int d, uint4* __restrict__ frag) {
  const int total = (d / 16) * (d / 8) * 32;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int lane = idx & 31, unit = idx >> 5;
  const int nt = unit % (d / 8), ks = unit / (d / 8);
  const int j0 = 16 * ks + 2 * (lane & 3), i = 8 * nt + (lane >> 2);
  const int rows[4] = {j0, j0 + 1, j0 + 8, j0 + 9};
  unsigned short hi[4], lo[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float v = s[(size_t)rows[r] * d + i];
    const __half h = __float2half_rn(v);
    hi[r] = __half_as_ushort(h);
    lo[r] = __half_as_ushort(__float2half_rn((v - __half2float(h)) * 2048.f));
  }
  frag[idx] = make_uint4(hi[0] | (uint32_t)hi[1] << 16, hi[2] | (uint32_t)hi[3] << 16, lo[0] | (uint32_t)lo[1] << 16,
                         lo[2] | (uint32_t)lo[3] << 16);
}

// Compressed tokens of sequence b, validated against the block table and the output rows.
__device__ __forceinline__ int dq_ntok(const DqArgs& a, int b) {
  const int n = a.n_tokens[b];
  if (n < 0 || (n & 15) || n > a.max_blocks * kPage || n > a.max_tokens) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) flag_error(a.err, TQ_DEVERR_POSITION);
    return 0;
  }
  return n;
}

// Copies this CTA's pages (`tile` bytes each, staged `stride` bytes apart) into shared memory;
// a bad block id is flagged and its page marked in ok[].
__device__ void load_tiles(const DqArgs& a, uint8_t* tiles, int stride, int tile, int b, int h, int page0,
                           int npages, bool* ok) {
  const int32_t* bt = a.block_table + (size_t)b * a.max_blocks;
  for (int p = 0; p < npages; ++p) {
    const int blk = bt[page0 + p];
    if (blk < 0 || blk >= a.num_blocks) {
      if (threadIdx.x == 0) {
        flag_error(a.err, TQ_DEVERR_BLOCK_ID);
        ok[p] = false;
      }
      continue;
    }
    if (threadIdx.x == 0) ok[p] = true;
    const uint4* src = reinterpret_cast<const uint4*>(a.pool + ((size_t)blk * a.hkv + h) * tile);
    uint4* dst = reinterpret_cast<uint4*>(tiles + (size_t)p * stride);
    for (int i = threadIdx.x; i < tile / 16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
}

// ------------------------------------------------------------------ main layout
// VB = value bits (2 or 4): value codes take VB * d / 8 bytes per token.  The key bits (2, 3 or
// 4) are a run-time value; the staging stride is the 4-bit-key tile.
template <int D, int VB>
struct MainDq {
  static constexpr int E = D / 32;
  static constexpr int TB = D >= 512 ? 16 : 32;          // tokens per CTA
  static constexpr int TILE = (10 + 2 * VB) * D + 64;    // staging stride
  static constexpr int THREADS = 256;
  static constexpr int PAGES = TB / 16;
  static constexpr int WPP = (THREADS / 32) / PAGES;       // warps per page
  static constexpr int NT = (D / 8) / WPP;                 // n-tiles (8 outputs) per warp
  static constexpr int KS = D / 16;                        // k-steps (16 sketch rows; m = d)
  static constexpr size_t SMEM_TILES = (size_t)PAGES * TILE;
  // S^T (2 sigma - 1) as [token][i], rows padded by 8 floats so that the fragment stores of a
  // half-warp (rows g = 0..3 / 4..7, 8-byte pairs 2t) fall on 16 distinct bank pairs
  static constexpr int CORR_STRIDE = D + 8;
  static constexpr size_t SMEM_CORR = sizeof(float) * TB * CORR_STRIDE;
  static constexpr size_t SMEM = SMEM_TILES + SMEM_CORR;
};

template <int D, int VB, typename OUT>
__global__ void __launch_bounds__(256) dequant_main_kernel(DqArgs a) {
  using C = MainDq<D, VB>;
  OUT* k_out = static_cast<OUT*>(a.k_out);
  OUT* v_out = static_cast<OUT*>(a.v_out);
  constexpr int E = C::E;
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* tiles = smem;
  float* corr = reinterpret_cast<float*>(smem + C::SMEM_TILES);
  __shared__ bool ok[C::TB / 16];
  const int b = blockIdx.z, h = blockIdx.y;
  const int tok0 = blockIdx.x * C::TB;
  const int n = dq_ntok(a, b);
  if (tok0 >= n) return;
  const int ntok = min(C::TB, n - tok0);  // multiple of 16
  const int kb = a.kb, o_vq = 2 * kb * D, o_vsm = o_vq + 2 * VB * D, o_norm = o_vsm + 2 * D;
  load_tiles(a, tiles, C::TILE, o_norm + 64, b, h, tok0 >> 4, ntok >> 4, ok);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // corr[t][i] = sum_j (2 sigma_tj - 1) S[j][i]: warp -> (page, NT n-tiles); A = -(2 sigma - 1)
  {
    const int page = warp / C::WPP, nt0 = (warp % C::WPP) * C::NT;
    const int g = lane >> 2, t = lane & 3;
    if (page * 16 < ntok) {
      const uint32_t* ks0 = reinterpret_cast<const uint32_t*>(tiles + (size_t)page * C::TILE + 2 * (kb - 1) * D +
                                                             g * (D / 8));
      const uint32_t* ks1 = ks0 + 8 * (D / 32);  // token g + 8
      float acc[C::NT][4];
#pragma unroll
      for (int j = 0; j < C::NT; ++j)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[j][r] = 0.f;
#pragma unroll 2
      for (int ks = 0; ks < C::KS; ++ks) {
        const uint32_t w0 = ks0[ks >> 1], w1 = ks1[ks >> 1];
        const int jj = 8 * (ks & 1) + t;
        const uint32_t m0 = 1u << (15 - jj), m1 = 1u << (11 - jj);
        const uint32_t x00 = w0 * m0, x10 = w1 * m0, x01 = w0 * m1, x11 = w1 * m1;
        uint4 ah, al;  // bit set -> -1 (-2^-11), clear -> +1 (+2^-11)
        ah.x = (x00 & 0x80008000u) | 0x3C003C00u;
        ah.y = (x10 & 0x80008000u) | 0x3C003C00u;
        ah.z = (x01 & 0x80008000u) | 0x3C003C00u;
        ah.w = (x11 & 0x80008000u) | 0x3C003C00u;
        al.x = (x00 & 0x80008000u) | 0x10001000u;
        al.y = (x10 & 0x80008000u) | 0x10001000u;
        al.z = (x01 & 0x80008000u) | 0x10001000u;
        al.w = (x11 & 0x80008000u) | 0x10001000u;
        const uint4* bf = a.sfrag + ((size_t)ks * (D / 8) + nt0) * 32 + lane;
#pragma unroll
        for (int j = 0; j < C::NT; ++j) {
          const uint4 bv = __ldg(bf + j * 32);
          mma_f16_acc(acc[j], ah, bv.x, bv.y);
          mma_f16_acc(acc[j], al, bv.z, bv.w);
        }
      }
      float* c0 = corr + (page * 16 + g) * C::CORR_STRIDE;
      float* c1 = c0 + 8 * C::CORR_STRIDE;
#pragma unroll
      for (int j = 0; j < C::NT; ++j) {
        const int i = 8 * (nt0 + j) + 2 * t;
        *reinterpret_cast<float2*>(c0 + i) = make_float2(-acc[j][0], -acc[j][1]);
        *reinterpret_cast<float2*>(c1 + i) = make_float2(-acc[j][2], -acc[j][3]);
      }
    }
  }
  __syncthreads();

  // keys and values, one warp per token
  const float rs = rsqrtf((float)D);
  float sg[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sg[e] = a.signs[coord_of(e, lane)];
  for (int tt = warp; tt < ntok; tt += C::THREADS / 32) {
    if (!ok[tt >> 4]) continue;
    const uint8_t* tile = tiles + (size_t)(tt >> 4) * C::TILE;
    const int slot = tt & 15;
    const uint32_t* kh = reinterpret_cast<const uint32_t*>(tile + slot * (D / 8));
    const uint32_t* kl = reinterpret_cast<const uint32_t*>(tile + 2 * D + slot * (D / 8));
    const uint32_t* k3 = reinterpret_cast<const uint32_t*>(tile + 4 * D + slot * (D / 8));
    const float nk = __half2float(reinterpret_cast<const __half*>(tile + o_norm)[slot]);
    const float nr = __half2float(reinterpret_cast<const __half*>(tile + o_norm + 32)[slot]);
    const int bit = 16 * (lane >> 4) + (lane & 15);
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      // c[idx] by a select tree on the index bits as they come from the planes (high bit first)
      const bool i0 = (kh[e] >> bit) & 1u;
      const bool i1 = kb >= 3 && ((kl[e] >> bit) & 1u), i2 = kb == 4 && ((k3[e] >> bit) & 1u);
      x[e] = fmaf(a.qjl_coef * nr, corr[tt * C::CORR_STRIDE + coord_of(e, lane)], sel_bits(a.tab, kb, i0, i1, i2));
    }
    wht_warp<E>(x, lane);
    const size_t row = (((size_t)b * a.hkv + h) * a.max_tokens + tok0 + tt) * D;
    // 2-bit: token 2j+e at bits 16e+2j of word c; 4-bit: tokens 8w+2j+e at bits 16e+4j of word w*d+c
    const uint32_t* vq = reinterpret_cast<const uint32_t*>(tile + o_vq) + (VB == 4 && slot >= 8 ? D : 0);
    const int vbit = VB == 2 ? 16 * (slot & 1) + 2 * (slot >> 1) : 16 * (slot & 1) + 4 * ((slot & 7) >> 1);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = coord_of(e, lane);
      store_out(k_out + row + c, nk * (x[e] * sg[e] * rs));
      const __half2 smn = *reinterpret_cast<const __half2*>(tile + o_vsm + (slot * (D / 32) + e) * 4);
      const float q = (float)((vq[c] >> vbit) & ((1u << VB) - 1u));
      store_out(v_out + row + c, fmaf(__low2float(smn), q, __high2float(smn)));
    }
  }
}

// ------------------------------------------------------------------ alternate layout
// Alternate-layout page: alt_tile_bytes(d, kb, vb) for kb-bit key codes (or fp16 keys) and vb-bit
// value indices (staging sized for fp16 keys and vb = 4).
template <int D>
struct AltDq {
  static constexpr int E = D / 32;
  static constexpr int TB = 32;
  static constexpr int TILE_MAX = alt_tile_bytes(D, 16, 8);
  static constexpr int THREADS = 256;
  static constexpr size_t SMEM = (size_t)(TB / 16) * TILE_MAX;
};

// Key coordinate c of token `slot` of a staged alternate-layout page: the fp16 key itself (kb 16),
// or mn + s code with the code a byte (kb 8) or taken from the token's little-endian kb-bit stream.
template <int D>
__device__ __forceinline__ float alt_key(const uint8_t* tile, int o_ksm, int slot, int c, int kb) {
  if (kb == 16) return __half2float(reinterpret_cast<const __half*>(tile)[slot * D + c]);
  const __half2 smn = *reinterpret_cast<const __half2*>(tile + o_ksm + (slot * (D / 32) + (c >> 5)) * 4);
  int kq;
  if (kb == 8) {
    kq = tile[slot * D + c];
  } else {
    const uint32_t* kw = reinterpret_cast<const uint32_t*>(tile + slot * (kb * D / 8));
    const int kbit = kb * c;
    const uint32_t klo = kw[kbit >> 5];
    const uint32_t khi = (kbit & 31) + kb > 32 ? kw[(kbit >> 5) + 1] : 0u;
    kq = (int)(__funnelshift_r(klo, khi, kbit & 31) & ((1u << kb) - 1u));
  }
  return fmaf(__low2float(smn), (float)kq, __high2float(smn));
}

template <int D, typename OUT>
__global__ void __launch_bounds__(256) dequant_alt_kernel(DqArgs a) {
  using C = AltDq<D>;
  OUT* k_out = static_cast<OUT*>(a.k_out);
  OUT* v_out = static_cast<OUT*>(a.v_out);
  constexpr int E = C::E;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ bool ok[C::TB / 16];
  __shared__ float lut[256];
  const int b = blockIdx.z, h = blockIdx.y;
  const int tok0 = blockIdx.x * C::TB;
  const int n = dq_ntok(a, b);
  if (tok0 >= n) return;
  const int ntok = min(C::TB, n - tok0);
  const int vb = a.avb, kb = a.kb, tile_bytes = alt_tile_bytes(D, kb, vb);
  const int o_ksm = 2 * kb * D, o_vi = alt_key_bytes(D, kb), o_vn = o_vi + 2 * vb * D;
  const uint32_t mask = (1u << vb) - 1u;
  for (int i = threadIdx.x; i < (1 << vb); i += C::THREADS) lut[i] = a.vcent[i];
  load_tiles(a, smem, tile_bytes, tile_bytes, b, h, tok0 >> 4, ntok >> 4, ok);  // ends with __syncthreads
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float rs = rsqrtf((float)D);
  float sg[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sg[e] = a.signs[coord_of(e, lane)];
  for (int tt = warp; tt < ntok; tt += C::THREADS / 32) {
    if (!ok[tt >> 4]) continue;
    const uint8_t* tile = smem + (size_t)(tt >> 4) * tile_bytes;
    const int slot = tt & 15;
    const size_t row = (((size_t)b * a.hkv + h) * a.max_tokens + tok0 + tt) * D;
    const uint32_t* vi = reinterpret_cast<const uint32_t*>(tile + o_vi + slot * (vb * D / 8));
    const float nv = __half2float(reinterpret_cast<const __half*>(tile + o_vn)[slot]);
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = coord_of(e, lane);
      store_out(k_out + row + c, alt_key<D>(tile, o_ksm, slot, c, kb));
      const int bit = vb * c;  // index c of the token's little-endian vb-bit stream
      const uint32_t lo = vi[bit >> 5];
      const uint32_t hi = (bit & 31) + vb > 32 ? vi[(bit >> 5) + 1] : 0u;
      x[e] = lut[__funnelshift_r(lo, hi, bit & 31) & mask];
    }
    wht_warp<E>(x, lane);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = coord_of(e, lane);
      store_out(v_out + row + c, nv * (x[e] * sg[e] * rs));
    }
  }
}

// ------------------------------------------------------------------ exact recent buffer
// Ring slots 0 .. n_buf-1 hold positions n_tokens .. n_tokens + n_buf - 1.
template <typename OUT>
__global__ void __launch_bounds__(256) dequant_ring_kernel(DqArgs a, int d) {
  const int b = blockIdx.y, h = blockIdx.x;
  const int n = dq_ntok(a, b);
  int nb = a.n_buf[b];
  if (nb < 0 || nb > kRing || n + nb > a.max_tokens) {
    if (threadIdx.x == 0 && h == 0) flag_error(a.err, TQ_DEVERR_RING);
    return;
  }
  const size_t src = ((size_t)b * a.hkv + h) * kRing * d;
  const size_t dst = (((size_t)b * a.hkv + h) * a.max_tokens + n) * d;
  const int n16 = nb * d / 8;  // 16-byte chunks of fp16 (d is a multiple of 64)
  OUT* k_out = static_cast<OUT*>(a.k_out);
  OUT* v_out = static_cast<OUT*>(a.v_out);
  for (int i = threadIdx.x; i < n16; i += blockDim.x) {
    const uint4 kv = reinterpret_cast<const uint4*>(a.ring_k + src)[i];
    const uint4 vv = reinterpret_cast<const uint4*>(a.ring_v + src)[i];
    if (std::is_same<OUT, __half>::value) {  // fp16 rows are copied as they are
      reinterpret_cast<uint4*>(k_out + dst)[i] = kv;
      reinterpret_cast<uint4*>(v_out + dst)[i] = vv;
    } else {
      const __half* kh = reinterpret_cast<const __half*>(&kv);
      const __half* vh = reinterpret_cast<const __half*>(&vv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        store_out(k_out + dst + 8 * i + j, __half2float(kh[j]));
        store_out(v_out + dst + 8 * i + j, __half2float(vh[j]));
      }
    }
  }
}

template <typename C, typename K>
cudaError_t launch_dq(K kern, const DqArgs& a, int batch, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((a.max_tokens + C::TB - 1) / C::TB, a.hkv, batch);
  kern<<<grid, C::THREADS, C::SMEM, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

template <typename OUT>
cudaError_t launch_dequantize_t(tq_ctx* ctx, const void* pool, int num_blocks, const int32_t* block_table,
                                int max_blocks, const int32_t* n_tokens, const void* ring_k, const void* ring_v,
                                const int32_t* n_buf, int batch, int max_tokens, void* k_out, void* v_out,
                                cudaStream_t s) {
  DqArgs a{};
  a.pool = static_cast<const uint8_t*>(pool);
  a.num_blocks = num_blocks;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.n_tokens = n_tokens;
  a.ring_k = static_cast<const __half*>(ring_k);
  a.ring_v = static_cast<const __half*>(ring_v);
  a.n_buf = n_buf;
  a.max_tokens = max_tokens;
  a.k_out = k_out;
  a.v_out = v_out;
  a.hkv = ctx->cfg.num_kv_heads;
  a.signs = ctx->d_signs;
  a.sfrag = ctx->d_sfrag;
  a.kb = ctx->cfg.key_bits;
  a.avb = ctx->cfg.value_bits;
  a.tab = ctx->tab;
  a.vcent = ctx->d_vcent;
  a.qjl_coef = (float)(1.2533141373155003 / (double)ctx->cfg.qjl_m);
  a.err = ctx->d_err;
  const int d = ctx->cfg.head_dim;
  const bool main = ctx->cfg.layout == TQ_LAYOUT_MAIN;
  const int vb = ctx->cfg.value_bits;
  cudaError_t e = cudaErrorInvalidValue;
  if (max_tokens > 0) {
    switch (d) {
      case 64: e = main ? (vb == 4 ? launch_dq<MainDq<64, 4>>(dequant_main_kernel<64, 4, OUT>, a, batch, s)
                                  : launch_dq<MainDq<64, 2>>(dequant_main_kernel<64, 2, OUT>, a, batch, s))
                        : launch_dq<AltDq<64>>(dequant_alt_kernel<64, OUT>, a, batch, s); break;
      case 128: e = main ? (vb == 4 ? launch_dq<MainDq<128, 4>>(dequant_main_kernel<128, 4, OUT>, a, batch, s)
                                  : launch_dq<MainDq<128, 2>>(dequant_main_kernel<128, 2, OUT>, a, batch, s))
                         : launch_dq<AltDq<128>>(dequant_alt_kernel<128, OUT>, a, batch, s); break;
      case 256: e = main ? (vb == 4 ? launch_dq<MainDq<256, 4>>(dequant_main_kernel<256, 4, OUT>, a, batch, s)
                                  : launch_dq<MainDq<256, 2>>(dequant_main_kernel<256, 2, OUT>, a, batch, s))
                         : launch_dq<AltDq<256>>(dequant_alt_kernel<256, OUT>, a, batch, s); break;
      case 512: e = main ? (vb == 4 ? launch_dq<MainDq<512, 4>>(dequant_main_kernel<512, 4, OUT>, a, batch, s)
                                  : launch_dq<MainDq<512, 2>>(dequant_main_kernel<512, 2, OUT>, a, batch, s))
                         : launch_dq<AltDq<512>>(dequant_alt_kernel<512, OUT>, a, batch, s); break;
    }
    if (e != cudaSuccess) return e;
    ctx->launches++;
  }
  if (n_buf) {
    dequant_ring_kernel<OUT><<<dim3(a.hkv, batch), 256, 0, s>>>(a, d);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ctx->launches++;
  }
  return cudaSuccess;
}

cudaError_t launch_dequantize(tq_ctx* ctx, const void* pool, int num_blocks, const int32_t* block_table,
                              int max_blocks, const int32_t* n_tokens, const void* ring_k, const void* ring_v,
                              const int32_t* n_buf, int batch, int max_tokens, void* k_out, void* v_out,
                              bool bf16, cudaStream_t s) {
  return bf16 ? launch_dequantize_t<__nv_bfloat16>(ctx, pool, num_blocks, block_table, max_blocks, n_tokens, ring_k,
                                                   ring_v, n_buf, batch, max_tokens, k_out, v_out, s)
              : launch_dequantize_t<__half>(ctx, pool, num_blocks, block_table, max_blocks, n_tokens, ring_k, ring_v,
                                            n_buf, batch, max_tokens, k_out, v_out, s);
}

size_t sketch_frag_bytes(int d) { return (size_t)(d / 16) * (d / 8) * 32 * sizeof(uint4); }

cudaError_t build_sketch_frags(const float* sketch, int d, void* frag) {
  const int total = (d / 16) * (d / 8) * 32;
  sketch_frag_kernel<<<(total + 255) / 256, 256>>>(sketch, d, static_cast<uint4*>(frag));
  cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : cudaDeviceSynchronize();
}

}  // namespace tq
