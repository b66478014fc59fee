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
//   k^  = mn_b + s_b q ;  v^ = n_v * D (H c[idx]) / sqrt(d).
//
// One CTA handles TB tokens (whole pages) of one (sequence, KV head).  The
// QJL back-projection S^T (2 sigma - 1) of all TB tokens is a CTA-wide FP32
// product (S streamed row by row, the +-1 vectors from shared memory); the
// rest is warp-per-token work: codes from the bit planes, the butterfly in
// registers and shuffles, coalesced fp16 stores.  The exact recent buffer is
// appended after the compressed tokens by a copy kernel.
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
  __half* k_out;
  __half* v_out;
  int hkv;
  const float* signs;
  const float* sketch;  // [m][d]
  CodeTables tab;
  float qjl_coef;       // sqrt(pi/2) / m
  uint32_t* err;
};

// Compressed tokens of sequence b, validated against the block table and the output rows.
__device__ __forceinline__ int dq_ntok(const DqArgs& a, int b) {
  const int n = a.n_tokens[b];
  if (n < 0 || (n & 15) || n > a.max_blocks * kPage || n > a.max_tokens) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) flag_error(a.err, TQ_DEVERR_POSITION);
    return 0;
  }
  return n;
}

// Copies this CTA's pages into shared memory; returns false (and flags) if a block id is bad.
template <int TILE>
__device__ bool load_tiles(const DqArgs& a, uint8_t* tiles, int b, int h, int page0, int npages, bool* ok) {
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
    const uint4* src = reinterpret_cast<const uint4*>(a.pool + ((size_t)blk * a.hkv + h) * TILE);
    uint4* dst = reinterpret_cast<uint4*>(tiles + (size_t)p * TILE);
    for (int i = threadIdx.x; i < TILE / 16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  return true;
}

// ------------------------------------------------------------------ main layout
template <int D>
struct MainDq {
  static constexpr int E = D / 32;
  static constexpr int TB = D >= 512 ? 16 : 32;          // tokens per CTA
  static constexpr int TILE = 12 * D + 64;
  static constexpr int THREADS = 256;
  static constexpr int IPT = D > THREADS ? D / THREADS : 1;  // outputs i per thread
  static constexpr int NSL = D >= THREADS ? 1 : THREADS / D;  // token slices
  static constexpr int TPS = TB / NSL;                     // tokens per slice
  static constexpr size_t SMEM_TILES = (size_t)(TB / 16) * TILE;
  static constexpr size_t SMEM_PM = sizeof(float) * D * TB;   // (2 sigma - 1) as [j][token]
  static constexpr size_t SMEM_CORR = sizeof(float) * TB * D; // S^T (2 sigma - 1) as [token][i]
  static constexpr size_t SMEM = SMEM_TILES + SMEM_PM + SMEM_CORR;
};

template <int D>
__global__ void __launch_bounds__(256) dequant_main_kernel(DqArgs a) {
  using C = MainDq<D>;
  constexpr int E = C::E;
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* tiles = smem;
  float* pmT = reinterpret_cast<float*>(smem + C::SMEM_TILES);
  float* corr = reinterpret_cast<float*>(smem + C::SMEM_TILES + C::SMEM_PM);
  __shared__ bool ok[C::TB / 16];
  const int b = blockIdx.z, h = blockIdx.y;
  const int tok0 = blockIdx.x * C::TB;
  const int n = dq_ntok(a, b);
  if (tok0 >= n) return;
  const int ntok = min(C::TB, n - tok0);  // multiple of 16
  load_tiles<C::TILE>(a, tiles, b, h, tok0 >> 4, ntok >> 4, ok);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // (2 sigma - 1) of every token, transposed: pmT[j][t]; tokens past ntok are 0
  for (int tt = warp; tt < C::TB; tt += C::THREADS / 32) {
    const uint32_t* ks = reinterpret_cast<const uint32_t*>(tiles + (size_t)(tt >> 4) * C::TILE + 4 * D +
                                                           (tt & 15) * (D / 8));
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float pm = 0.f;
      if (tt < ntok) pm = (ks[e] >> (16 * (lane >> 4) + (lane & 15))) & 1u ? 1.f : -1.f;
      pmT[coord_of(e, lane) * C::TB + tt] = pm;
    }
  }
  __syncthreads();

  // corr[t][i] = sum_j S[j][i] pm[t][j]
  {
    const int slice = threadIdx.x / (C::THREADS / C::NSL);
    const int i0 = threadIdx.x % (C::THREADS / C::NSL);
    const int t0 = slice * C::TPS;
    float acc[C::IPT][C::TPS];
#pragma unroll
    for (int u = 0; u < C::IPT; ++u)
#pragma unroll
      for (int t = 0; t < C::TPS; ++t) acc[u][t] = 0.f;
    for (int j = 0; j < D; ++j) {
      float sv[C::IPT];
#pragma unroll
      for (int u = 0; u < C::IPT; ++u) sv[u] = __ldg(a.sketch + (size_t)j * D + i0 + u * (D / C::IPT));
      const float* pj = pmT + j * C::TB + t0;
#pragma unroll
      for (int t4 = 0; t4 < C::TPS; t4 += 4) {
        const float4 p4 = *reinterpret_cast<const float4*>(pj + t4);
#pragma unroll
        for (int u = 0; u < C::IPT; ++u) {
          acc[u][t4] = fmaf(sv[u], p4.x, acc[u][t4]);
          acc[u][t4 + 1] = fmaf(sv[u], p4.y, acc[u][t4 + 1]);
          acc[u][t4 + 2] = fmaf(sv[u], p4.z, acc[u][t4 + 2]);
          acc[u][t4 + 3] = fmaf(sv[u], p4.w, acc[u][t4 + 3]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < C::IPT; ++u)
#pragma unroll
      for (int t = 0; t < C::TPS; ++t) corr[(t0 + t) * D + i0 + u * (D / C::IPT)] = acc[u][t];
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
    const float nk = __half2float(reinterpret_cast<const __half*>(tile + 12 * D)[slot]);
    const float nr = __half2float(reinterpret_cast<const __half*>(tile + 12 * D + 32)[slot]);
    const int bit = 16 * (lane >> 4) + (lane & 15);
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int idx = (int)(((kh[e] >> bit) & 1u) << 1 | ((kl[e] >> bit) & 1u));
      x[e] = fmaf(a.qjl_coef * nr, corr[tt * D + coord_of(e, lane)], sel4(a.tab, idx));
    }
    wht_warp<E>(x, lane);
    const size_t row = (((size_t)b * a.hkv + h) * a.max_tokens + tok0 + tt) * D;
    const uint32_t* vq = reinterpret_cast<const uint32_t*>(tile + 6 * D);
    const int vbit = 16 * (slot & 1) + 2 * (slot >> 1);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = coord_of(e, lane);
      a.k_out[row + c] = __float2half_rn(nk * (x[e] * sg[e] * rs));
      const __half2 smn = *reinterpret_cast<const __half2*>(tile + 10 * D + (slot * (D / 32) + e) * 4);
      const float q = (float)((vq[c] >> vbit) & 3u);
      a.v_out[row + c] = __float2half_rn(fmaf(__low2float(smn), q, __high2float(smn)));
    }
  }
}

// ------------------------------------------------------------------ alternate layout
template <int D>
struct AltDq {
  static constexpr int E = D / 32;
  static constexpr int TB = 32;
  static constexpr int TILE = 24 * D + 32;
  static constexpr int THREADS = 256;
  static constexpr size_t SMEM = (size_t)(TB / 16) * TILE;
};

template <int D>
__global__ void __launch_bounds__(256) dequant_alt_kernel(DqArgs a) {
  using C = AltDq<D>;
  constexpr int E = C::E;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ bool ok[C::TB / 16];
  const int b = blockIdx.z, h = blockIdx.y;
  const int tok0 = blockIdx.x * C::TB;
  const int n = dq_ntok(a, b);
  if (tok0 >= n) return;
  const int ntok = min(C::TB, n - tok0);
  load_tiles<C::TILE>(a, smem, b, h, tok0 >> 4, ntok >> 4, ok);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float rs = rsqrtf((float)D);
  float sg[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sg[e] = a.signs[coord_of(e, lane)];
  for (int tt = warp; tt < ntok; tt += C::THREADS / 32) {
    if (!ok[tt >> 4]) continue;
    const uint8_t* tile = smem + (size_t)(tt >> 4) * C::TILE;
    const int slot = tt & 15;
    const size_t row = (((size_t)b * a.hkv + h) * a.max_tokens + tok0 + tt) * D;
    const uint32_t* vi = reinterpret_cast<const uint32_t*>(tile + 18 * D + slot * (3 * D / 8));
    const float nv = __half2float(reinterpret_cast<const __half*>(tile + 24 * D)[slot]);
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = coord_of(e, lane);
      const __half2 smn = *reinterpret_cast<const __half2*>(tile + 16 * D + (slot * (D / 32) + e) * 4);
      a.k_out[row + c] = __float2half_rn(fmaf(__low2float(smn), (float)tile[slot * D + c], __high2float(smn)));
      const int bit = 3 * c;
      const uint32_t lo = vi[bit >> 5];
      const uint32_t hi = (bit & 31) > 29 ? vi[(bit >> 5) + 1] : 0u;
      const int idx = (int)(__funnelshift_r(lo, hi, bit & 31) & 7u);
      float cv = a.tab.c[0];
#pragma unroll
      for (int j = 1; j < 8; ++j) cv = idx == j ? a.tab.c[j] : cv;
      x[e] = cv;
    }
    wht_warp<E>(x, lane);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = coord_of(e, lane);
      a.v_out[row + c] = __float2half_rn(nv * (x[e] * sg[e] * rs));
    }
  }
}

// ------------------------------------------------------------------ exact recent buffer
// Ring slots 0 .. n_buf-1 hold positions n_tokens .. n_tokens + n_buf - 1.
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
  const int n16 = nb * d / 8;  // 16-byte chunks (d is a multiple of 64)
  for (int i = threadIdx.x; i < n16; i += blockDim.x) {
    reinterpret_cast<uint4*>(a.k_out + dst)[i] = reinterpret_cast<const uint4*>(a.ring_k + src)[i];
    reinterpret_cast<uint4*>(a.v_out + dst)[i] = reinterpret_cast<const uint4*>(a.ring_v + src)[i];
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

cudaError_t launch_dequantize(tq_ctx* ctx, const void* pool, int num_blocks, const int32_t* block_table,
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
  a.k_out = static_cast<__half*>(k_out);
  a.v_out = static_cast<__half*>(v_out);
  a.hkv = ctx->cfg.num_kv_heads;
  a.signs = ctx->d_signs;
  a.sketch = ctx->d_sketch;
  a.tab = ctx->tab;
  a.qjl_coef = (float)(1.2533141373155003 / (double)ctx->cfg.qjl_m);
  a.err = ctx->d_err;
  const int d = ctx->cfg.head_dim;
  const bool main = ctx->cfg.layout == TQ_LAYOUT_MAIN;
  cudaError_t e = cudaErrorInvalidValue;
  if (max_tokens > 0) {
    switch (d) {
      case 64: e = main ? launch_dq<MainDq<64>>(dequant_main_kernel<64>, a, batch, s)
                        : launch_dq<AltDq<64>>(dequant_alt_kernel<64>, a, batch, s); break;
      case 128: e = main ? launch_dq<MainDq<128>>(dequant_main_kernel<128>, a, batch, s)
                         : launch_dq<AltDq<128>>(dequant_alt_kernel<128>, a, batch, s); break;
      case 256: e = main ? launch_dq<MainDq<256>>(dequant_main_kernel<256>, a, batch, s)
                         : launch_dq<AltDq<256>>(dequant_alt_kernel<256>, a, batch, s); break;
      case 512: e = main ? launch_dq<MainDq<512>>(dequant_main_kernel<512>, a, batch, s)
                         : launch_dq<AltDq<512>>(dequant_alt_kernel<512>, a, batch, s); break;
    }
    if (e != cudaSuccess) return e;
    ctx->launches++;
  }
  if (n_buf) {
    dequant_ring_kernel<<<dim3(a.hkv, batch), 256, 0, s>>>(a, d);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ctx->launches++;
  }
  return cudaSuccess;
}

}  // namespace tq
