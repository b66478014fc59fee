// Read path: fused decode attention straight from the packed pages.
//
//  1. prep   (main layout) q_r = H (D q) / sqrt(d) and t = S q_r once per
//            query head ("TurboQuant-MLX overview", GPU kernel section:
//            pre-rotated q scoring).
//  2. decode split-K over (part, KV-head group, sequence).  Parts 0..n-1
//            cover fixed-size chunks of compressed tokens, part n the exact
//            recent buffer.  Per page of 16 tokens: stage the tile in shared
//            memory, score every token from its packed bits (no fp16
//            intermediate in global memory; framework-status survey, oMLX
//            fused two-pass kernel), update the online softmax with
//            shuffle reductions ("TurboQuant-MLX overview": SIMD-group sums),
//            accumulate values.  All n_rep query heads of the KV head share
//            one pass over the bytes (GQA via n_rep).
//            Main:  logit = n_k (<q_r, c[idx]> + sqrt(pi/2)/m n_r <t, 2 sigma - 1>) / sqrt(d)
//                   o += p (mn_g + s_g q)          (mn part summed once per group)
//            Alt:   logit = sum_blocks s_b <q_b, code_b> + mn_b sum(q_b), / sqrt(d)
//                   (fp16 keys: <q, k> / sqrt(d))
//                   o_rot += p n_v c[idx], one inverse rotation per chunk
//                   ("TurboQuant-MLX overview": butterfly pulled out of the V sum)
//  3. merge  o = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i per query head.
#include "common.cuh"
#include "tc.cuh"

namespace tq {

bool alt_v2_supported(const tq_ctx* ctx);
cudaError_t launch_decode_alt_v2(tq_ctx* ctx, const void* q, const void* pool, int num_blocks,
                                 const int32_t* block_table, int max_blocks, const int32_t* n_compressed, int max_ctx,
                                 float* parts, int chunk_tokens, int n_chunks, int n_parts, int batch, cudaStream_t s);

namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct DecArgs {
  const __half* q;
  int batch;
  const uint8_t* pool;
  int num_blocks;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* n_compressed;
  const __half* ring_k;
  const __half* ring_v;
  const int32_t* n_buf;
  int max_ctx;
  float* out;
  float* qprep;  // [B][Hq][2d] (main)
  float* parts;  // [B][Hq][n_parts][d + 2]
  int chunk_tokens, n_chunks, n_parts;
  int first_part;  // blockIdx.x + first_part = part index
  int hq, hkv, n_rep, nrg, groups;
  const float* signs;
  const float* sketch_t;
  int kb;  // main layout key bits (3 or 2)
  int avb;  // alternate layout value index bits (2 .. 8)
  CodeTables tab;
  const float* vcent;  // alternate layout: value centroids in device memory (2^avb of them)
  uint32_t* err;
};

__device__ __forceinline__ int seq_nc(const DecArgs& a, int b) {
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

__device__ __forceinline__ int seq_nb(const DecArgs& a, int b) {
  if (!a.n_buf) return 0;
  const int nb = a.n_buf[b];
  if (nb < 0 || nb > kRing) {
    if (threadIdx.x == 0) flag_error(a.err, TQ_DEVERR_RING);
    return 0;
  }
  return nb;
}

// ------------------------------------------------------------------ prep
template <int D>
__global__ void __launch_bounds__(32) prep_main_kernel(DecArgs a) {
  constexpr int E = D / 32;
  __shared__ float qr[D];
  const int h = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
  const __half* qp = a.q + ((size_t)b * a.hq + h) * D;
  float x[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int c = coord_of(e, lane);
    x[e] = __half2float(qp[c]) * a.signs[c];
  }
  wht_warp<E>(x, lane);
  const float sc = rsqrtf((float)D);
  float* dst = a.qprep + ((size_t)b * a.hq + h) * 2 * D;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int c = coord_of(e, lane);
    qr[c] = x[e] * sc;
    dst[c] = x[e] * sc;
  }
  __syncwarp();
  for (int j = lane; j < D; j += 32) {
    float t = 0.f;
    for (int i = 0; i < D; ++i) t = fmaf(__ldg(a.sketch_t + (size_t)i * D + j), qr[i], t);
    dst[D + j] = t;
  }
}

// ------------------------------------------------------------------ shared pieces
template <int NR>
struct SoftState {
  float m[NR], l[NR], alpha[NR];
};

// Online-softmax update for one page of 16 tokens, executed by all 128
// threads (h = tid >> 4, tok = tid & 15; heads >= nrg are padding).  sc holds
// log2-domain logits (-inf = absent token).  Writes p into pbuf[tok][h] and
// updates the running maximum, sum and rescale factor of each head.
template <int NR>
__device__ __forceinline__ void softmax_page(const float (*sc)[16], float (*pbuf)[NR], SoftState<NR>& st, int nrg) {
  const int h = threadIdx.x >> 4, tok = threadIdx.x & 15;
  const bool act = h < nrg;
  const float s = act ? sc[h][tok] : -INFINITY;
  float mx = s;
#pragma unroll
  for (int m = 8; m; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m, 16));
  const float m_old = act ? st.m[h] : -INFINITY;
  const float m_new = fmaxf(m_old, mx);
  float p = 0.f, alpha = 1.f;
  if (act && m_new != -INFINITY) {
    p = exp2f(s - m_new);
    alpha = exp2f(m_old - m_new);
  }
  float ps = p;
#pragma unroll
  for (int m = 8; m; m >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, m, 16);
  if (h < NR) {
    pbuf[tok][h] = p;
    if (tok == 0) {
      if (act) {
        st.m[h] = m_new;
        st.l[h] = st.l[h] * alpha + ps;
      }
      st.alpha[h] = alpha;
    }
  }
}

// Exact fp16 recent-buffer part: tokens 0..nb-1 of ring[b][kvh].
template <int D, int NR>
__device__ void ring_part(const DecArgs& a, int b, int kvh, int h0, int nb, float (*qf)[D], float (*sc)[16],
                          float (*pbuf)[NR], SoftState<NR>& st, float (&o)[(D + 127) / 128][NR]) {
  constexpr int DPT = (D + 127) / 128;
  const int tid = threadIdx.x;
  const float scale = rsqrtf((float)D) * kLog2e;
  const __half* rk = a.ring_k + ((size_t)b * a.hkv + kvh) * kRing * D;
  const __half* rv = a.ring_v + ((size_t)b * a.hkv + kvh) * kRing * D;
  for (int t0 = 0; t0 < nb; t0 += 16) {
    const int tok = tid >> 3, pp = tid & 7;
    float acc[NR];
#pragma unroll
    for (int h = 0; h < NR; ++h) acc[h] = 0.f;
    if (t0 + tok < nb) {
      const __half* kp = rk + (size_t)(t0 + tok) * D;
      for (int k = 0; k < D / 8; ++k) {
        const int dim = pp * (D / 8) + k;
        const float kv = __half2float(kp[dim]);
#pragma unroll
        for (int h = 0; h < NR; ++h) acc[h] = fmaf(qf[h][dim], kv, acc[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < NR; ++h) {
#pragma unroll
      for (int m = 1; m < 8; m <<= 1) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], m);
    }
    if (pp == 0) {
#pragma unroll
      for (int h = 0; h < NR; ++h) sc[h][tok] = (t0 + tok < nb) ? acc[h] * scale : -INFINITY;
    }
    __syncthreads();
    softmax_page<NR>(sc, pbuf, st, a.nrg);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < DPT; ++r) {
      const int i = tid + 128 * r;
      if (i < D) {
#pragma unroll
        for (int h = 0; h < NR; ++h) o[r][h] *= st.alpha[h];
        const int cnt = min(16, nb - t0);
        for (int tk = 0; tk < cnt; ++tk) {
          const float vv = __half2float(rv[(size_t)(t0 + tk) * D + i]);
#pragma unroll
          for (int h = 0; h < NR; ++h) o[r][h] = fmaf(pbuf[tk][h], vv, o[r][h]);
        }
      }
    }
    __syncthreads();
  }
}

template <int D, int NR>
__device__ void write_part(const DecArgs& a, int b, int h0, int part, const SoftState<NR>& st,
                           const float (&o)[(D + 127) / 128][NR], const float (*msum)[D / 32]) {
  constexpr int DPT = (D + 127) / 128;
#pragma unroll
  for (int h = 0; h < NR; ++h) {
    if (h >= a.nrg) break;
    float* dst = a.parts + (((size_t)b * a.hq + h0 + h) * a.n_parts + part) * (D + 2);
#pragma unroll
    for (int r = 0; r < DPT; ++r) {
      const int i = threadIdx.x + 128 * r;
      if (i < D) dst[i] = o[r][h] + (msum ? msum[h][i >> 5] : 0.f);
    }
    if (threadIdx.x == 0) {
      dst[D] = st.m[h];
      dst[D + 1] = st.l[h];
    }
  }
}

// ------------------------------------------------------------------ main layout
// VB = value bits (2 or 4): value codes take VB * d / 8 bytes per token.  The key bits (2, 3 or 4:
// kb - 1 Lloyd-Max index planes before the QJL plane) are a run-time value; the page buffer is
// sized for 4.
template <int D, int NR, int VB>
struct MainDec {
  static constexpr int TILE = (10 + 2 * VB) * D + 64;
  static constexpr int G = D / 32;
};

template <int D, int NR, int VB>
__global__ void __launch_bounds__(128) decode_main_kernel(DecArgs a) {
  using C = MainDec<D, NR, VB>;
  constexpr int G = C::G;
  constexpr int DPT = (D + 127) / 128;
  __shared__ float qr[NR][D];
  __shared__ float qt[NR][D];
  extern __shared__ __align__(16) uint8_t tile[];  // one page of one KV head (C::TILE bytes)
  __shared__ float sc[NR][16];
  __shared__ float pbuf[16][NR];
  __shared__ float pw[G][16][NR];
  __shared__ float msum[NR][G];
  __shared__ SoftState<NR> st;

  const int part = blockIdx.x + a.first_part, hg = blockIdx.y, b = blockIdx.z;
  const int kvh = hg / a.groups;
  const int h0 = kvh * a.n_rep + (hg % a.groups) * a.nrg;
  const int tid = threadIdx.x;
  const int nc = seq_nc(a, b);
  const int nb = seq_nb(a, b);
  int tbeg = 0, tend = 0;
  const bool ring = part == a.n_chunks;
  if (ring) {
    if (nb == 0) return;
  } else {
    tbeg = part * a.chunk_tokens;
    tend = min(nc, tbeg + a.chunk_tokens);
    if (tbeg >= tend) return;
  }
  if (tid < NR) {
    st.m[tid] = -INFINITY;
    st.l[tid] = 0.f;
    st.alpha[tid] = 1.f;
  }
  for (int i = tid; i < NR * G; i += 128) msum[i / G][i % G] = 0.f;
  // stage the queries: pre-rotated (compressed part) or raw (ring part)
  for (int i = tid; i < NR * D; i += 128) {
    const int h = i / D, c = i % D;
    float vr = 0.f, vt = 0.f;
    if (h < a.nrg) {
      if (ring) {
        vr = __half2float(a.q[((size_t)b * a.hq + h0 + h) * D + c]);
      } else {
        const float* src = a.qprep + ((size_t)b * a.hq + h0 + h) * 2 * D;
        vr = src[c];
        vt = src[D + c];
      }
    }
    qr[h][c] = vr;
    qt[h][c] = vt;
  }
  float o[DPT][NR];
#pragma unroll
  for (int r = 0; r < DPT; ++r)
#pragma unroll
    for (int h = 0; h < NR; ++h) o[r][h] = 0.f;
  __syncthreads();

  if (ring) {
    ring_part<D, NR>(a, b, kvh, h0, nb, qr, sc, pbuf, st, o);
    write_part<D, NR>(a, b, h0, a.n_chunks, st, o, nullptr);
    return;
  }

  const float coef = 1.2533141373155003f / (float)D;  // sqrt(pi/2) / m, m = d
  const float scale = rsqrtf((float)D) * kLog2e;
  const int kb = a.kb, tile_bytes = (2 * kb + 2 * VB + 2) * D + 64;
  const uint32_t* kh_w = reinterpret_cast<const uint32_t*>(tile);
  const uint32_t* kl_w = reinterpret_cast<const uint32_t*>(tile + 2 * D);  // 3- and 4-bit keys
  const uint32_t* k3_w = reinterpret_cast<const uint32_t*>(tile + 4 * D);  // 4-bit keys
  const uint32_t* ks_w = reinterpret_cast<const uint32_t*>(tile + 2 * (kb - 1) * D);
  const uint32_t* vq_w = reinterpret_cast<const uint32_t*>(tile + 2 * kb * D);
  const __half* vsm = reinterpret_cast<const __half*>(tile + (2 * kb + 2 * VB) * D);
  const __half* kn = reinterpret_cast<const __half*>(tile + (2 * kb + 2 * VB + 2) * D);
  const __half* rn = kn + 16;

  for (int t0 = tbeg; t0 < tend; t0 += kPage) {
    const int page = t0 >> 4;
    const int blk = a.block_table[(size_t)b * a.max_blocks + page];
    if (blk < 0 || blk >= a.num_blocks) {
      if (tid == 0) flag_error(a.err, TQ_DEVERR_BLOCK_ID);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(a.pool + ((size_t)blk * a.hkv + kvh) * tile_bytes);
    for (int i = tid; i < tile_bytes / 16; i += 128) reinterpret_cast<uint4*>(tile)[i] = src[i];
    __syncthreads();
    // ---- scores: 8 threads per token
    {
      const int tok = tid >> 3, pp = tid & 7;
      float lm[NR], qj[NR];
#pragma unroll
      for (int h = 0; h < NR; ++h) lm[h] = qj[h] = 0.f;
      const uint32_t* khr = kh_w + tok * (D / 32);
      const uint32_t* klr = kl_w + tok * (D / 32);
      const uint32_t* k3r = k3_w + tok * (D / 32);
      const uint32_t* ksr = ks_w + tok * (D / 32);
#pragma unroll 4
      for (int k = 0; k < D / 8; ++k) {
        const int dim = pp * (D / 8) + k;
        const int w = dim >> 5, bp = 16 * (dim & 1) + ((dim & 31) >> 1);
        const bool i0 = (khr[w] >> bp) & 1;
        const bool i1 = kb >= 3 && ((klr[w] >> bp) & 1), i2 = kb == 4 && ((k3r[w] >> bp) & 1);
        const float cv = sel_bits(a.tab, kb, i0, i1, i2);
        const float sv = ((ksr[w] >> bp) & 1) ? 1.f : -1.f;
#pragma unroll
        for (int h = 0; h < NR; ++h) {
          lm[h] = fmaf(qr[h][dim], cv, lm[h]);
          qj[h] = fmaf(qt[h][dim], sv, qj[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < NR; ++h) {
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) {
          lm[h] += __shfl_xor_sync(0xffffffffu, lm[h], m);
          qj[h] += __shfl_xor_sync(0xffffffffu, qj[h], m);
        }
      }
      if (pp == 0) {
        const float nkv = __half2float(kn[tok]), nrv = __half2float(rn[tok]);
#pragma unroll
        for (int h = 0; h < NR; ++h) sc[h][tok] = nkv * (lm[h] + coef * nrv * qj[h]) * scale;
      }
    }
    __syncthreads();
    softmax_page<NR>(sc, pbuf, st, a.nrg);
    __syncthreads();
    // per (tok, head): weights p * s_g and the running sum of p * mn_g (all threads shuffle)
    {
      const int h = tid >> 4, tok = tid & 15;
      const bool hv = h < NR;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float p = hv ? pbuf[tok][h] : 0.f;
        const float s = __half2float(vsm[(tok * G + g) * 2]);
        const float mn = __half2float(vsm[(tok * G + g) * 2 + 1]);
        if (hv) pw[g][tok][h] = p * s;
        float pm = p * mn;
#pragma unroll
        for (int m = 8; m; m >>= 1) pm += __shfl_xor_sync(0xffffffffu, pm, m, 16);
        if (hv && tok == 0) msum[h][g] = msum[h][g] * st.alpha[h] + pm;
      }
    }
    __syncthreads();
    // ---- values: one thread per dimension
#pragma unroll
    for (int r = 0; r < DPT; ++r) {
      const int i = tid + 128 * r;
      if (i < D) {
        const int g = i >> 5;
        // 2-bit: token 2j+e at bits 16e+2j of word i; 4-bit: tokens 8w+2j+e at bits 16e+4j of
        // word w*d + i
        const uint32_t w = vq_w[i];
        const uint32_t w1 = VB == 4 ? vq_w[D + i] : 0u;
#pragma unroll
        for (int h = 0; h < NR; ++h) o[r][h] *= st.alpha[h];
#pragma unroll
        for (int tk = 0; tk < 16; ++tk) {
          const float cf = VB == 2 ? (float)((w >> (16 * (tk & 1) + 2 * (tk >> 1))) & 3u)
                                   : (float)(((tk < 8 ? w : w1) >> (16 * (tk & 1) + 4 * ((tk & 7) >> 1))) & 15u);
#pragma unroll
          for (int h = 0; h < NR; ++h) o[r][h] = fmaf(pw[g][tk][h], cf, o[r][h]);
        }
      }
    }
    __syncthreads();
  }
  write_part<D, NR>(a, b, h0, part, st, o, msum);
}

// ------------------------------------------------------------------ alternate layout
template <int D, int NR>
__global__ void __launch_bounds__(128) decode_alt_kernel(DecArgs a) {
  // page: alt_tile_bytes(D, kb, vb) for kb-bit key codes (or fp16 keys) and vb-bit value
  // indices, staged in dynamic shared memory
  constexpr int G = D / 32;
  constexpr int DPT = (D + 127) / 128;
  constexpr int E = D / 32;
  __shared__ float qf[NR][D];
  __shared__ float qsum[NR][G];
  extern __shared__ __align__(16) uint8_t tile[];
  __shared__ float sc[NR][16];
  __shared__ float pbuf[16][NR];
  __shared__ float ob[NR][D];
  __shared__ SoftState<NR> st;
  __shared__ float vlut[256];  // value centroids (2^avb used)

  const int part = blockIdx.x + a.first_part, hg = blockIdx.y, b = blockIdx.z;
  const int kvh = hg / a.groups;
  const int h0 = kvh * a.n_rep + (hg % a.groups) * a.nrg;
  const int tid = threadIdx.x;
  const int nc = seq_nc(a, b);
  const int nb = seq_nb(a, b);
  int tbeg = 0, tend = 0;
  const bool ring = part == a.n_chunks;
  if (ring) {
    if (nb == 0) return;
  } else {
    tbeg = part * a.chunk_tokens;
    tend = min(nc, tbeg + a.chunk_tokens);
    if (tbeg >= tend) return;
  }
  if (tid < NR) {
    st.m[tid] = -INFINITY;
    st.l[tid] = 0.f;
    st.alpha[tid] = 1.f;
  }
  for (int i = tid; i < (1 << a.avb); i += 128) vlut[i] = a.vcent[i];
  for (int i = tid; i < NR * D; i += 128) {
    const int h = i / D, c = i % D;
    qf[h][c] = h < a.nrg ? __half2float(a.q[((size_t)b * a.hq + h0 + h) * D + c]) : 0.f;
  }
  __syncthreads();
  for (int i = tid; i < NR * G; i += 128) {
    const int h = i / G, g = i % G;
    float s = 0.f;
    for (int c = 0; c < 32; ++c) s += qf[h][g * 32 + c];
    qsum[h][g] = s;
  }
  float o[DPT][NR];
#pragma unroll
  for (int r = 0; r < DPT; ++r)
#pragma unroll
    for (int h = 0; h < NR; ++h) o[r][h] = 0.f;
  __syncthreads();

  if (ring) {
    ring_part<D, NR>(a, b, kvh, h0, nb, qf, sc, pbuf, st, o);
    write_part<D, NR>(a, b, h0, a.n_chunks, st, o, nullptr);
    return;
  }

  const float scale = rsqrtf((float)D) * kLog2e;
  const int vb = a.avb, kb = a.kb, TILE = alt_tile_bytes(D, kb, vb);
  const uint32_t vmask = (1u << vb) - 1u;
  const __half* ksm = reinterpret_cast<const __half*>(tile + 2 * kb * D);  // (scale, minimum); none for fp16 keys
  const uint32_t* vi = reinterpret_cast<const uint32_t*>(tile + alt_key_bytes(D, kb));
  const __half* vn = reinterpret_cast<const __half*>(tile + alt_key_bytes(D, kb) + 2 * vb * D);

  for (int t0 = tbeg; t0 < tend; t0 += kPage) {
    const int page = t0 >> 4;
    const int blk = a.block_table[(size_t)b * a.max_blocks + page];
    if (blk < 0 || blk >= a.num_blocks) {
      if (tid == 0) flag_error(a.err, TQ_DEVERR_BLOCK_ID);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(a.pool + ((size_t)blk * a.hkv + kvh) * TILE);
    for (int i = tid; i < TILE / 16; i += 128) reinterpret_cast<uint4*>(tile)[i] = src[i];
    __syncthreads();
    {
      const int tok = tid >> 3, pp = tid & 7;
      float acc[NR];
#pragma unroll
      for (int h = 0; h < NR; ++h) acc[h] = 0.f;
      const uint8_t* kq = tile + tok * (kb * D / 8);  // the token's key codes (a kb-bit stream) or fp16 keys
      const __half* kh = reinterpret_cast<const __half*>(kq);
      const uint32_t* kw = reinterpret_cast<const uint32_t*>(kq);
      const uint32_t kmask = (1u << kb) - 1u;
      // D/8 dims per thread, inside whole 32-blocks or half of one
      constexpr int SEG = D / 8 < 32 ? D / 8 : 32;
#pragma unroll
      for (int s0 = 0; s0 < D / 8; s0 += SEG) {
        const int dim0 = pp * (D / 8) + s0;
        const int g = dim0 >> 5;
        float part_acc[NR];
#pragma unroll
        for (int h = 0; h < NR; ++h) part_acc[h] = 0.f;
#pragma unroll 8
        for (int k = 0; k < SEG; ++k) {
          const int i = dim0 + k;
          float cv;
          if (kb == 16) {
            cv = __half2float(kh[i]);
          } else if (kb == 8) {
            cv = (float)kq[i];
          } else {
            const int kbit = kb * i;
            const uint32_t klo = kw[kbit >> 5];
            const uint32_t khi = (kbit & 31) + kb > 32 ? kw[(kbit >> 5) + 1] : 0u;
            cv = (float)(__funnelshift_r(klo, khi, kbit & 31) & kmask);
          }
#pragma unroll
          for (int h = 0; h < NR; ++h) part_acc[h] = fmaf(qf[h][dim0 + k], cv, part_acc[h]);
        }
        const float s = kb == 16 ? 1.f : __half2float(ksm[(tok * G + g) * 2]);
        const float mn = kb == 16 ? 0.f : __half2float(ksm[(tok * G + g) * 2 + 1]);
        float qs[NR];
        if (SEG == 32) {
#pragma unroll
          for (int h = 0; h < NR; ++h) qs[h] = qsum[h][g];
        } else {
#pragma unroll
          for (int h = 0; h < NR; ++h) {
            float t = 0.f;
            for (int k = 0; k < SEG; ++k) t += qf[h][dim0 + k];
            qs[h] = t;
          }
        }
#pragma unroll
        for (int h = 0; h < NR; ++h) acc[h] += s * part_acc[h] + mn * qs[h];
      }
#pragma unroll
      for (int h = 0; h < NR; ++h) {
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], m);
      }
      if (pp == 0) {
#pragma unroll
        for (int h = 0; h < NR; ++h) sc[h][tok] = acc[h] * scale;
      }
    }
    __syncthreads();
    softmax_page<NR>(sc, pbuf, st, a.nrg);
    __syncthreads();
    {
      const int h = tid >> 4, tok = tid & 15;
      if (h < NR) pbuf[tok][h] *= __half2float(vn[tok]);
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < DPT; ++r) {
      const int i = tid + 128 * r;
      if (i < D) {
#pragma unroll
        for (int h = 0; h < NR; ++h) o[r][h] *= st.alpha[h];
        const int bit = vb * i;  // index i of each token's little-endian vb-bit stream
        for (int tk = 0; tk < 16; ++tk) {
          const uint32_t* row = vi + tk * (vb * D / 32);
          uint32_t v = row[bit >> 5] >> (bit & 31);
          if ((bit & 31) + vb > 32) v |= row[(bit >> 5) + 1] << (32 - (bit & 31));
          const float cv = vlut[v & vmask];
#pragma unroll
          for (int h = 0; h < NR; ++h) o[r][h] = fmaf(pbuf[tk][h], cv, o[r][h]);
        }
      }
    }
    __syncthreads();
  }
  // inverse rotation of the rotated-domain accumulator, once per chunk
#pragma unroll
  for (int r = 0; r < DPT; ++r) {
    const int i = tid + 128 * r;
    if (i < D)
#pragma unroll
      for (int h = 0; h < NR; ++h) ob[h][i] = o[r][h];
  }
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5;
  for (int h = warp; h < a.nrg; h += 4) {
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = ob[h][coord_of(e, lane)];
    wht_warp<E>(x, lane);
    float* dst = a.parts + (((size_t)b * a.hq + h0 + h) * a.n_parts + part) * (D + 2);
    const float sc2 = rsqrtf((float)D);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = coord_of(e, lane);
      dst[c] = x[e] * sc2 * a.signs[c];
    }
    if (lane == 0) {
      dst[D] = st.m[h];
      dst[D + 1] = st.l[h];
    }
  }
}

// ------------------------------------------------------------------ merge
// grid (hq, batch, d / 32): one block per query head and 32 output dimensions.
// The part weights 2^(m_i - M) are computed once into shared memory; each warp
// then sums every fourth part over the block's 32 dimensions (one coalesced
// 128-byte row per part) and the four warp sums are added at the end.
__global__ void __launch_bounds__(128) merge_kernel(DecArgs a, int d) {
  extern __shared__ float sw[];  // [n_parts]
  __shared__ float red[4][32];
  __shared__ float s_m[4], s_l[4];
  const int h = blockIdx.x, b = blockIdx.y, col = blockIdx.z * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nc = seq_nc(a, b);
  const int nb = seq_nb(a, b);
  const int nch = (nc + a.chunk_tokens - 1) / a.chunk_tokens;
  const int nparts = nch + (nb > 0 ? 1 : 0);
  const float* base = a.parts + ((size_t)b * a.hq + h) * a.n_parts * (d + 2);
  auto part = [&](int i) { return base + (size_t)(i < nch ? i : a.n_chunks) * (d + 2); };
  float M = -INFINITY;
  for (int i = tid; i < nparts; i += 128) {
    const float m = part(i)[d];
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
    den = fmaf(w, part(i)[d + 1], den);
  }
  den = warp_sum(den);
  if (lane == 0) s_l[warp] = den;
  __syncthreads();  // weights and s_l
  den = (s_l[0] + s_l[1]) + (s_l[2] + s_l[3]);
  float acc = 0.f;
#pragma unroll 4
  for (int i = warp; i < nparts; i += 4) acc = fmaf(sw[i], part(i)[col + lane], acc);
  red[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    const float o = (red[0][lane] + red[1][lane]) + (red[2][lane] + red[3][lane]);
    a.out[((size_t)b * a.hq + h) * d + col + lane] = den > 0.f ? o / den : 0.f;
  }
}

template <int D, int NR, int VB>
cudaError_t launch_main_vb(const DecArgs& a, dim3 grid, cudaStream_t s) {
  auto kern = decode_main_kernel<D, NR, VB>;
  constexpr int TILE = MainDec<D, NR, VB>::TILE;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TILE);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, TILE, s>>>(a);
  return cudaGetLastError();
}

template <int D, int NR>
cudaError_t launch_tpl(const DecArgs& a, int vb, dim3 grid, cudaStream_t s) {
  if (vb == 4) return launch_main_vb<D, NR, 4>(a, grid, s);
  if (vb == 2) return launch_main_vb<D, NR, 2>(a, grid, s);
  auto kern = decode_alt_kernel<D, NR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, alt_tile_bytes(D, 16, 8));
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, alt_tile_bytes(D, a.kb, a.avb), s>>>(a);
  return cudaGetLastError();
}

// vb: value bits of the main layout (2 or 4), 0 for the alternate layout
template <int D>
cudaError_t launch_d(const DecArgs& a, int vb, dim3 grid, cudaStream_t s) {
  if (a.nrg <= 1) return launch_tpl<D, 1>(a, vb, grid, s);
  if (a.nrg <= 2) return launch_tpl<D, 2>(a, vb, grid, s);
  if (a.nrg <= 4) return launch_tpl<D, 4>(a, vb, grid, s);
  return launch_tpl<D, 8>(a, vb, grid, s);
}

}  // namespace

cudaError_t launch_decode(tq_ctx* ctx, const DecodePlan& plan, const void* q, int batch, const void* pool,
                          int num_blocks, const int32_t* block_table, int max_blocks, const int32_t* n_compressed,
                          const void* ring_k, const void* ring_v, const int32_t* n_buf, int max_ctx, float* out,
                          void* workspace, cudaStream_t s) {
  if (plan.tensor_core) {
    TcArgs t{};
    t.q = static_cast<const __half*>(q);
    t.pool = static_cast<const uint8_t*>(pool);
    t.num_blocks = num_blocks;
    t.block_table = block_table;
    t.max_blocks = max_blocks;
    t.n_compressed = n_compressed;
    t.ring_k = static_cast<const __half*>(ring_k);
    t.ring_v = static_cast<const __half*>(ring_v);
    t.n_buf = n_buf;
    t.max_ctx = max_ctx;
    t.out = out;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    t.afrag = (plan.fused_prep || plan.hybrid) ? nullptr : reinterpret_cast<uint4*>(ws);
    t.parts = reinterpret_cast<float*>(ws + plan.q_bytes);
    t.chunk_pages = plan.chunk_tokens / kPage;
    t.n_chunks = plan.n_chunks;
    t.n_parts = plan.n_parts;
    t.hq = ctx->cfg.num_q_heads;
    t.hkv = ctx->cfg.num_kv_heads;
    t.n_rep = ctx->n_rep;
    t.groups = (ctx->n_rep + kMaxRep - 1) / kMaxRep;
    t.nrg = ctx->n_rep / t.groups;
    t.signs = ctx->d_signs;
    t.sfrag_enc = ctx->d_sfrag_enc;
    t.kb = ctx->cfg.key_bits;
    t.cta_warps = plan.cta_warps;
    t.err = ctx->d_err;
    if (plan.hybrid) return launch_decode_hy(ctx, t, batch, ws, s);
    return launch_decode_tc(ctx, t, batch, s);
  }
  DecArgs a;
  a.q = static_cast<const __half*>(q);
  a.batch = batch;
  a.pool = static_cast<const uint8_t*>(pool);
  a.num_blocks = num_blocks;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.n_compressed = n_compressed;
  a.ring_k = static_cast<const __half*>(ring_k);
  a.ring_v = static_cast<const __half*>(ring_v);
  a.n_buf = n_buf;
  a.max_ctx = max_ctx;
  a.out = out;
  a.qprep = static_cast<float*>(workspace);
  a.parts = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.q_bytes);
  a.chunk_tokens = plan.chunk_tokens;
  a.n_chunks = plan.n_chunks;
  a.n_parts = plan.n_parts;
  a.hq = ctx->cfg.num_q_heads;
  a.hkv = ctx->cfg.num_kv_heads;
  a.n_rep = ctx->n_rep;
  a.groups = (ctx->n_rep + kMaxRep - 1) / kMaxRep;
  a.nrg = ctx->n_rep / a.groups;
  a.signs = ctx->d_signs;
  a.sketch_t = ctx->d_sketch_t;
  a.tab = ctx->tab;
  a.vcent = ctx->d_vcent;
  a.kb = ctx->cfg.key_bits;
  a.avb = ctx->cfg.value_bits;
  a.err = ctx->d_err;
  const int d = ctx->cfg.head_dim;
  const bool main = ctx->cfg.layout == TQ_LAYOUT_MAIN;
  cudaError_t e = cudaSuccess;
  if (main) {
    dim3 g(a.hq, batch);
    switch (d) {
      case 64: prep_main_kernel<64><<<g, 32, 0, s>>>(a); break;
      case 128: prep_main_kernel<128><<<g, 32, 0, s>>>(a); break;
      case 256: prep_main_kernel<256><<<g, 32, 0, s>>>(a); break;
      case 512: prep_main_kernel<512><<<g, 32, 0, s>>>(a); break;
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ctx->launches++;
  }
  a.first_part = 0;
  dim3 grid(plan.n_parts, a.hkv * a.groups, batch);
  bool done = false;
  if (!main && alt_v2_supported(ctx)) {
    // compressed chunks: warp-per-page kernel; the exact buffer (if any): the part kernel below
    ctx->decode_kernel = "decode_alt_v2_kernel";
    prof_start(ctx, kProfDecode, s);
    e = launch_decode_alt_v2(ctx, q, pool, num_blocks, block_table, max_blocks, n_compressed, max_ctx, a.parts,
                             plan.chunk_tokens, plan.n_chunks, plan.n_parts, batch, s);
    prof_stop(ctx, kProfDecode, s);
    if (e == cudaSuccess) {
      ctx->launches++;
      done = true;
      a.first_part = plan.n_chunks;
      grid.x = 1;
    } else if (e != cudaErrorNotSupported) {
      return e;
    } else {
      cudaGetLastError();
    }
  }
  if (!done || n_buf) {
    if (!done) {
      ctx->decode_kernel = main ? "decode_main_kernel" : "decode_alt_kernel";
      prof_start(ctx, kProfDecode, s);
    }
    switch (d) {
      case 64: e = launch_d<64>(a, main ? ctx->cfg.value_bits : 0, grid, s); break;
      case 128: e = launch_d<128>(a, main ? ctx->cfg.value_bits : 0, grid, s); break;
      case 256: e = launch_d<256>(a, main ? ctx->cfg.value_bits : 0, grid, s); break;
      case 512: e = launch_d<512>(a, main ? ctx->cfg.value_bits : 0, grid, s); break;
    }
    if (!done) prof_stop(ctx, kProfDecode, s);
    if (e != cudaSuccess) return e;
    ctx->launches++;
  }
  prof_start(ctx, kProfMerge, s);
  merge_kernel<<<dim3(a.hq, batch, d / 32), 128, sizeof(float) * plan.n_parts, s>>>(a, d);
  prof_stop(ctx, kProfMerge, s);
  e = cudaGetLastError();
  if (e == cudaSuccess) ctx->launches++;
  return e;
}

}  // namespace tq
