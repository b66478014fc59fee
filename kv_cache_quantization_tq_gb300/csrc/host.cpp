// Host side of libtq: argument checking, context and table setup, host bit
// packing, profiling and the extern "C" entry points that forward to the
// CUDA launchers.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "tq_internal.h"

namespace {

// ------------------------------------------------------------------ Lloyd-Max
// Gauss-Legendre nodes/weights on [-1, 1] by Newton iteration on P_n, using
// the three-term recurrence (n+1) P_{n+1} = (2n+1) x P_n - n P_{n-1}.
void gauss_legendre(int n, std::vector<double>& x, std::vector<double>& w) {
  x.assign(n, 0.0);
  w.assign(n, 0.0);
  for (int i = 0; i < n; ++i) {
    double z = cos(M_PI * (i + 0.75) / (n + 0.5));
    double dp = 1.0;
    for (int it = 0; it < 100; ++it) {
      double p0 = 1.0, p1 = z;
      for (int k = 2; k <= n; ++k) {
        double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
        p0 = p1;
        p1 = p2;
      }
      dp = n * (z * p1 - p0) / (z * z - 1.0);
      double dz = p1 / dp;
      z -= dz;
      if (fabs(dz) < 1e-16) break;
    }
    x[i] = z;
    w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
  }
}

struct SphereCoord {
  int d;
  double logc;
  std::vector<double> gx, gw;
  explicit SphereCoord(int dim) : d(dim) {
    logc = lgamma(d / 2.0) - 0.5 * log(M_PI) - lgamma((d - 1) / 2.0);
    gauss_legendre(20, gx, gw);
  }
  double pdf(double x) const {
    double u = 1.0 - x * x;
    if (u <= 0.0) return 0.0;
    return exp(logc + 0.5 * (d - 3) * log(u));
  }
  // int_a^b f, composite Gauss-Legendre on 64 pieces.
  double prob(double a, double b) const {
    const int pieces = 64;
    double h = (b - a) / pieces, acc = 0.0;
    for (int p = 0; p < pieces; ++p) {
      double mid = a + (p + 0.5) * h, half = 0.5 * h, s = 0.0;
      for (size_t k = 0; k < gx.size(); ++k) s += gw[k] * pdf(mid + half * gx[k]);
      acc += s * half;
    }
    return acc;
  }
  // int_a^b x f = C/(d-1) [(1-a^2)^((d-1)/2) - (1-b^2)^((d-1)/2)]
  double moment(double a, double b) const {
    double e = 0.5 * (d - 1);
    double ta = (1.0 - a * a) > 0 ? exp(e * log(1.0 - a * a)) : 0.0;
    double tb = (1.0 - b * b) > 0 ? exp(e * log(1.0 - b * b)) : 0.0;
    return exp(logc) / (d - 1) * (ta - tb);
  }
};

// Standard normal quantile by bisection on Phi(x) = erfc(-x / sqrt 2) / 2 (start values only).
double normal_quantile(double u) {
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 200; ++it) {
    const double mid = 0.5 * (lo + hi);
    (0.5 * erfc(-mid / sqrt(2.0)) < u ? lo : hi) = mid;
  }
  return 0.5 * (lo + hi);
}

// 32 levels and up (the q5_0 .. q8_0 value formats of the vllm-metal TurboQuant guide): Lloyd's
// iteration contracts too slowly there, so the same conditions are solved by Newton's method on
// F(c) = c - T(c).  T_j depends only on its cell's edges (dT/db = f(b)(b - T)/P,
// dT/da = f(a)(T - a)/P) and each inner edge is the midpoint of two centroids, so the Jacobian
// is tridiagonal (Thomas algorithm).  A step is halved while the residual does not shrink.
void lloyd_newton(const SphereCoord& f, std::vector<double>& c) {
  const int k = (int)c.size();
  std::vector<double> e(k + 1), t(k), p(k), F(k), lo(k), di(k), up(k), r(k), cn(k), en(k + 1), tn(k), pn(k), Fn(k);
  auto eval = [&](const std::vector<double>& cc, std::vector<double>& ee, std::vector<double>& tt,
                  std::vector<double>& pp, std::vector<double>& ff) {
    ee[0] = -1.0;
    ee[k] = 1.0;
    for (int j = 1; j < k; ++j) ee[j] = 0.5 * (cc[j - 1] + cc[j]);
    double worst = 0.0;
    for (int j = 0; j < k; ++j) {
      pp[j] = f.prob(ee[j], ee[j + 1]);
      tt[j] = f.moment(ee[j], ee[j + 1]) / pp[j];
      ff[j] = cc[j] - tt[j];
      worst = std::max(worst, fabs(ff[j]));
    }
    return worst;
  };
  double res = eval(c, e, t, p, F);
  for (int it = 0; it < 100 && res > 1e-15; ++it) {
    for (int j = 0; j < k; ++j) {
      const double dta = f.pdf(e[j]) * (t[j] - e[j]) / p[j];
      const double dtb = f.pdf(e[j + 1]) * (e[j + 1] - t[j]) / p[j];
      di[j] = 1.0 - 0.5 * (dta + dtb);
      lo[j] = -0.5 * dta;  // coefficient of c_{j-1}
      up[j] = -0.5 * dtb;  // coefficient of c_{j+1}
      r[j] = -F[j];
    }
    for (int j = 1; j < k; ++j) {  // forward elimination
      const double m = lo[j] / di[j - 1];
      di[j] -= m * up[j - 1];
      r[j] -= m * r[j - 1];
    }
    r[k - 1] /= di[k - 1];
    for (int j = k - 2; j >= 0; --j) r[j] = (r[j] - up[j] * r[j + 1]) / di[j];
    double lam = 1.0, rn = res;
    for (;;) {
      for (int j = 0; j < k; ++j) cn[j] = c[j] + lam * r[j];
      bool sorted = true;
      for (int j = 1; j < k; ++j) sorted = sorted && cn[j] > cn[j - 1];
      if (sorted) rn = eval(cn, en, tn, pn, Fn);
      if ((sorted && rn < res) || lam < 1e-6) break;
      lam *= 0.5;
    }
    if (!(rn < res)) break;  // no further progress at this precision
    c.swap(cn);
    e.swap(en);
    t.swap(tn);
    p.swap(pn);
    F.swap(Fn);
    res = rn;
  }
}

void lloyd_max(int d, int bits, double* cent, double* bound) {
  const int k = 1 << bits;
  SphereCoord f(d);
  std::vector<double> c(k), edges(k + 1), cn(k);
  if (bits >= 5) {
    for (int j = 0; j < k; ++j) c[j] = normal_quantile((j + 0.5) / k) / sqrt((double)d);
    lloyd_newton(f, c);
  } else {
    for (int j = 0; j < k; ++j) c[j] = (2.0 * j + 1.0 - k) / k * 2.0 / sqrt((double)d);
  }
  for (int it = 0; it < (bits >= 5 ? 0 : 200000); ++it) {
    edges[0] = -1.0;
    edges[k] = 1.0;
    for (int j = 1; j < k; ++j) edges[j] = 0.5 * (c[j - 1] + c[j]);
    double delta = 0.0;
    for (int j = 0; j < k; ++j) {
      cn[j] = f.moment(edges[j], edges[j + 1]) / f.prob(edges[j], edges[j + 1]);
      delta = std::max(delta, fabs(cn[j] - c[j]));
    }
    c = cn;
    if (delta < 1e-15) break;
  }
  for (int j = 0; j < k; ++j) cent[j] = 0.5 * (c[j] - c[k - 1 - j]);
  if (bound)
    for (int j = 0; j + 1 < k; ++j) bound[j] = 0.5 * (cent[j] + cent[j + 1]);
}

// ------------------------------------------------------------------ tables
// SplitMix64 output n of the generator with initial state s0.
inline uint64_t splitmix_word(uint64_t s0, uint64_t n) {
  uint64_t z = s0 + (n + 1) * 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

void make_tables(uint64_t seed, int d, int m, float* signs, float* sketch) {
  const uint64_t s_sign = seed + (1ULL << 40), s_gauss = seed + (2ULL << 40);
  for (int i = 0; i < d; ++i) signs[i] = (splitmix_word(s_sign, i) >> 63) ? -1.0f : 1.0f;
  if (!sketch) return;
  const int64_t n = (int64_t)m * d;
  for (int64_t k = 0; 2 * k < n; ++k) {
    uint64_t a = splitmix_word(s_gauss, 2 * k), b = splitmix_word(s_gauss, 2 * k + 1);
    double u1 = ((double)(a >> 11) + 1.0) * 0x1.0p-53;
    double u2 = (double)(b >> 11) * 0x1.0p-53;
    double r = sqrt(-2.0 * log(u1));
    sketch[2 * k] = (float)(r * cos(2.0 * M_PI * u2));
    if (2 * k + 1 < n) sketch[2 * k + 1] = (float)(r * sin(2.0 * M_PI * u2));
  }
}

bool valid_dim(int d) { return d == 64 || d == 128 || d == 256 || d == 512; }

tq_status check_config(const tq_config* c) {
  if (!c) return TQ_ERR_INVALID_ARG;
  if (c->num_kv_heads < 1 || c->num_q_heads < 1 || c->head_dim < 1) return TQ_ERR_INVALID_ARG;
  if (c->num_q_heads % c->num_kv_heads) return TQ_ERR_INVALID_ARG;
  if (!valid_dim(c->head_dim)) return TQ_ERR_UNSUPPORTED;
  if (c->page_size != tq::kPage || c->ring_capacity != tq::kRing || c->group_size != tq::kGroup)
    return TQ_ERR_UNSUPPORTED;
  const int n_rep = c->num_q_heads / c->num_kv_heads;
  const int groups = (n_rep + tq::kMaxRep - 1) / tq::kMaxRep;
  if (n_rep % groups) return TQ_ERR_UNSUPPORTED;
  if (c->layout == TQ_LAYOUT_MAIN) {
    if (c->key_bits < 2 || c->key_bits > 4 || (c->value_bits != 2 && c->value_bits != 4) ||
        c->qjl_m != c->head_dim || c->key_format != TQ_KEY_AFFINE)
      return TQ_ERR_UNSUPPORTED;
  } else if (c->layout == TQ_LAYOUT_ALT) {
    const int kb = c->key_bits;
    if ((kb != 16 && kb != 8 && kb != 5 && kb != 4 && kb != 2) || c->value_bits < 2 || c->value_bits > 8)
      return TQ_ERR_UNSUPPORTED;
    if (c->key_format != TQ_KEY_AFFINE && !(c->key_format == TQ_KEY_SIGNED && kb == 2)) return TQ_ERR_UNSUPPORTED;
  } else {
    return TQ_ERR_INVALID_ARG;
  }
  return TQ_OK;
}

tq_status finish_create(const tq_config* cfg, std::vector<float> cent, std::vector<float> signs,
                        std::vector<float> sketch, tq_ctx** out) {
  tq_ctx* ctx = new (std::nothrow) tq_ctx();
  if (!ctx) return TQ_ERR_INVALID_ARG;
  ctx->cfg = *cfg;
  ctx->n_rep = cfg->num_q_heads / cfg->num_kv_heads;
  ctx->ncent = (int)cent.size();
  const int d = cfg->head_dim;
  ctx->h_centroids = cent;
  ctx->h_boundaries.resize(cent.size() - 1);
  for (size_t j = 0; j + 1 < cent.size(); ++j)
    ctx->h_boundaries[j] = (float)(0.5 * ((double)cent[j] + (double)cent[j + 1]));
  // kernel-parameter tables: codebooks of up to 16 entries; wider value codebooks (alternate layout,
  // 5- to 8-bit values) live in device memory only
  for (size_t j = 0; j < cent.size() && j < 16; ++j) ctx->tab.c[j] = cent[j];
  for (size_t j = 0; j + 1 < cent.size() && j < 16; ++j) ctx->tab.b[j] = ctx->h_boundaries[j];
  ctx->h_signs = signs;
  ctx->h_sketch = sketch;
  bool ok = cudaGetDevice(&ctx->device) == cudaSuccess;
  ok = ok && cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, ctx->device) == cudaSuccess;
  ok = ok && cudaMalloc(&ctx->d_signs, sizeof(float) * d) == cudaSuccess;
  ok = ok && cudaMalloc(&ctx->d_err, sizeof(uint32_t)) == cudaSuccess;
  ok = ok && cudaMemcpy(ctx->d_signs, signs.data(), sizeof(float) * d, cudaMemcpyHostToDevice) == cudaSuccess;
  ok = ok && cudaMemset(ctx->d_err, 0, sizeof(uint32_t)) == cudaSuccess;
  if (ok && cfg->layout == TQ_LAYOUT_ALT) {
    // value codebook and its decision boundaries as device tables (up to 256 / 255 floats)
    const size_t nc = cent.size();
    ok = cudaMalloc(&ctx->d_vcent, sizeof(float) * 256) == cudaSuccess;
    ok = ok && cudaMalloc(&ctx->d_vbound, sizeof(float) * 256) == cudaSuccess;
    ok = ok && cudaMemset(ctx->d_vbound, 0, sizeof(float) * 256) == cudaSuccess;
    ok = ok && cudaMemcpy(ctx->d_vcent, cent.data(), sizeof(float) * nc, cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemcpy(ctx->d_vbound, ctx->h_boundaries.data(), sizeof(float) * (nc - 1),
                          cudaMemcpyHostToDevice) == cudaSuccess;
  }
  if (ok && cfg->layout == TQ_LAYOUT_MAIN) {
    const int m = cfg->qjl_m;
    std::vector<float> st((size_t)m * d);
    for (int j = 0; j < m; ++j)
      for (int i = 0; i < d; ++i) st[(size_t)i * m + j] = sketch[(size_t)j * d + i];
    ok = cudaMalloc(&ctx->d_sketch, sizeof(float) * m * d) == cudaSuccess;
    ok = ok && cudaMalloc(&ctx->d_sketch_t, sizeof(float) * m * d) == cudaSuccess;
    ok = ok && cudaMemcpy(ctx->d_sketch, sketch.data(), sizeof(float) * m * d, cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemcpy(ctx->d_sketch_t, st.data(), sizeof(float) * m * d, cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMalloc(&ctx->d_sfrag, tq::sketch_frag_bytes(d)) == cudaSuccess;
    ok = ok && tq::build_sketch_frags(ctx->d_sketch, d, ctx->d_sfrag) == cudaSuccess;
    ok = ok && cudaMalloc(&ctx->d_sfrag_enc, tq::sketch_frag_bytes(d)) == cudaSuccess;
    ok = ok && tq::build_sketch_frags_enc(ctx->d_sketch, d, ctx->d_sfrag_enc) == cudaSuccess;
  }
  if (!ok) {
    tq_destroy(ctx);
    return TQ_ERR_CUDA;
  }
  *out = ctx;
  return TQ_OK;
}

}  // namespace

namespace tq {

// Inside stream capture an ordinary record only orders the captured work;
// the "external" flavour makes the event a node that records a timestamp
// each time the graph runs.
static void record_event(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

void prof_start(tq_ctx* ctx, int kind, cudaStream_t s) {
  if (!ctx->profiling) return;
  ProfileKind& p = ctx->prof[kind];
  if (p.used >= 65536) return;
  if (p.used == p.ev.size()) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return;
    if (cudaEventCreate(&b) != cudaSuccess) {
      cudaEventDestroy(a);
      return;
    }
    p.ev.push_back({a, b});
  }
  record_event(p.ev[p.used].first, s);
}

void prof_stop(tq_ctx* ctx, int kind, cudaStream_t s) {
  if (!ctx->profiling) return;
  ProfileKind& p = ctx->prof[kind];
  if (p.used >= 65536 || p.used >= p.ev.size()) return;
  record_event(p.ev[p.used].second, s);
  p.used++;
}

DecodePlan decode_plan(const tq_ctx* ctx, int batch, int max_ctx) {
  DecodePlan pl{};
  const int d = ctx->cfg.head_dim;
  const int hkv = ctx->cfg.num_kv_heads;
  const int hq = ctx->cfg.num_q_heads;
  const int groups = (ctx->n_rep + kMaxRep - 1) / kMaxRep;
  const int64_t pages = ((int64_t)max_ctx + kPage - 1) / kPage;
  const int64_t total_pages = pages * batch * hkv * groups;
  auto align = [](size_t x) { return (x + 255) & ~(size_t)255; };
  pl.tensor_core = ctx->cfg.layout == TQ_LAYOUT_MAIN && d == 128;
  int64_t per;
  pl.cta_warps = 4;
  if (pl.tensor_core) {
    // At most one 8-warp CTA per SM when that fits in one wave with chunks of up to 64 pages (a
    // multiple of 8, one page per warp and round): each SM then builds the query side once, and
    // the merge sees half the partials.
    int64_t per8 = (total_pages + ctx->sm_count - 1) / std::max(1, ctx->sm_count);
    per8 = std::max<int64_t>(16, (per8 + 7) / 8 * 8);
    const int64_t parts8 = (pages + per8 - 1) / per8 + 1;
    if (per8 <= 64 && pages <= (int64_t)per8 * kMaxChunks && parts8 * hkv * groups * batch <= ctx->sm_count) {
      pl.cta_warps = 8;
      per = per8;
    } else {
      // About 2 CTAs per SM, i.e. one wave at the occupancy the kernel gets, with 16..64 pages
      // per chunk (4..16 per warp).  Measured on GB300 over 8K..65K-page decode steps (16..64-page
      // sweeps): fewer, longer chunks leave SMs idle; shorter ones pay the per-CTA query fragments
      // and combine more often than they gain parallelism.  Large steps stay at 64 pages, where
      // whole-wave chunk counts (36..56 pages) measured no better.
      const int64_t target = std::max<int64_t>(1, (int64_t)ctx->sm_count * 2);
      per = (total_pages + target - 1) / target;
      per = std::max<int64_t>(16, std::min<int64_t>(64, per));
      per = (per + 3) / 4 * 4;
      // One wave: when every sequence's chunks (plus its ring item) fit in kOneWaveCtas CTAs per
      // SM with chunks of at most kOneWaveMaxPages pages, size the chunks for exactly that, so
      // no SM idles through a last partial wave.
      constexpr int kOneWaveCtas = 3;
      constexpr int64_t kOneWaveMaxPages = 256;
      const int64_t bh = (int64_t)batch * hkv * groups;
      const int64_t slots = (int64_t)kOneWaveCtas * std::max(1, ctx->sm_count);
      const int64_t cps = (slots - bh) / std::max<int64_t>(1, bh);  // chunks per sequence and head group
      if (cps >= 1) {
        const int64_t per1 = ((pages + cps - 1) / cps + 3) / 4 * 4;
        if (per1 > per && per1 <= kOneWaveMaxPages) per = per1;
      }
    }
  } else {
    // about 8 CTAs per SM worth of split-K chunks, each between 4 and 64 pages
    per = (total_pages + 1215) / 1216;
    per = std::max<int64_t>(4, std::min<int64_t>(64, per));
  }
  // The tcgen05 score path (decode_hy.cu): 3-bit keys, 2-bit values, m = d.  One 14-warp CTA per
  // SM (it holds all 512 tensor-memory columns) walks its chunk in tiles of 8 pages.  The chunks
  // per sequence and head group minimise waves x (tiles per chunk + 3), the 3 standing for the
  // pipeline's fill and drain; ring items (short, launched after every chunk) are not counted.
  // TQ_DECODE_AUTO keeps the mma.sync kernels: on GB300 they measured faster (88 against 102 us per
  // launch at batch 8 x 32K, 28 / 4 heads).
  const bool hy_ok = pl.tensor_core && ctx->cfg.key_bits == 3 && ctx->cfg.value_bits == 2 && ctx->cfg.qjl_m == d;
  pl.hybrid = hy_ok && ctx->decode_path == TQ_DECODE_TCGEN05;
  if (pl.hybrid) {
    const int64_t bh = (int64_t)batch * hkv * groups;
    const int64_t sms = std::max(1, ctx->sm_count);
    int64_t best_cost = -1;
    // beyond about two waves more chunks only add partials
    const int64_t cmax = std::min<int64_t>(kMaxChunks, 2 * ((sms + bh - 1) / bh) + 2);
    for (int64_t c = 1; c <= cmax; ++c) {
      const int64_t per_c = ((pages + c - 1) / c + 7) / 8 * 8;
      const int64_t chunks = (pages + per_c - 1) / per_c;
      const int64_t cost = ((bh * chunks + sms - 1) / sms) * (per_c / 8 + 3);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        per = per_c;
      }
      if (per_c == 8) break;
    }
  }
  // at most kMaxChunks chunks per sequence: the merge keeps one weight per part in shared memory
  per = std::max<int64_t>(per, (pages + kMaxChunks - 1) / kMaxChunks);
  if (pl.hybrid)
    per = (per + 7) / 8 * 8;
  else if (pl.tensor_core)
    per = (per + pl.cta_warps - 1) / pl.cta_warps * pl.cta_warps;
  pl.chunk_tokens = (int)(per * kPage);
  pl.n_chunks = (int)((pages + per - 1) / per);
  pl.n_parts = pl.n_chunks + 1;
  if (pl.tensor_core) {
    // A grid that fits in one wave (3 CTAs per SM) builds the query fragments in every CTA,
    // saving a kernel; larger grids build them once per (sequence, head group) in a prep
    // kernel, because there the per-CTA cost (~3 us) outweighs the saved launch.
    const int64_t ctas = (int64_t)pl.n_parts * hkv * groups * batch;
    pl.fused_prep = !pl.hybrid && (pl.cta_warps == 8 || ctas <= (int64_t)ctx->sm_count * 3);
    if (pl.hybrid) {
      pl.cta_warps = 4;
      pl.q_bytes = align((size_t)batch * hkv * groups * kHyQueryBytes);
    } else {
      pl.q_bytes = pl.fused_prep ? 0 : align((size_t)batch * hkv * groups * kTcQueryU4 * 16);
    }
  } else
    pl.q_bytes = ctx->cfg.layout == TQ_LAYOUT_MAIN ? align(sizeof(float) * batch * hq * 2 * d) : 0;
  pl.part_bytes = align(sizeof(float) * (size_t)batch * hq * pl.n_parts * (d + (pl.tensor_core ? 4 : 2)));
  pl.total = pl.q_bytes + pl.part_bytes;
  return pl;
}

}  // namespace tq

// ====================================================================== C ABI
extern "C" {

const char* tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "TQ_OK";
    case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG: invalid argument";
    case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED: configuration not supported";
    case TQ_ERR_WORKSPACE: return "TQ_ERR_WORKSPACE: workspace too small";
    case TQ_ERR_CUDA: return "TQ_ERR_CUDA: CUDA runtime or launch failure";
  }
  return "unknown tq_status";
}

tq_status tq_config_init(tq_config* cfg, int layout, int head_dim, int num_q_heads, int num_kv_heads,
                         uint64_t seed) {
  if (!cfg) return TQ_ERR_INVALID_ARG;
  memset(cfg, 0, sizeof(*cfg));
  cfg->head_dim = head_dim;
  cfg->num_q_heads = num_q_heads;
  cfg->num_kv_heads = num_kv_heads;
  cfg->page_size = tq::kPage;
  cfg->ring_capacity = tq::kRing;
  cfg->layout = layout;
  cfg->group_size = tq::kGroup;
  cfg->seed = seed;
  if (layout == TQ_LAYOUT_MAIN) {
    cfg->key_bits = 3;
    cfg->value_bits = 2;
    cfg->qjl_m = head_dim;
  } else {
    cfg->key_bits = 8;
    cfg->value_bits = 3;
    cfg->qjl_m = 0;
  }
  return check_config(cfg);
}

tq_status tq_lloyd_max(int d, int bits, double* centroids, double* boundaries) {
  if (!centroids || d < 8 || bits < 1 || bits > 8) return TQ_ERR_INVALID_ARG;
  lloyd_max(d, bits, centroids, boundaries);
  return TQ_OK;
}

tq_status tq_generate_tables(uint64_t seed, int d, int m, float* signs, float* sketch) {
  if (!signs || d < 1 || (sketch && m < 1)) return TQ_ERR_INVALID_ARG;
  make_tables(seed, d, m, signs, sketch);
  return TQ_OK;
}

tq_status tq_create(const tq_config* cfg, tq_ctx** out) {
  if (!out) return TQ_ERR_INVALID_ARG;
  tq_status st = check_config(cfg);
  if (st != TQ_OK) return st;
  const int d = cfg->head_dim;
  // main: key_bits - 1 Lloyd-Max bits (one key bit is the QJL sign); alternate: value_bits
  const int bits = cfg->layout == TQ_LAYOUT_MAIN ? cfg->key_bits - 1 : cfg->value_bits;
  std::vector<double> c64(1 << bits);
  lloyd_max(d, bits, c64.data(), nullptr);
  std::vector<float> cent(c64.begin(), c64.end());
  std::vector<float> signs(d), sketch;
  if (cfg->layout == TQ_LAYOUT_MAIN) sketch.resize((size_t)cfg->qjl_m * d);
  make_tables(cfg->seed, d, cfg->qjl_m, signs.data(), sketch.empty() ? nullptr : sketch.data());
  return finish_create(cfg, cent, signs, sketch, out);
}

tq_status tq_create_with_tables(const tq_config* cfg, const float* centroids, const float* signs,
                                const float* sketch, tq_ctx** out) {
  if (!out || !centroids || !signs) return TQ_ERR_INVALID_ARG;
  tq_status st = check_config(cfg);
  if (st != TQ_OK) return st;
  const int d = cfg->head_dim;
  const int k = 1 << (cfg->layout == TQ_LAYOUT_MAIN ? cfg->key_bits - 1 : cfg->value_bits);
  if (cfg->layout == TQ_LAYOUT_MAIN && !sketch) return TQ_ERR_INVALID_ARG;
  for (int j = 0; j < k; ++j) {
    if (!(centroids[j] == -centroids[k - 1 - j])) return TQ_ERR_INVALID_ARG;
    if (j && !(centroids[j] > centroids[j - 1])) return TQ_ERR_INVALID_ARG;
  }
  for (int i = 0; i < d; ++i)
    if (signs[i] != 1.0f && signs[i] != -1.0f) return TQ_ERR_INVALID_ARG;
  std::vector<float> cent(centroids, centroids + k), sg(signs, signs + d), sk;
  if (cfg->layout == TQ_LAYOUT_MAIN) sk.assign(sketch, sketch + (size_t)cfg->qjl_m * d);
  return finish_create(cfg, cent, sg, sk, out);
}

void tq_destroy(tq_ctx* ctx) {
  if (!ctx) return;
  cudaFree(ctx->d_signs);
  cudaFree(ctx->d_sketch);
  cudaFree(ctx->d_sketch_t);
  cudaFree(ctx->d_sfrag);
  cudaFree(ctx->d_sfrag_enc);
  cudaFree(ctx->d_vcent);
  cudaFree(ctx->d_vbound);
  cudaFree(ctx->d_err);
  for (auto& p : ctx->prof)
    for (auto& e : p.ev) {
      cudaEventDestroy(e.first);
      cudaEventDestroy(e.second);
    }
  delete ctx;
}

tq_status tq_get_tables(const tq_ctx* ctx, float* centroids, float* boundaries, float* signs, float* sketch) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  if (centroids) memcpy(centroids, ctx->h_centroids.data(), sizeof(float) * ctx->h_centroids.size());
  if (boundaries) memcpy(boundaries, ctx->h_boundaries.data(), sizeof(float) * ctx->h_boundaries.size());
  if (signs) memcpy(signs, ctx->h_signs.data(), sizeof(float) * ctx->h_signs.size());
  if (sketch && !ctx->h_sketch.empty()) memcpy(sketch, ctx->h_sketch.data(), sizeof(float) * ctx->h_sketch.size());
  return TQ_OK;
}

namespace {
// main: key_bits key bits, value_bits value bits and one fp16 scale + minimum per group of 32 per
// coordinate, two fp16 norms; alternate: key_bits-bit key codes + 4 B per block of 32 (or fp16
// keys alone, key_bits 16), value_bits-bit value indices, fp16 norm
size_t record_bytes(const tq_config& c) {
  const size_t d = c.head_dim, vb = c.value_bits, kb = c.key_bits;
  return c.layout == TQ_LAYOUT_MAIN ? (kb * d) / 8 + (vb * d) / 8 + d / 8 + 4
                                    : (kb * d) / 8 + (kb == 16 ? 0 : (d / 32) * 4) + (vb * d) / 8 + 2;
}
}  // namespace

tq_status tq_config_check(const tq_config* cfg, size_t* bytes_per_token_head) {
  if (!cfg) return TQ_ERR_INVALID_ARG;
  const tq_status st = check_config(cfg);
  if (st == TQ_OK && bytes_per_token_head) *bytes_per_token_head = record_bytes(*cfg);
  return st;
}

size_t tq_bytes_per_token_head(const tq_ctx* ctx) { return ctx ? record_bytes(ctx->cfg) : 0; }

size_t tq_page_bytes(const tq_ctx* ctx) { return tq::kPage * tq_bytes_per_token_head(ctx); }

tq_status tq_workspace_size(const tq_ctx* ctx, int batch, int max_ctx, size_t* bytes) {
  if (!ctx || !bytes || batch < 0 || max_ctx < 0) return TQ_ERR_INVALID_ARG;
  *bytes = tq::decode_plan(ctx, batch, max_ctx).total;
  return TQ_OK;
}

static tq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA; }

tq_status tq_encode_flush(tq_ctx* ctx, const void* k, const void* v, int batch, int src_tokens, int n_tokens,
                          const int32_t* start_pos, const int32_t* block_table, int max_blocks, void* pool,
                          int num_blocks, cudaStream_t stream) {
  if (!ctx || batch < 0 || n_tokens < 0 || src_tokens < n_tokens || max_blocks < 0 || num_blocks < 0)
    return TQ_ERR_INVALID_ARG;
  if (n_tokens % tq::kPage) return TQ_ERR_INVALID_ARG;
  if (batch == 0 || n_tokens == 0) return TQ_OK;
  if (!k || !v || !start_pos || !block_table || !pool) return TQ_ERR_INVALID_ARG;
  if ((((uintptr_t)k) | ((uintptr_t)v)) & 15) return TQ_ERR_INVALID_ARG;  // 16-byte row copies
  return cuda_status(tq::launch_encode(ctx, k, v, batch, src_tokens, n_tokens, start_pos, block_table, max_blocks,
                                       pool, num_blocks, stream));
}

tq_status tq_append_token(tq_ctx* ctx, const void* k_new, const void* v_new, const int32_t* pos, int batch,
                          void* ring_k, void* ring_v, const int32_t* block_table, int max_blocks, void* pool,
                          int num_blocks, cudaStream_t stream) {
  if (!ctx || batch < 0 || max_blocks < 0 || num_blocks < 0) return TQ_ERR_INVALID_ARG;
  if (batch == 0) return TQ_OK;
  if (!k_new || !v_new || !pos || !ring_k || !ring_v || !block_table || !pool) return TQ_ERR_INVALID_ARG;
  if ((((uintptr_t)ring_k) | ((uintptr_t)ring_v)) & 15) return TQ_ERR_INVALID_ARG;  // 16-byte row copies
  return cuda_status(tq::launch_append(ctx, k_new, v_new, pos, batch, ring_k, ring_v, block_table, max_blocks, pool,
                                       num_blocks, stream));
}

tq_status tq_decode_attention(tq_ctx* ctx, const void* q, int batch, const void* pool, int num_blocks,
                              const int32_t* block_table, int max_blocks, const int32_t* n_compressed,
                              const void* ring_k, const void* ring_v, const int32_t* n_buf, int max_ctx,
                              float* out, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!ctx || batch < 0 || max_blocks < 0 || num_blocks < 0 || max_ctx < 0) return TQ_ERR_INVALID_ARG;
  if (batch == 0) return TQ_OK;
  if (!q || !out || !n_compressed || !block_table || (max_ctx > 0 && !pool)) return TQ_ERR_INVALID_ARG;
  if (n_buf && (!ring_k || !ring_v)) return TQ_ERR_INVALID_ARG;
  if (max_ctx % tq::kPage) return TQ_ERR_INVALID_ARG;
  tq::DecodePlan plan = tq::decode_plan(ctx, batch, max_ctx);
  if (!workspace || ws_bytes < plan.total) return TQ_ERR_WORKSPACE;
  if (((uintptr_t)workspace) & 255) return TQ_ERR_INVALID_ARG;
  return cuda_status(tq::launch_decode(ctx, plan, q, batch, pool, num_blocks, block_table, max_blocks, n_compressed,
                                       ring_k, ring_v, n_buf, max_ctx, out, workspace, stream));
}

static tq_status dequantize_common(tq_ctx* ctx, const void* pool, int num_blocks, const int32_t* block_table,
                                   int max_blocks, const int32_t* n_compressed, const void* ring_k, const void* ring_v,
                                   const int32_t* n_buf, int batch, int max_tokens, void* k_out, void* v_out, bool bf16,
                                   cudaStream_t stream) {
  if (!ctx || batch < 0 || max_blocks < 0 || num_blocks < 0 || max_tokens < 0) return TQ_ERR_INVALID_ARG;
  if (batch == 0 || max_tokens == 0) return TQ_OK;
  if (!k_out || !v_out || !n_compressed || !block_table || !pool) return TQ_ERR_INVALID_ARG;
  if (n_buf && (!ring_k || !ring_v)) return TQ_ERR_INVALID_ARG;
  if ((((uintptr_t)k_out) | ((uintptr_t)v_out)) & 15) return TQ_ERR_INVALID_ARG;
  if (n_buf && ((((uintptr_t)ring_k) | ((uintptr_t)ring_v)) & 15)) return TQ_ERR_INVALID_ARG;
  return cuda_status(tq::launch_dequantize(ctx, pool, num_blocks, block_table, max_blocks, n_compressed, ring_k,
                                           ring_v, n_buf, batch, max_tokens, k_out, v_out, bf16, stream));
}

tq_status tq_dequantize(tq_ctx* ctx, const void* pool, int num_blocks, const int32_t* block_table, int max_blocks,
                        const int32_t* n_compressed, const void* ring_k, const void* ring_v, const int32_t* n_buf,
                        int batch, int max_tokens, void* k_out, void* v_out, cudaStream_t stream) {
  return dequantize_common(ctx, pool, num_blocks, block_table, max_blocks, n_compressed, ring_k, ring_v, n_buf, batch,
                           max_tokens, k_out, v_out, false, stream);
}

tq_status tq_dequantize_bf16(tq_ctx* ctx, const void* pool, int num_blocks, const int32_t* block_table,
                             int max_blocks, const int32_t* n_compressed, const void* ring_k, const void* ring_v,
                             const int32_t* n_buf, int batch, int max_tokens, void* k_out, void* v_out,
                             cudaStream_t stream) {
  return dequantize_common(ctx, pool, num_blocks, block_table, max_blocks, n_compressed, ring_k, ring_v, n_buf, batch,
                           max_tokens, k_out, v_out, true, stream);
}

int tq_should_materialize(int64_t history_tokens, int64_t query_tokens, int head_dim, int num_kv_heads,
                          int64_t max_mib) {
  if (history_tokens < 0 || query_tokens < 0 || head_dim <= 0 || num_kv_heads <= 0) return -1;
  if (max_mib == 0) return 0;                          // materialisation switched off
  if (history_tokens < 8192) return 0;                 // short histories stay on the compressed path
  const int64_t threshold = head_dim == 128 ? 64 : std::max<int64_t>(128, head_dim / 2);
  if (query_tokens < threshold) return 0;              // decode steps and short suffixes
  if (max_mib > 0) {
    // dense K and V of the history, 2 bytes per element
    const double bytes = (double)history_tokens * num_kv_heads * head_dim * 2.0 * 2.0;
    if (bytes > (double)max_mib * 1048576.0) return 0;
  }
  return 1;
}

tq_status tq_pack(const uint8_t* codes, int64_t n, int bits, void* dst, cudaStream_t stream) {
  if (n < 0 || bits < 1 || bits > 8) return TQ_ERR_INVALID_ARG;
  if (n == 0) return TQ_OK;
  if (!codes || !dst) return TQ_ERR_INVALID_ARG;
  return cuda_status(tq::launch_pack(codes, n, bits, dst, stream));
}

tq_status tq_unpack(const void* src, int64_t n, int bits, uint8_t* codes, cudaStream_t stream) {
  if (n < 0 || bits < 1 || bits > 8) return TQ_ERR_INVALID_ARG;
  if (n == 0) return TQ_OK;
  if (!codes || !src) return TQ_ERR_INVALID_ARG;
  return cuda_status(tq::launch_unpack(src, n, bits, codes, stream));
}

tq_status tq_pack_host(const uint8_t* codes, int64_t n, int bits, void* dst) {
  if (n < 0 || bits < 1 || bits > 8) return TQ_ERR_INVALID_ARG;
  if (n == 0) return TQ_OK;
  if (!codes || !dst) return TQ_ERR_INVALID_ARG;
  uint8_t* out = (uint8_t*)dst;
  const int64_t nbytes = (n * bits + 7) / 8;
  memset(out, 0, (size_t)nbytes);
  const unsigned mask = (1u << bits) - 1u;
  for (int64_t i = 0; i < n; ++i) {
    if (codes[i] & ~mask) return TQ_ERR_INVALID_ARG;
    int64_t bit = i * bits;
    unsigned v = (unsigned)codes[i] << (bit & 7);
    out[bit >> 3] |= (uint8_t)(v & 0xFF);
    if ((bit & 7) + bits > 8) out[(bit >> 3) + 1] |= (uint8_t)(v >> 8);
  }
  return TQ_OK;
}

tq_status tq_unpack_host(const void* src, int64_t n, int bits, uint8_t* codes) {
  if (n < 0 || bits < 1 || bits > 8) return TQ_ERR_INVALID_ARG;
  if (n == 0) return TQ_OK;
  if (!codes || !src) return TQ_ERR_INVALID_ARG;
  const uint8_t* in = (const uint8_t*)src;
  const int64_t nbytes = (n * bits + 7) / 8;
  const unsigned mask = (1u << bits) - 1u;
  for (int64_t i = 0; i < n; ++i) {
    int64_t bit = i * bits;
    unsigned v = in[bit >> 3];
    if ((bit >> 3) + 1 < nbytes) v |= (unsigned)in[(bit >> 3) + 1] << 8;
    codes[i] = (uint8_t)((v >> (bit & 7)) & mask);
  }
  return TQ_OK;
}

tq_status tq_get_device_errors(tq_ctx* ctx, uint32_t* flags, cudaStream_t stream) {
  if (!ctx || !flags) return TQ_ERR_INVALID_ARG;
  uint32_t h = 0;
  if (cudaMemcpyAsync(&h, ctx->d_err, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaMemsetAsync(ctx->d_err, 0, sizeof(uint32_t), stream) != cudaSuccess) return TQ_ERR_CUDA;
  *flags = h;
  return TQ_OK;
}

int64_t tq_launch_count(const tq_ctx* ctx) { return ctx ? ctx->launches : 0; }

tq_status tq_set_decode_path(tq_ctx* ctx, int path) {
  if (!ctx || path < TQ_DECODE_AUTO || path > TQ_DECODE_TCGEN05) return TQ_ERR_INVALID_ARG;
  ctx->decode_path = path;
  return TQ_OK;
}

tq_status tq_profile_begin(tq_ctx* ctx) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  for (auto& p : ctx->prof) p.used = 0;
  ctx->profiling = true;
  return TQ_OK;
}

tq_status tq_profile_end(tq_ctx* ctx, tq_profile* out) {
  if (!ctx || !out) return TQ_ERR_INVALID_ARG;
  ctx->profiling = false;
  double ms[3] = {0, 0, 0};
  int64_t n[3] = {0, 0, 0};
  for (int kind = 0; kind < 3; ++kind) {
    tq::ProfileKind& p = ctx->prof[kind];
    for (size_t i = 0; i < p.used; ++i) {
      if (cudaEventSynchronize(p.ev[i].second) != cudaSuccess) return TQ_ERR_CUDA;
      float t = 0.f;
      if (cudaEventElapsedTime(&t, p.ev[i].first, p.ev[i].second) != cudaSuccess) return TQ_ERR_CUDA;
      ms[kind] += t;
      n[kind]++;
    }
    p.used = 0;
  }
  out->decode_launches = n[0];
  out->decode_ms = ms[0];
  out->encode_launches = n[1];
  out->encode_ms = ms[1];
  out->merge_launches = n[2];
  out->merge_ms = ms[2];
  out->decode_kernel = ctx->decode_kernel;
  return TQ_OK;
}

}  // extern "C"
