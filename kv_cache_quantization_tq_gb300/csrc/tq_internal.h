// Internal declarations shared by the host glue (host.cpp) and the CUDA
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>
#include <vector>

#include "tq.h"

namespace tq {

constexpr int kPage = 16;        // tokens per page
constexpr int kRing = 128;       // exact recent-token buffer
constexpr int kGroup = 32;       // value group / key block
constexpr int kMaxRep = 8;       // query heads handled by one decode CTA
constexpr int kMaxChunks = 8192;  // split-K chunks per sequence (merge weights in shared memory)
// Tensor-core decode query workspace per (sequence, head group), in 16-byte units: the score A
// fragments of up to 5 planes x 8 k-steps x 32 lanes, then 4 prep slices x 2 x kMaxRep partial
// score offsets (floats).
constexpr int kTcQueryU4 = 5 * 8 * 32 + 4 * 2 * kMaxRep / 4;
// tcgen05 decode (decode_hy.cu) query record per (sequence, head group), bytes: the e4m3 query
// operand (12 K-slices x 48 columns x 32 bytes), then 2 x 2 x kMaxRep floats (scales, offsets).
constexpr int kHyQueryBytes = 12 * 48 * 32 + 4 * 4 * kMaxRep;

// Small per-context tables passed by value as kernel parameters.
struct CodeTables {
  float c[16];  // centroids, ascending (2..8 used by main keys, 4..16 by alt values)
  float b[16];  // decision boundaries (midpoints), K-1 used
};

struct ProfileKind {
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev;  // recorded pairs
  size_t used = 0;
};

}  // namespace tq

struct tq_ctx {
  tq_config cfg;
  int device = 0;
  int sm_count = 152;  // multiprocessors of the context's device (split-K sizing)
  int n_rep = 1;
  int ncent = 4;
  tq::CodeTables tab{};
  std::vector<float> h_centroids, h_boundaries, h_signs, h_sketch;
  float* d_signs = nullptr;     // [d]
  float* d_sketch = nullptr;    // [m][d]
  float* d_sketch_t = nullptr;  // [d][m]
  uint4* d_sfrag = nullptr;     // S as fp16 high/low mma.sync B fragments (back-projection)
  uint4* d_sfrag_enc = nullptr; // S^T as fp16 high/low mma.sync B fragments (encode projection)
  float* d_vcent = nullptr;     // alternate layout: value centroids [256] (2^value_bits used)
  float* d_vbound = nullptr;    // alternate layout: their decision boundaries [256] (2^value_bits - 1 used)
  uint32_t* d_err = nullptr;    // device error word
  int64_t launches = 0;
  int decode_path = 0;          // TQ_DECODE_AUTO / _MMA_SYNC / _TCGEN05
  const char* decode_kernel = nullptr;  // kernel of the last decode call (profiling reports)
  bool profiling = false;
  tq::ProfileKind prof[3];      // 0 decode, 1 encode, 2 merge
};

namespace tq {

enum ProfKind { kProfDecode = 0, kProfEncode = 1, kProfMerge = 2 };

// Event bracketing for the profiler (no-ops unless profiling is on).
void prof_start(tq_ctx* ctx, int kind, cudaStream_t s);
void prof_stop(tq_ctx* ctx, int kind, cudaStream_t s);

// Decode chunking policy shared by tq_workspace_size and tq_decode_attention.
struct DecodePlan {
  bool tensor_core;   // main layout, head_dim 128: decode_tc.cu (or decode_hy.cu)
  bool hybrid;        // tensor-core path with the score on tcgen05: decode_hy.cu
  bool fused_prep;    // tensor-core path: each CTA builds its own query fragments (one-wave grids)
  int cta_warps;      // tensor-core path: 8 (at most one CTA per SM) or 4 warps per decode CTA
  int chunk_tokens;   // compressed tokens per split-K chunk (multiple of 16)
  int n_chunks;       // chunks for max_ctx compressed tokens
  int n_parts;        // n_chunks + 1 (ring part)
  size_t q_bytes;     // pre-rotated queries / score fragments
  size_t part_bytes;  // split-K partials
  size_t total;
};
DecodePlan decode_plan(const tq_ctx* ctx, int batch, int max_ctx);

// ---- launchers implemented in the .cu files (return a cudaError_t) ----
cudaError_t launch_encode(tq_ctx* ctx, const void* k, const void* v, int batch, int src_tokens, int n_tokens,
                          const int32_t* start_pos, const int32_t* block_table, int max_blocks, void* pool,
                          int num_blocks, cudaStream_t s);
cudaError_t launch_append(tq_ctx* ctx, const void* k_new, const void* v_new, const int32_t* pos, int batch,
                          void* ring_k, void* ring_v, const int32_t* block_table, int max_blocks, void* pool,
                          int num_blocks, cudaStream_t s);
cudaError_t launch_decode(tq_ctx* ctx, const DecodePlan& plan, const void* q, int batch, const void* pool,
                          int num_blocks, const int32_t* block_table, int max_blocks, const int32_t* n_compressed,
                          const void* ring_k, const void* ring_v, const int32_t* n_buf, int max_ctx, float* out,
                          void* workspace, cudaStream_t s);
cudaError_t launch_dequantize(tq_ctx* ctx, const void* pool, int num_blocks, const int32_t* block_table,
                              int max_blocks, const int32_t* n_tokens, const void* ring_k, const void* ring_v,
                              const int32_t* n_buf, int batch, int max_tokens, void* k_out, void* v_out,
                              bool bf16, cudaStream_t s);
size_t sketch_frag_bytes(int d);
cudaError_t build_sketch_frags(const float* sketch, int d, void* frag);
cudaError_t build_sketch_frags_enc(const float* sketch, int d, void* frag);
cudaError_t launch_pack(const uint8_t* codes, int64_t n, int bits, void* dst, cudaStream_t s);
cudaError_t launch_unpack(const void* src, int64_t n, int bits, uint8_t* codes, cudaStream_t s);

}  // namespace tq
