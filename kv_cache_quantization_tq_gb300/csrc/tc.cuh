// Arguments and entry points of the tensor-core main-layout decode (decode_tc.cu).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "tq_internal.h"

namespace tq {

struct TcArgs {
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
  float* out;
  uint4* afrag;    // [B][Hkv * groups][kTcQueryU4] query fragments and score offsets, or NULL: built per CTA
  float* parts;    // [B][Hq][n_parts][d + 4] split-K partials (o, m, l, pad)
  int chunk_pages, n_chunks, n_parts;
  int hq, hkv, n_rep, nrg, groups;
  int kb;          // key bits: 2, 3 or 4 (kb - 1 stored index planes, high bit first, then QJL)
  int cta_warps;   // warps per decode CTA: 8 (at most one CTA per SM) or 4
  const float* signs;
  const uint4* sfrag_enc;  // S^T as mma.sync B fragments (k = coordinate, n = sketch row), hi / lo
  uint32_t* err;
  int n_lm;        // Lloyd-Max A planes: 1 (2-bit keys), 2 (3-bit), 4 (4-bit: three bits + their XOR)
  float lm_w[4];   // weight of each Lloyd-Max A plane (Walsh coefficient of the codebook)
  float qjl_coef, logit_scale;
};

bool tc_supported(const tq_ctx* ctx);
cudaError_t launch_decode_tc(tq_ctx* ctx, TcArgs& a, int batch, cudaStream_t s);
// Score constants of a context (Lloyd-Max Walsh weights, QJL coefficient, logit scale) into a.
void tc_set_score_constants(const tq_ctx* ctx, TcArgs& a);
// Split-K merge of the partials in a.parts (sequences with one part were written directly).
cudaError_t launch_tc_merge(tq_ctx* ctx, TcArgs& a, int batch, cudaStream_t s);
// tcgen05 score path (decode_hy.cu): 3-bit keys, 2-bit values, head_dim 128.
bool hy_supported(const tq_ctx* ctx);
cudaError_t launch_decode_hy(tq_ctx* ctx, TcArgs& a, int batch, uint8_t* qrec, cudaStream_t s);

}  // namespace tq
