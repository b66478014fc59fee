/*
 * tq.h -- C ABI of libtq: TurboQuant-style KV-cache compression and decode
 * attention read directly from the compressed cache, for one NVIDIA GB300
 * (sm_103a).
 *
 * What the library computes (page titles as printed on the source pages):
 *
 *  - keys, main layout: random-sign diagonal D + normalised Walsh-Hadamard
 *    rotation, 2-bit Lloyd-Max index per rotated coordinate, 1-bit QJL sign
 *    sketch of the residual with its fp16 norm, fp16 key norm
 *    (turboquant vLLM guide, section 2 "quantisation flow", steps 1-3 and 5;
 *    TurboQuant-MLX overview, PolarQuant steps 1-3);
 *  - values, main layout: asymmetric min/max quantisation in groups of 32,
 *    2 bits per value (turboquant-bench, "compression algorithm details");
 *  - alternate layout: keys per-block affine 8-bit without rotation, values
 *    Walsh-Hadamard + 3-bit Lloyd-Max with an fp16 norm (vllm-metal
 *    TurboQuant guide, "quantisation principle" table);
 *  - decode attention: softmax(q k^T / sqrt(d)) v over the compressed tokens
 *    plus an exact fp16 buffer of the newest <= 128 tokens (turboquant-bench,
 *    "buffer strategy"; turboquant vLLM guide, section 5.1 ring buffer and
 *    hybrid attention), grouped-query aware (TurboQuant-MLX overview, GPU
 *    kernel section: n_rep).
 *
 * Conventions for every call:
 *  - All tensors are caller-owned.  "device" pointers are CUDA device
 *    memory on the current device; "host" pointers are ordinary host memory.
 *    fp16 tensors are IEEE binary16 passed as void*.
 *  - Every device call is asynchronous on the given stream (0 = legacy
 *    default stream) and performs no implicit synchronisation.
 *  - Errors are returned as tq_status, never thrown.  Arguments are checked
 *    on the host before any launch (TQ_ERR_INVALID_ARG / TQ_ERR_UNSUPPORTED /
 *    TQ_ERR_WORKSPACE); a failed launch returns TQ_ERR_CUDA.  Per-sequence
 *    values that live on the device (positions, lengths, block ids) are
 *    checked by the kernels: an out-of-range value makes the kernel skip that
 *    work item and set a bit in the context's device error word, read with
 *    tq_get_device_errors().  No kernel traps or spins.
 *
 * Page tiles and pool.  A page holds 16 consecutive tokens; a tile is one
 * page of one KV head; pool = uint8[num_blocks][num_kv_heads][tile] and
 * token p of sequence b lives in block block_table[b * max_blocks + p / 16]
 * at slot p % 16.  Multi-byte fields are little-endian.
 *
 *   main layout tile, 12 d + 64 bytes (100 B per token-head at d = 128):
 *     [0, 2d)       KH  high bit of each 2-bit key index   } token-major rows of d/8 B;
 *     [2d, 4d)      KL  low bit of each 2-bit key index    } coordinate 32w+2j+e (j<16,
 *     [4d, 6d)      KS  QJL sign bits [(S r)_j >= 0]       } e<2) = bit 16e+j of word w
 *     [6d, 10d)     VQ  value codes, uint32 per dimension: token 2j+e at bits 16e+2j..+1
 *     [10d, 12d)    VSM token t, group g at (t*d/32+g)*4: fp16 scale, fp16 minimum
 *     [12d, +32)    KN  fp16 key norm per token
 *     [12d+32, +32) RN  fp16 residual norm per token
 *   alternate layout tile, 24 d + 32 bytes:
 *     [0, 16d)      KQ  8-bit affine key codes, token-major, dimension i at byte i
 *     [16d, 18d)    KSM token t, block g at (t*d/32+g)*4: fp16 scale, fp16 minimum
 *     [18d, 24d)    VI  per token a 3d/8-byte stream of 3-bit value indices (tq_pack order)
 *     [24d, +32)    VN  fp16 value norm per token
 *
 * Other widths (tq_config key_bits / value_bits) keep the plane order:
 *   main: kb - 1 Lloyd-Max index planes (high bit first) then KS, each 2d
 *     bytes; VQ 2 vb d bytes (4-bit codes: two sub-planes of one uint32 per
 *     dimension, tokens 0-7 then 8-15, token 8w+2j+e at bits 16e+4j of word
 *     w); tile (2 kb + 2 vb + 2) d + 64 bytes.
 *   alternate: KQ is a dense kb-bit code stream per token (code c at bit
 *     kb c), 2 kb d bytes, followed by KSM; with key_bits 16 KQ holds the
 *     fp16 keys (32 d bytes) and there is no KSM.  VI is a dense vb-bit
 *     stream per token, 2 vb d bytes.  tq_config_check gives the size.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent shape */
  TQ_ERR_UNSUPPORTED = 2, /* valid but not implemented (head_dim, bits, ...) */
  TQ_ERR_WORKSPACE = 3,   /* workspace smaller than tq_workspace_size() */
  TQ_ERR_CUDA = 4         /* a CUDA runtime call or launch failed */
} tq_status;

typedef enum { TQ_LAYOUT_MAIN = 0, TQ_LAYOUT_ALT = 1 } tq_layout;

/* Device error word bits (tq_get_device_errors). */
#define TQ_DEVERR_BLOCK_ID   0x1u /* block-table entry outside [0, num_blocks) */
#define TQ_DEVERR_POSITION   0x2u /* position / length beyond the block table or not page aligned */
#define TQ_DEVERR_RING       0x4u /* n_buf outside [0, ring_capacity] */
#define TQ_DEVERR_CHUNKS     0x8u /* n_compressed larger than the max_ctx given to decode */
#define TQ_DEVERR_TIMEOUT    0x10u /* a decode CTA gave up waiting (about a second) for its own
                                      copies or tensor-core products; its output rows are not written */

/* Decode kernels for the main layout at head_dim 128 (tq_set_decode_path). */
#define TQ_DECODE_AUTO     0 /* the library chooses per call (default) */
#define TQ_DECODE_MMA_SYNC 1 /* scores and values on mma.sync (every key / value width) */
#define TQ_DECODE_TCGEN05  2 /* scores on tcgen05 (fp8 operands in tensor memory), values on mma.sync:
                                3-bit keys and 2-bit values only (other widths use mma.sync) */

typedef struct {
  int head_dim;      /* d: 64, 128, 256 or 512 (the sizes the pages' rotation kernels accept) */
  int num_q_heads;   /* Hq, a multiple of num_kv_heads (n_rep = Hq / Hkv) */
  int num_kv_heads;  /* Hkv */
  int page_size;     /* tokens per page: must be 16 */
  int ring_capacity; /* exact recent-token buffer: must be 128 */
  int layout;        /* tq_layout */
  int key_bits;      /* main: 3 (2-bit Lloyd-Max + 1-bit QJL, default), 2 or 4 (1- or 3-bit
                        Lloyd-Max + 1-bit QJL; turboquant vLLM guide, --key-bits); alt: 8
                        (default), 5, 4 or 2 bits per affine key code (the vllm-metal guide's
                        q8_0 / q5_0 / q4_0 / uint2 key formats), or 16: keys kept as fp16 and
                        only the values quantised (the V-only cache of the TurboQuant-MLX
                        overview) */
  int value_bits;    /* main: 2 (default) or 4 (turboquant vLLM guide, --value-bits); alt: 3
                        (default) or 2 .. 8 Lloyd-Max index bits per value coordinate (the
                        vllm-metal guide's q2_0 .. q8_0 value formats; 8 + 4 is its K8+V4) */
  int group_size;    /* value group / key block: must be 32 */
  int qjl_m;         /* main: sketch rows m, must equal head_dim; alt: 0 */
  uint64_t seed;     /* table seed; one table set per layer (base seed + layer) */
  int key_format;    /* alt layout, 2-bit keys: TQ_KEY_AFFINE (0, default: uint2, min/max affine codes)
                        or TQ_KEY_SIGNED (1: int2, signed symmetric mid-rise codes, see below); must
                        be 0 otherwise */
} tq_config;

/* Key formats of the alternate layout at key_bits 2 (the vllm-metal guide lists int2 and uint2,
 * with the same bytes; the pages give no rule that tells them apart, so this library reads them as):
 *   uint2 (TQ_KEY_AFFINE): s = fp16((max - min) / 3), mn = min, q = clamp(rint((x - mn) / s), 0, 3);
 *   int2  (TQ_KEY_SIGNED): s = fp16(max |x| / 1.5), mn = fp16(-1.5 s), q = clamp(rint((x - mn) / s),
 *         0, 3): the four levels (q - 1.5) s, symmetric about zero (up to the fp16 rounding of mn).
 * Both store (s, mn) per block of 32 and decode as mn + s q (IEEE fp32 arithmetic, ties to even). */
#define TQ_KEY_AFFINE 0
#define TQ_KEY_SIGNED 1

typedef struct tq_ctx tq_ctx;

/* Timing of the dominant kernels between tq_profile_begin and tq_profile_end
 * (CUDA events recorded on the launching stream around each launch). */
typedef struct {
  int64_t decode_launches; /* fused decode-attention main kernel */
  double decode_ms;
  int64_t encode_launches; /* encode / flush kernel (flush inside append included) */
  double encode_ms;
  int64_t merge_launches;  /* split-K merge kernel */
  double merge_ms;
  const char* decode_kernel; /* name of the decode kernel of the last decode call (static string), or NULL */
} tq_profile;

/* ------------------------------------------------------------------ setup */

/* Human-readable name of a status code (static string). */
const char* tq_status_string(tq_status s);

/* Fill *cfg with the main (key_bits 3 / value_bits 2) or alternate (8 / 3)
 * layout defaults: page 16, ring 128, group 32, qjl_m = head_dim (main).
 * key_bits / value_bits may be changed afterwards within the ranges above. */
tq_status tq_config_init(tq_config* cfg, int layout, int head_dim, int num_q_heads, int num_kv_heads,
                         uint64_t seed);

/* Check a configuration without creating a context and without any CUDA call:
 * TQ_OK, TQ_ERR_INVALID_ARG or TQ_ERR_UNSUPPORTED, the answer tq_create gives
 * for it.  When the configuration is valid and bytes_per_token_head is not
 * NULL, it receives the pool bytes one token of one KV head occupies (what
 * tq_bytes_per_token_head returns for a context made from it). */
tq_status tq_config_check(const tq_config* cfg, size_t* bytes_per_token_head);

/* Create a context on the current CUDA device.  Computes on the host the
 * Lloyd-Max codebook for the rotated-coordinate density of head_dim
 * (tq_lloyd_max) and the random tables of cfg->seed (tq_generate_tables),
 * then uploads them (a few KB; S is qjl_m x head_dim floats).  The context
 * owns those device tables and frees them in tq_destroy.  *out is set only on
 * success. */
tq_status tq_create(const tq_config* cfg, tq_ctx** out);

/* As tq_create, with caller-supplied host tables instead of the generated
 * ones: centroids [2^bits] ascending and antisymmetric (c[j] == -c[K-1-j],
 * bits = key_bits - 1 for main keys, value_bits for alt values), signs [head_dim] of +-1, sketch
 * [qjl_m][head_dim] row-major (main only; may be NULL for alt).  Decision
 * boundaries are the midpoints of consecutive centroids. */
tq_status tq_create_with_tables(const tq_config* cfg, const float* centroids, const float* signs,
                                const float* sketch, tq_ctx** out);

/* Free the context and its device tables.  NULL is ignored. */
void tq_destroy(tq_ctx* ctx);

/* Copy the context's tables to host arrays (any pointer may be NULL):
 * centroids [K], boundaries [K-1], signs [head_dim], sketch [qjl_m * head_dim]. */
tq_status tq_get_tables(const tq_ctx* ctx, float* centroids, float* boundaries, float* signs, float* sketch);

/* Host only, no CUDA.  Lloyd-Max codebook (float64) for one coordinate of a
 * uniformly rotated unit vector of dimension d (density proportional to
 * (1 - x^2)^((d-3)/2) on [-1, 1]; turboquant vLLM guide, section 2 step 2,
 * "Beta distribution" codebook): centroids [2^bits] ascending, boundaries
 * [2^bits - 1] = midpoints.  d >= 8, 1 <= bits <= 8 (5..8 bits: the 32- to
 * 256-level codebooks of the vllm-metal guide's q5_0 .. q8_0 value formats,
 * solved by Newton's method on the same fixed-point conditions). */
tq_status tq_lloyd_max(int d, int bits, double* centroids, double* boundaries);

/* Host only, no CUDA.  The random tables for a seed (SplitMix64 counter
 * stream + Box-Muller, this library's documented recipe): signs [d] (+-1) and,
 * if sketch != NULL, sketch [m][d] iid N(0, 1) rounded to float32. */
tq_status tq_generate_tables(uint64_t seed, int d, int m, float* signs, float* sketch);

/* Bytes one token of one KV head occupies in the pool (100 at main d = 128). */
size_t tq_bytes_per_token_head(const tq_ctx* ctx);

/* Bytes of one tile (one page of one KV head) = 16 * tq_bytes_per_token_head. */
size_t tq_page_bytes(const tq_ctx* ctx);

/* Workspace bytes tq_decode_attention needs for `batch` sequences whose
 * compressed lengths are all <= max_ctx tokens (for the decode path selected
 * when it is called: query the size again after tq_set_decode_path). */
tq_status tq_workspace_size(const tq_ctx* ctx, int batch, int max_ctx, size_t* bytes);

/* Select the main-layout decode kernels (TQ_DECODE_AUTO, TQ_DECODE_MMA_SYNC or
 * TQ_DECODE_TCGEN05).  The results agree within the decode tolerance; the
 * choice only changes speed and workspace size.  This switch has no
 * counterpart in the source pages: it exists to compare and test the two
 * tensor-core designs.  Host only; TQ_ERR_INVALID_ARG for another value. */
tq_status tq_set_decode_path(tq_ctx* ctx, int path);

/* ------------------------------------------------------------------ write path */

/* Encode (flush) n_tokens page-aligned tokens per (sequence, KV head) into
 * the pool: the encode kernel of the write path (turboquant-bench, "batch
 * flush" of 128 tokens; any multiple of 16 is accepted so that a prefix can
 * be compressed in one call).
 *   k, v        device fp16 [batch][Hkv][src_tokens][d], 16-byte aligned; tokens 0..n_tokens-1
 *               are read
 *   start_pos   device int32 [batch]: position of token 0, a multiple of 16
 *   block_table device int32 [batch][max_blocks]
 *   pool        device uint8 [num_blocks][Hkv][tq_page_bytes()], written
 * Tokens whose page falls outside the block table, or whose block id is not
 * in [0, num_blocks), are skipped and flagged in the device error word. */
tq_status tq_encode_flush(tq_ctx* ctx, const void* k, const void* v, int batch, int src_tokens, int n_tokens,
                          const int32_t* start_pos, const int32_t* block_table, int max_blocks, void* pool,
                          int num_blocks, cudaStream_t stream);

/* Append one decode token per sequence: the ring-buffer write of the decode
 * step with flush-on-overflow (turboquant vLLM guide, section 5.1: single
 * decode tokens go to a ring buffer of buffer_size = 128).
 *   k_new, v_new  device fp16 [batch][Hkv][d]
 *   pos           device int32 [batch]: position of the new token (its
 *                 sequence length before the append)
 *   ring_k/v      device fp16 [batch][Hkv][ring_capacity][d], 16-byte aligned; slot = pos % 128
 * If pos > 0 and pos % 128 == 0 the ring holds tokens pos-128 .. pos-1: they
 * are first encoded into the pool at positions pos-128.. (same kernel as
 * tq_encode_flush), then the new token is written to slot 0.  After the call
 * a sequence of length L = pos + 1 has n_compressed = 128 * ((L - 1) / 128)
 * compressed tokens and n_buf = L - n_compressed ring tokens. */
tq_status tq_append_token(tq_ctx* ctx, const void* k_new, const void* v_new, const int32_t* pos, int batch,
                          void* ring_k, void* ring_v, const int32_t* block_table, int max_blocks, void* pool,
                          int num_blocks, cudaStream_t stream);

/* ------------------------------------------------------------------ read path */

/* One decode step of attention for every query head (turboquant vLLM guide,
 * section 3 hybrid mode: compressed history + exact recent buffer; fused
 * scoring on packed indices without an fp16 intermediate, framework-status
 * survey, oMLX section).
 *   q             device fp16 [batch][Hq][d]
 *   pool          device uint8 [num_blocks][Hkv][page bytes]
 *   block_table   device int32 [batch][max_blocks]
 *   n_compressed  device int32 [batch]: compressed tokens (positions
 *                 0..n-1), a multiple of 16, at most max_ctx
 *   ring_k/ring_v device fp16 [batch][Hkv][ring_capacity][d]; may be NULL if
 *                 n_buf is NULL
 *   n_buf         device int32 [batch]: exact tokens in ring slots 0..n_buf-1
 *                 (0..128), or NULL for none
 *   out           device float32 [batch][Hq][d]
 *   workspace     device scratch of at least tq_workspace_size(batch, max_ctx)
 *                 bytes, 256-byte aligned
 * A sequence with no tokens at all gets an all-zero output row. */
tq_status tq_decode_attention(tq_ctx* ctx, const void* q, int batch, const void* pool, int num_blocks,
                              const int32_t* block_table, int max_blocks, const int32_t* n_compressed,
                              const void* ring_k, const void* ring_v, const int32_t* n_buf, int max_ctx,
                              float* out, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Decode attention without a caller-provided workspace.  This call has no
 * counterpart in the source pages; it exists for callers that cannot allocate
 * device memory when they decode, such as an engine that fixes its memory
 * budget before it starts serving, a caller recording its work into a CUDA
 * graph, or a host whose device allocator belongs to another runtime.
 * Arguments and results are those of tq_decode_attention minus the workspace.
 * The scratch is one file-scope device array of 16 MiB (16 << 20 bytes) that
 * every GPU which loads libtq holds until the process exits; a call whose
 * tq_workspace_size(batch, max_ctx) exceeds 16 MiB returns TQ_ERR_WORKSPACE
 * and launches nothing.  Every call made outside stream capture looks up the
 * current context's address of the array (cudaGetSymbolAddress, with the
 * device current) and remembers it per device; a call made while `stream` is
 * capturing uses the remembered address, so make one uncaptured call on a
 * device (again after cudaDeviceReset or a change of context) before
 * capturing; otherwise the captured call returns TQ_ERR_CUDA.  Arguments are
 * checked as by tq_decode_attention, in the same order, before the size.  The
 * call itself allocates no device memory.  All calls share the one array and it keeps the last call's
 * contents (nothing in it needs to start at zero): calls that can overlap on
 * the GPU (different streams, or different host threads without ordering)
 * race on it, so keep them ordered on one stream. */
tq_status tq_decode_attention_static(tq_ctx* ctx, const void* q, int batch, const void* pool, int num_blocks,
                                     const int32_t* block_table, int max_blocks, const int32_t* n_compressed,
                                     const void* ring_k, const void* ring_v, const int32_t* n_buf, int max_ctx,
                                     float* out, cudaStream_t stream);

/* Prefill materialisation: the compressed history read back as dense fp16
 * keys and values (vllm-metal TurboQuant guide, advanced settings: history
 * pages dequantised to fp16/bf16 before a long prefill).  Keys are the
 * reconstruction the decode estimator stands for, k^ = n_k D H x / sqrt(d)
 * with x = c[idx] + sqrt(pi/2)/m n_r S^T (2 sigma - 1) (turboquant vLLM
 * guide, section 2 steps 2-3); values are mn + s q (main layout); in the
 * alternate layout keys are mn + s q and values n_v D H c[idx] / sqrt(d)
 * (vllm-metal TurboQuant guide, quantisation table).
 *   pool, block_table, max_blocks, num_blocks   as for tq_decode_attention
 *   n_compressed  device int32 [batch]: tokens 0..n-1 read from the pool; a
 *                 multiple of 16, at most min(max_tokens, 16 max_blocks)
 *   ring_k/v      device fp16 [batch][Hkv][ring_capacity][d] and
 *   n_buf         device int32 [batch], or all NULL: ring slots
 *                 0..n_buf-1 are copied to rows n .. n+n_buf-1
 *   k_out, v_out  device fp16 [batch][Hkv][max_tokens][d], 16-byte aligned;
 *                 rows past n + n_buf are not written
 * Bad device values (lengths, block ids, ring counts) skip the affected rows
 * and set bits of the device error word. */
tq_status tq_dequantize(tq_ctx* ctx, const void* pool, int num_blocks, const int32_t* block_table, int max_blocks,
                        const int32_t* n_compressed, const void* ring_k, const void* ring_v, const int32_t* n_buf,
                        int batch, int max_tokens, void* k_out, void* v_out, cudaStream_t stream);

/* tq_dequantize with bfloat16 outputs (the guide's "FP16/BF16" materialisation): the same
 * reconstruction in fp32, rounded to nearest even bf16; k_out, v_out device bf16
 * [batch][Hkv][max_tokens][d]; ring rows are converted from fp16.  Same checks and errors. */
tq_status tq_dequantize_bf16(tq_ctx* ctx, const void* pool, int num_blocks, const int32_t* block_table,
                             int max_blocks, const int32_t* n_compressed, const void* ring_k, const void* ring_v,
                             const int32_t* n_buf, int batch, int max_tokens, void* k_out, void* v_out,
                             cudaStream_t stream);

/* Prefill admission rule of the materialisation (vllm-metal TurboQuant guide, advanced settings,
 * VLLM_METAL_TQ_PREFILL): a prefill chunk of query_tokens new tokens over history_tokens
 * compressed tokens materialises the history (tq_dequantize, then dense attention) when
 *   history_tokens >= 8192, and
 *   query_tokens >= 64 at head_dim 128 (the calibrated geometry), else >= max(128, head_dim / 2),
 *   and the dense K and V (history x num_kv_heads x head_dim x 2 tensors x 2 bytes) fit in
 *   max_mib MiB (VLLM_METAL_TQ_PREFILL_MAX_MIB: max_mib < 0 no cap, 0 never materialise).
 * Otherwise (decode steps, short suffixes) the compressed path stays.  Host only, no CUDA call.
 * Returns 1 (materialise), 0 (stay compressed) or -1 (negative counts, head_dim or heads <= 0). */
int tq_should_materialize(int64_t history_tokens, int64_t query_tokens, int head_dim, int num_kv_heads,
                          int64_t max_mib);

/* ------------------------------------------------------------------ bit packing */

/* Pack n codes (each < 2^bits, 1 <= bits <= 8) into a little-endian,
 * least-significant-bit-first stream: code i occupies stream bits
 * [bits*i, bits*i + bits), stream bit k is bit k % 8 of byte k / 8
 * (turboquant vLLM guide, section 2 step 5: four 2-bit values per byte).
 * dst receives ceil(n*bits/8) bytes.  Device pointers, asynchronous. */
tq_status tq_pack(const uint8_t* codes, int64_t n, int bits, void* dst, cudaStream_t stream);
/* Inverse of tq_pack: codes[i] = bits of value i.  Device pointers. */
tq_status tq_unpack(const void* src, int64_t n, int bits, uint8_t* codes, cudaStream_t stream);
/* Same two operations on host memory (no CUDA). */
tq_status tq_pack_host(const uint8_t* codes, int64_t n, int bits, void* dst);
tq_status tq_unpack_host(const void* src, int64_t n, int bits, uint8_t* codes);

/* ------------------------------------------------------------------ diagnostics */

/* Read and clear the device error word (synchronises `stream`). */
tq_status tq_get_device_errors(tq_ctx* ctx, uint32_t* flags, cudaStream_t stream);

/* Number of kernels this context has launched since creation. */
int64_t tq_launch_count(const tq_ctx* ctx);

/* Start recording CUDA events around the encode, decode and merge kernels
 * launched through ctx (at most 65536 launches per kind are recorded). */
tq_status tq_profile_begin(tq_ctx* ctx);
/* Stop recording, synchronise the recorded events and report their sums. */
tq_status tq_profile_end(tq_ctx* ctx, tq_profile* out);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
