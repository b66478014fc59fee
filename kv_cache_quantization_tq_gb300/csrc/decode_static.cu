// tq_decode_attention_static: decode attention for callers that cannot
// allocate device memory.
//
// Some callers of this library may not call cudaMalloc at decode time: an
// engine that must not allocate once it is serving (fixed memory budget),
// work recorded into a CUDA graph where allocation is not allowed, or hosts
// whose allocator is owned by another runtime.  This entry point takes the
// same inputs and outputs as tq_decode_attention but no workspace: the
// split-K scratch lives in a file-scope device array of fixed size that every
// GPU loading the library holds until the process exits.
#include <mutex>

#include "tq_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)16 << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

// One array per device context (a __device__ variable is instantiated on every
// device that loads the module).  Host code must not pass &g_scratch to a kernel:
// on the host the name is only a stand-in; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch in the current device's context.  Outside stream capture the
// address is looked up again on every call (cudaGetSymbolAddress is cheap) and cached per device
// ordinal, so a context created after cudaDeviceReset, or another context made current on the
// device, is seen at its next uncaptured call; while `stream` is capturing, the cached address
// (from an earlier uncaptured call on this device) is used, and a device never set up fails.
cudaError_t scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  } else if (!g_addr[dev]) {
    return cudaErrorStreamCaptureUnsupported;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" tq_status tq_decode_attention_static(tq_ctx* ctx, const void* q, int batch, const void* pool,
                                                int num_blocks, const int32_t* block_table, int max_blocks,
                                                const int32_t* n_compressed, const void* ring_k, const void* ring_v,
                                                const int32_t* n_buf, int max_ctx, float* out, cudaStream_t stream) {
  // the argument checks of tq_decode_attention, in its order, before the scratch size
  if (!ctx || batch < 0 || max_blocks < 0 || num_blocks < 0 || max_ctx < 0) return TQ_ERR_INVALID_ARG;
  if (batch == 0) return TQ_OK;
  if (!q || !out || !n_compressed || !block_table || (max_ctx > 0 && !pool)) return TQ_ERR_INVALID_ARG;
  if (n_buf && (!ring_k || !ring_v)) return TQ_ERR_INVALID_ARG;
  if (max_ctx % tq::kPage) return TQ_ERR_INVALID_ARG;
  size_t need = 0;
  tq_status st = tq_workspace_size(ctx, batch, max_ctx, &need);
  if (st != TQ_OK) return st;
  if (need > kStaticScratchBytes) return TQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(stream, &scratch) != cudaSuccess) return TQ_ERR_CUDA;
  return tq_decode_attention(ctx, q, batch, pool, num_blocks, block_table, max_blocks, n_compressed, ring_k, ring_v,
                             n_buf, max_ctx, out, scratch, kStaticScratchBytes, stream);
}
