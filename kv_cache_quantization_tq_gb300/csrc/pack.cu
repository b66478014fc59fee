// Generic low-bit packing (turboquant vLLM guide, section 2 step 5: four
// 2-bit values per byte; "TurboQuant-MLX overview": 3-bit indices).  Code i
// occupies stream bits [bits*i, bits*i + bits), least significant first;
// stream bit k is bit k % 8 of byte k / 8.
#include "common.cuh"

namespace tq {
namespace {

// One thread per output byte: OR together the slices of every code that
// overlaps the byte.
__global__ void pack_kernel(const uint8_t* __restrict__ codes, int64_t n, int bits, uint8_t* __restrict__ dst,
                            int64_t nbytes) {
  const unsigned mask = (1u << bits) - 1u;
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < nbytes; j += (int64_t)gridDim.x * blockDim.x) {
    const int64_t lo = (8 * j) / bits;
    int64_t hi = (8 * j + 7) / bits;
    if (hi >= n) hi = n - 1;
    unsigned out = 0;
    for (int64_t i = lo; i <= hi; ++i) {
      const int64_t shift = bits * i - 8 * j;  // may be negative for the first code
      const unsigned c = codes[i] & mask;
      out |= shift >= 0 ? (c << shift) : (c >> (-shift));
    }
    dst[j] = (uint8_t)(out & 0xFFu);
  }
}

__global__ void unpack_kernel(const uint8_t* __restrict__ src, int64_t n, int bits, uint8_t* __restrict__ codes,
                              int64_t nbytes) {
  const unsigned mask = (1u << bits) - 1u;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bit = bits * i;
    unsigned v = src[bit >> 3];
    if ((bit >> 3) + 1 < nbytes) v |= (unsigned)src[(bit >> 3) + 1] << 8;
    codes[i] = (uint8_t)((v >> (bit & 7)) & mask);
  }
}

int grid_for(int64_t work) {
  const int64_t g = (work + 255) / 256;
  return (int)(g < 152 * 16 ? (g < 1 ? 1 : g) : 152 * 16);
}

}  // namespace

cudaError_t launch_pack(const uint8_t* codes, int64_t n, int bits, void* dst, cudaStream_t s) {
  const int64_t nbytes = (n * bits + 7) / 8;
  pack_kernel<<<grid_for(nbytes), 256, 0, s>>>(codes, n, bits, static_cast<uint8_t*>(dst), nbytes);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const void* src, int64_t n, int bits, uint8_t* codes, cudaStream_t s) {
  const int64_t nbytes = (n * bits + 7) / 8;
  unpack_kernel<<<grid_for(n), 256, 0, s>>>(static_cast<const uint8_t*>(src), n, bits, codes, nbytes);
  return cudaGetLastError();
}

}  // namespace tq
