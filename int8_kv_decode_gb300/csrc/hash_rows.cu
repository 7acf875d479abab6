// Row hashes for parity dumps: FNV-1a 64 of every row of a device buffer.
//
// "Kestrel_VLLM - 18" §3.4 localises the first divergence between two runs
// by hashing buffers on both sides with the same FNV-1a 64 and comparing the
// lists.  Here one thread hashes one row (rows in parallel, bytes in order),
// so a buffer gives a list of row hashes and the first differing row is the
// first divergence.  The offset basis is FNV's 14695981039346656037; the
// page prints a truncation of it.
#include <cstdint>

#include <cuda_runtime.h>

#include "kattn_internal.cuh"

namespace kattn {
namespace {

constexpr uint64_t kFnvOffset = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;
constexpr int kThreads = 256;

__device__ __forceinline__ uint64_t fnv_byte(uint64_t h, uint32_t byte) {
  return (h ^ (uint64_t)byte) * kFnvPrime;
}

__global__ void __launch_bounds__(kThreads)
hash_rows_kernel(const uint8_t* __restrict__ data, int64_t n_rows, int64_t row_bytes,
                 int64_t stride, uint64_t* __restrict__ out) {
  for (int64_t r = (int64_t)blockIdx.x * kThreads + threadIdx.x; r < n_rows;
       r += (int64_t)gridDim.x * kThreads) {
    const uint8_t* row = data + r * stride;
    uint64_t h = kFnvOffset;
    int64_t i = 0;
    // 16-byte loads where the row start allows them, bytes in address order
    if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
      for (; i + 16 <= row_bytes; i += 16) {
        const uint4 w = *reinterpret_cast<const uint4*>(row + i);
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int s = 0; s < 32; s += 8) h = fnv_byte(h, (words[k] >> s) & 0xffu);
      }
    }
    for (; i < row_bytes; ++i) h = fnv_byte(h, row[i]);
    out[r] = h;
  }
}

}  // namespace

cudaError_t launch_hash_rows(const void* data, int64_t n_rows, int64_t row_bytes, int64_t stride,
                             uint64_t* out, cudaStream_t stream) {
  const int64_t blocks = (n_rows + kThreads - 1) / kThreads;
  hash_rows_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), kThreads, 0, stream>>>(
      static_cast<const uint8_t*>(data), n_rows, row_bytes, stride, out);
  return cudaGetLastError();
}

}  // namespace kattn
