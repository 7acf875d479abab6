// KV row quantization into the int8 cache ("Kestrel_VLLM - 18" §四: int8
// K/V rows with one float scale per row).  One warp per (row, kv head).
#include "device_common.cuh"

namespace kattn {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
quantize_kv_kernel(const float* __restrict__ x, int n_rows, int n_kv, int64_t row_stride,
                   int8_t* __restrict__ out_q, float* __restrict__ out_scale,
                   int64_t dst_row0, const int64_t* __restrict__ dst_rows, int cap_rows) {
  const int64_t item = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (item >= (int64_t)n_rows * n_kv) return;
  const int r = (int)(item / n_kv);
  const int h = (int)(item % n_kv);
  // Destination row: contiguous from dst_row0, or scattered by dst_rows[r]
  // (checked here because the index array lives on the device).
  const int64_t row = dst_rows ? dst_rows[r] : dst_row0 + r;
  if (row < 0 || row >= cap_rows) return;
  warp_quantize_into_cache(x + (int64_t)r * row_stride + (int64_t)h * kD, out_q, out_scale,
                           (int64_t)h * cap_rows + row);
}

}  // namespace

cudaError_t launch_quantize_kv(const float* x, int n_rows, int n_kv, int64_t row_stride,
                               int8_t* out_q, float* out_scale, int64_t dst_row0,
                               const int64_t* dst_rows, int cap_rows, cudaStream_t stream) {
  const int64_t items = (int64_t)n_rows * n_kv;
  const int64_t blocks = (items + kWarps - 1) / kWarps;
  quantize_kv_kernel<<<(unsigned)blocks, kWarps * 32, 0, stream>>>(
      x, n_rows, n_kv, row_stride, out_q, out_scale, dst_row0, dst_rows, cap_rows);
  return cudaGetLastError();
}

}  // namespace kattn
