// Integer QK scores for parity checks ("Kestrel_VLLM - 18" §3.3: int8 query
// quantization, int32 dot products against the int8 K rows).
// Grid: (key chunks of 128, M*Hq, B); one thread per key.
#include "device_common.cuh"

namespace kattn {
namespace {

__global__ void __launch_bounds__(128)
qk_debug_kernel(DecodeParams p, int32_t* __restrict__ scores, int8_t* __restrict__ q_i8,
                float* __restrict__ q_scale) {
  __shared__ __align__(16) uint32_t q8[kD / 4];
  const int b = blockIdx.z;
  const int j = blockIdx.y / p.Hq;
  const int h = blockIdx.y % p.Hq;
  const int kh = h / p.g;
  const int64_t rs = p.row_start[b];            // contiguous layout only
  const int ctx = p.ctx_len[b];
  if (!sequence_valid(p, b)) return;
  const int L = ctx + j;
  const int64_t qrow = ((int64_t)b * p.M + j) * p.Hq + h;
  if (threadIdx.x < 32) {
    float qs;
    const uint32_t w = warp_quantize_row(p.q + qrow * kD, &qs);
    q8[threadIdx.x] = w;
    if (blockIdx.x == 0) {
      if (q_i8) reinterpret_cast<uint32_t*>(q_i8 + qrow * kD)[threadIdx.x] = w;
      if (q_scale && threadIdx.x == 0) q_scale[qrow] = qs;
    }
  }
  __syncthreads();
  const int t = blockIdx.x * 128 + threadIdx.x;
  if (t >= L) return;
  const int4* krow = reinterpret_cast<const int4*>(p.k + ((int64_t)kh * p.cap_rows + rs + t) * kD);
  int acc = 0;
#pragma unroll
  for (int c = 0; c < kD / 16; ++c) {
    const int4 kv = krow[c];
    acc = __dp4a((int)kv.x, (int)q8[4 * c + 0], acc);
    acc = __dp4a((int)kv.y, (int)q8[4 * c + 1], acc);
    acc = __dp4a((int)kv.z, (int)q8[4 * c + 2], acc);
    acc = __dp4a((int)kv.w, (int)q8[4 * c + 3], acc);
  }
  const int width = p.max_ctx + p.M - 1;
  scores[qrow * width + t] = acc;
}

}  // namespace

cudaError_t launch_qk_debug(const DecodeParams& p, int32_t* scores, int8_t* q_i8,
                            float* q_scale, cudaStream_t stream) {
  dim3 grid((unsigned)((p.max_ctx + p.M - 1 + 127) / 128), (unsigned)(p.M * p.Hq),
            (unsigned)p.B);
  qk_debug_kernel<<<grid, 128, 0, stream>>>(p, scores, q_i8, q_scale);
  return cudaGetLastError();
}

}  // namespace kattn
