// Device helpers shared by the kattn kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "kattn_internal.cuh"

namespace kattn {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Butterfly sum: every lane ends with the same value, summed in a fixed order.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Per-row int8 quantization ("Kestrel_VLLM - 18" §3.3 int8 query; cache
// fields §四): scale = f32(absmax)/127, q = clamp(rint_even(x/scale), +-127),
// zero row -> 0.  Both divisions are IEEE float32.
__device__ __forceinline__ float quant_scale(float amax) {
  return __fdiv_rn(amax, 127.0f);
}

__device__ __forceinline__ int quant_one(float x, float scale) {
  if (scale == 0.0f) return 0;
  int q = __float2int_rn(__fdiv_rn(x, scale));
  return max(-127, min(127, q));
}

__device__ __forceinline__ uint32_t pack_i8x4(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) |
         ((uint32_t)(c & 0xff) << 16) | ((uint32_t)(d & 0xff) << 24);
}

// One warp quantizes one 128-element float row: lane l owns elements
// 4l..4l+3.  Returns the packed int8x4 word for the lane and the scale.
__device__ __forceinline__ uint32_t warp_quantize_row(const float* __restrict__ row,
                                                      float* scale_out) {
  const int lane = threadIdx.x & 31;
  float4 x = reinterpret_cast<const float4*>(row)[lane];
  float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
  amax = warp_max(amax);
  float s = quant_scale(amax);
  *scale_out = s;
  return pack_i8x4(quant_one(x.x, s), quant_one(x.y, s), quant_one(x.z, s),
                   quant_one(x.w, s));
}

// One warp quantizes a 128-float row into cache row `dst` of the 2-D view
// [Hkv * cap_rows][128] (int8 bytes and the float scale).
__device__ __forceinline__ void warp_quantize_into_cache(const float* __restrict__ x_row,
                                                         int8_t* __restrict__ out_q,
                                                         float* __restrict__ out_scale,
                                                         int64_t dst) {
  float scale;
  const uint32_t w = warp_quantize_row(x_row, &scale);
  reinterpret_cast<uint32_t*>(out_q + dst * KATTN_HEAD_DIM)[threadIdx.x & 31] = w;
  if ((threadIdx.x & 31) == 0) out_scale[dst] = scale;
}

// Rounding of P before it multiplies V (susun-blog page, section "注意力权重").
__device__ __forceinline__ float e4m3_round(float x) {
  __nv_fp8_storage_t s = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
  __half_raw h = __nv_cvt_fp8_to_halfraw(s, __NV_E4M3);
  return __half2float(__half(h));
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// Row (b, column j) validity: the cache rows it reads must lie in the arrays.
__device__ __forceinline__ bool sequence_ok(int64_t rs, int ctx, int M, int cap_rows,
                                            int max_ctx) {
  return ctx >= 1 && ctx <= max_ctx && rs >= 0 &&
         rs + (int64_t)ctx + (int64_t)(M - 1) <= (int64_t)cap_rows;
}

// Whether every key of sequence b lies in the cache, in either layout: the
// contiguous rows [row_start, row_start + ctx + M - 1), or the first
// ceil((ctx + M - 1) / page) entries of its block-table row.  (The entries
// themselves are checked where they are read: paged_row.)
// In shard mode only the shard's keys must lie in the cache: the rows
// [row_start, row_start + n) for the n keys of windows [win_begin, win_begin
// + part_ws); a merge of shards checks ctx_len against the windows gathered.
__device__ __forceinline__ bool sequence_valid(const DecodeParams& p, int b) {
  const int ctx = p.ctx_len[b];
  if (p.merge_all)
    return ctx >= 1 && ctx <= p.max_ctx &&
           nsplit_for(ctx + p.M - 1) <= (int64_t)p.n_shards * p.part_ws;
  if (p.shard_mode) {
    if (ctx < 1 || ctx > p.max_ctx) return false;
    const int64_t k0 = (int64_t)p.win_begin * kSplitC;
    const int64_t k1 = min((int64_t)ctx + p.M - 1, k0 + (int64_t)p.part_ws * kSplitC);
    if (k1 <= k0) return true;                    // no key of b in this shard
    const int64_t rs = p.row_start[b];
    return rs >= 0 && rs + (k1 - k0) <= (int64_t)p.cap_rows;
  }
  if (p.block_table == nullptr) return sequence_ok(p.row_start[b], ctx, p.M, p.cap_rows, p.max_ctx);
  if (ctx < 1 || ctx > p.max_ctx) return false;
  const int64_t keys = (int64_t)ctx + p.M - 1;
  return ((keys + (1 << p.page_shift) - 1) >> p.page_shift) <= (int64_t)p.max_pages;
}

// Row of key `key` of sequence b within its kv-head plane (paged layout).  An
// entry outside the cache sets KATTN_DEVERR_BAD_PAGE and reads page 0, so no
// access leaves the arrays.
// The block-table entry of a key, and the row that entry gives it (an entry
// outside the plane flags KATTN_DEVERR_BAD_PAGE and reads page 0): apart, so
// that a caller can load the entry well before it needs the row.
__device__ __forceinline__ int page_entry(const DecodeParams& p, int b, int key) {
  return __ldg(p.block_table + (int64_t)b * p.max_pages + (key >> p.page_shift));
}
__device__ __forceinline__ int page_row_of(const DecodeParams& p, int page, int key) {
  if ((unsigned)page >= (unsigned)p.n_pages) {
    if (p.err_word) atomicOr(p.err_word, KATTN_DEVERR_BAD_PAGE);
    page = 0;
  }
  return (page << p.page_shift) | (key & ((1 << p.page_shift) - 1));
}
__device__ __forceinline__ int paged_row(const DecodeParams& p, int b, int key) {
  return page_row_of(p, page_entry(p, b, key), key);
}

// Row of key 0 of sequence b within its plane: the contiguous layout's
// row_start; 0 when paged (rows then come from paged_row).  In shard mode the
// cache holds the shard's keys from row_start on, so key t sits at row
// row_start + t - win_begin * kSplitC (this value may be negative; a key of
// the shard never is).
__device__ __forceinline__ int sequence_row0(const DecodeParams& p, int b) {
  if (p.block_table != nullptr) return 0;
  return (int)p.row_start[b] - (p.shard_mode ? p.win_begin * kSplitC : 0);
}

// Windows of sequence b (ctx_len ctx) that this call reduces: all of them,
// or in shard mode those of windows [win_begin, win_begin + part_ws).
__device__ __forceinline__ int local_windows(const DecodeParams& p, int ctx) {
  const int nw = nsplit_for(ctx + p.M - 1);
  return p.shard_mode ? min(max(nw - p.win_begin, 0), p.part_ws) : nw;
}

// ------------------------------------------------------------ cp.async ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte copy global -> shared; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)),
               "l"(src), "r"(src_bytes));
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(dst)),
               "l"(src), "r"(src_bytes));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

}  // namespace kattn
