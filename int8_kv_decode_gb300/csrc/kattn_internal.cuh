// Internal declarations shared by the kattn CUDA translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "kattn.h"

namespace kattn {

constexpr int kD = KATTN_HEAD_DIM;    // head_dim
// Fast-path tiling (fixed at compile time, so a row's result never depends on
// the batch): keys are cut into spans of kSpanC at absolute positions; one
// warp reduces a span with its own running max, updated every kBlockBk keys
// (the rounding points of a rounded P).  A CTA owns kSpansPerCta consecutive
// spans and merges them; CTAs (windows of kSplitC keys) are merged last.
constexpr int kSpanC = 128;
constexpr int kBlockBk = 32;
constexpr int kSpansPerCta = 4;
constexpr int kSplitC = kSpanC * kSpansPerCta;   // 512 keys per CTA window
constexpr int kMaxRows = KATTN_MAX_ROWS;
constexpr int kMaxM = KATTN_MAX_M;
static_assert(kSpanC % kBlockBk == 0, "a span is a whole number of blocks");
static_assert(kSplitC == KATTN_WINDOW_KEYS, "the window of the public header");

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- workspace
// [0, 256)      header: uint32 error word at byte 0, uint32 work-item count at 4
// [X0, ...)     int32 prefix[B + 1]: work items (512-key window x kv head) of
//               the valid sequences before sequence b; prefix[B] is the total
// [I0, ...)     int4 work items, one per (valid sequence, window, kv head):
//               at most B * nsplit_max * Hkv <= B * nsplit_max * Hq
// [Q0, ...)     quantized queries per (b, kv head), rpad rows: rpad x 128 int8,
//               then rpad float32 scales (rows >= R are zero)
// [P0, ...)     float partials per (b, window, kv head): o[R][d], then m[R],
//               then l[R], padded to a multiple of 4 floats (16-byte rows)
// Only the header must be zero before the first call; the rest is written
// by every call before it is read.
struct WorkspaceLayout {
  size_t prefix_off, items_off, q_off, partials_off, total;
  int nsplit_max;
};

__host__ __device__ inline int nsplit_for(int keys) { return (keys + kSplitC - 1) / kSplitC; }

// Query rows a decode CTA holds: R rounded up to the row tile of its variant.
__host__ __device__ inline int row_tile(int R) {
  return R <= 8 ? 8 : R <= 16 ? 16 : R <= 32 ? 32 : R <= 48 ? 48 : 64;
}
__host__ __device__ inline int qpack_bytes(int rpad) { return rpad * (kD + 4); }
__host__ __device__ inline int partial_stride(int R) { return R * kD + ((2 * R + 3) / 4) * 4; }

inline WorkspaceLayout workspace_layout(int B, int M, int Hq, int max_ctx) {
  // Bounds that hold for every Hkv dividing Hq (R = Hq / Hkv * M):
  //   Hkv * row_tile(R) <= Hq * max(8, 2M);  Hkv * partial_stride(R) <= Hq * (M * 130 + 3).
  WorkspaceLayout w{};
  w.nsplit_max = nsplit_for(max_ctx + M - 1);
  const size_t nb = (size_t)B;
  w.prefix_off = 256;
  w.items_off = (w.prefix_off + (nb + 1) * sizeof(int) + 255) / 256 * 256;
  const size_t items = nb * (size_t)w.nsplit_max * (size_t)Hq * 16;
  w.q_off = (w.items_off + items + 255) / 256 * 256;
  const size_t qb = nb * (size_t)Hq * (size_t)(M > 4 ? 2 * M : 8) * (size_t)(kD + 4);
  w.partials_off = (w.q_off + qb + 255) / 256 * 256;
  const size_t part = nb * (size_t)w.nsplit_max * (size_t)Hq * (size_t)(M * (kD + 2) + 3) *
                      sizeof(float);
  w.total = (w.partials_off + part + 255) / 256 * 256;
  return w;
}

struct DecodeParams {
  const float* q;
  const int8_t* k;
  const float* k_scale;
  const int8_t* v;
  const float* v_scale;
  const int64_t* row_start;   // contiguous layout (block_table == nullptr)
  const int32_t* ctx_len;
  // Paged layout: key t of sequence b is row
  // (block_table[b * max_pages + (t >> page_shift)] << page_shift) + (t & (page - 1))
  // of its kv-head plane; n_pages = cap_rows >> page_shift.
  const int32_t* block_table;
  int max_pages, page_shift, n_pages;
  float* out;
  uint32_t* err_word;   // workspace header (fast mode), may be null in exact mode
  uint32_t* item_count; // workspace header + 4
  int* prefix;          // [B + 1]
  int4* items;
  uint8_t* qpack;
  float* partials;
  int B, M, Hq, Hkv, g, R;
  int rpad;             // row_tile(R)
  int row_groups;       // > 1: every work item split into this many units of
                        // 8 query rows, one CTA each (the one-tile kernel)
  int list_blocks;      // > 0: prepare_kernel writes the work items in this many blocks
  // Rows appended before the decode (kattn_decode_append), n_new = 0 if none:
  // row r of k_new / v_new goes to cache row dst_rows[r] of every kv head.
  const float* k_new;
  const float* v_new;
  const int64_t* dst_rows;
  int64_t new_stride;   // floats between rows of k_new / v_new
  int n_new;
  int8_t* k_w;          // the caches, writable (the same arrays as k, v)
  float* ks_w;
  int8_t* v_w;
  float* vs_w;
  int cap_rows, max_ctx, nsplit_max;
  float sm_scale;       // already resolved (never 0)
  int p_mode;
  // Window partials and context-parallel shards.  The partial of window w of
  // (b, kv head kh) sits at float offset partial_stride(R) times
  //   ((w / part_ws * B + b) * part_ws + w % part_ws) * Hkv + kh
  // of partials: part_ws = nsplit_max and one shard for kattn_decode; for
  // kattn_decode_shard / kattn_merge_shards, part_ws windows per sequence in
  // each of n_shards shards, shard s holding windows [s * part_ws, (s + 1) * part_ws).
  int part_ws;
  int n_shards;
  int win_begin;        // first window this call reduces (shard mode), else 0
  int shard_mode;       // 1: write every window's partial and nothing of out
  int merge_all;        // 1: merge every sequence (also single-window ones),
                        //    validating ctx_len only (kattn_merge_shards)
};

// Constants of the table-driven exp used by exact mode; computed on the host
// from first principles (see expf_constants.cpp) and passed by value.
struct ExpfConsts {
  double K, C2, C0, C1;
  double T[64];
};

const ExpfConsts& expf_constants();

// Launchers (return a cudaError_t of the launch).
cudaError_t launch_quantize_kv(const float* x, int n_rows, int n_kv, int64_t row_stride,
                               int8_t* out_q, float* out_scale, int64_t dst_row0,
                               const int64_t* dst_rows, int cap_rows, cudaStream_t stream);
cudaError_t launch_decode_fast(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream);
int decode_launch_count(const DecodeParams& p);   // kernels launch_decode_fast launches
cudaError_t launch_decode_exact(const DecodeParams& p, const ExpfConsts& c,
                                cudaStream_t stream);
cudaError_t launch_hash_rows(const void* data, int64_t n_rows, int64_t row_bytes, int64_t stride,
                             uint64_t* out, cudaStream_t stream);
cudaError_t launch_qk_debug(const DecodeParams& p, int32_t* scores, int8_t* q_i8,
                            float* q_scale, cudaStream_t stream);

}  // namespace kattn
