// C ABI entry points (include/kattn.h): host-side validation and launches.
#include <cmath>
#include <cstring>

#include "kattn_internal.cuh"

using namespace kattn;

namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

float resolve_sm_scale(float sm_scale, int d) {
  // RN_f32(1/sqrt(d)): sqrt and the division are correctly rounded in double,
  // and for d = 128 the double is far from a float32 rounding tie.
  return sm_scale != 0.0f ? sm_scale : (float)(1.0 / std::sqrt((double)d));
}

// Shared argument checks of the decode entry points and kattn_qk_scores_debug.
// seq_rows is row_start (int64, contiguous layout) or block_table (int32,
// paged layout), aligned to seq_align bytes.
int check_common(const float* q, const int8_t* k, const float* k_scale, const void* seq_rows,
                 size_t seq_align, const int32_t* ctx_len, int B, int M, int Hq, int Hkv, int d,
                 int cap_rows, int max_ctx) {
  if (B < 0 || M < 1 || Hq < 1 || Hkv < 1 || cap_rows < 1 || max_ctx < 1)
    return KATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || B > 65535 || Hkv > 65535) return KATTN_ERR_INVALID_ARG;
  if (d != KATTN_HEAD_DIM) return KATTN_ERR_UNSUPPORTED;
  if (M > KATTN_MAX_M || (Hq / Hkv) * M > KATTN_MAX_ROWS) return KATTN_ERR_UNSUPPORTED;
  if ((int64_t)max_ctx + M - 1 > (int64_t)INT32_MAX / 2) return KATTN_ERR_INVALID_ARG;
  // the fast path addresses cache rows of all heads with int32 TMA coordinates
  if ((int64_t)Hkv * cap_rows > (int64_t)INT32_MAX - 4096) return KATTN_ERR_UNSUPPORTED;
  if (B == 0) return KATTN_OK;
  if (!q || !k || !k_scale || !seq_rows || !ctx_len) return KATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(k_scale, 4) || !aligned(seq_rows, seq_align) ||
      !aligned(ctx_len, 4))
    return KATTN_ERR_MISALIGNED;
  return KATTN_OK;
}

DecodeParams make_params(const float* q, const int8_t* k, const float* k_scale,
                         const int8_t* v, const float* v_scale, const int64_t* row_start,
                         const int32_t* ctx_len, int B, int M, int Hq, int Hkv, int cap_rows,
                         int max_ctx, float sm_scale, int p_mode, float* out) {
  DecodeParams p{};
  p.q = q;
  p.k = k;
  p.k_scale = k_scale;
  p.v = v;
  p.v_scale = v_scale;
  p.row_start = row_start;
  p.ctx_len = ctx_len;
  p.out = out;
  p.B = B;
  p.M = M;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.R = p.g * M;
  p.rpad = row_tile(p.R);
  p.row_groups = 1;
  p.cap_rows = cap_rows;
  p.max_ctx = max_ctx;
  p.nsplit_max = nsplit_for(max_ctx + M - 1);
  p.part_ws = p.nsplit_max;
  p.n_shards = 1;
  p.sm_scale = resolve_sm_scale(sm_scale, KATTN_HEAD_DIM);
  p.p_mode = p_mode;
  return p;
}

void set_workspace(DecodeParams& p, const WorkspaceLayout& w, void* workspace);

// The decode proper, once the layout-specific arguments are in p: the checks
// kattn_decode and kattn_decode_paged share, then the exact or the fast path.
int run_decode(DecodeParams& p, int p_mode, int exact_mode, float sm_scale, const int8_t* v,
               const float* v_scale, float* out, void* workspace, size_t workspace_bytes,
               void* stream) {
  if (p_mode < KATTN_P_F32 || p_mode > KATTN_P_E4M3_DIRECT) return KATTN_ERR_INVALID_ARG;
  if (exact_mode != 0 && exact_mode != 1) return KATTN_ERR_INVALID_ARG;
  if (exact_mode && p_mode == KATTN_P_E4M3_DIRECT) return KATTN_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return KATTN_ERR_INVALID_ARG;
  if (p.B == 0) return KATTN_OK;
  if (!v || !v_scale || !out) return KATTN_ERR_INVALID_ARG;
  if (!aligned(v, 16) || !aligned(v_scale, 4) || !aligned(out, 16)) return KATTN_ERR_MISALIGNED;
  cudaError_t e;
  if (exact_mode) {
    // no workspace needed; one that is given receives the device error bits
    if (workspace != nullptr) {
      if (!aligned(workspace, 256) || workspace_bytes < 256) return KATTN_ERR_WORKSPACE;
      p.err_word = static_cast<uint32_t*>(workspace);
    }
    e = launch_decode_exact(p, expf_constants(), as_stream(stream));
  } else {
    const WorkspaceLayout w = workspace_layout(p.B, p.M, p.Hq, p.max_ctx);
    // work items x kv heads are counted in int32 on the device
    if ((int64_t)p.B * w.nsplit_max * p.Hkv > (int64_t)INT32_MAX / 4) return KATTN_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < w.total)
      return KATTN_ERR_WORKSPACE;
    set_workspace(p, w, workspace);
    e = launch_decode_fast(p, as_stream(stream));
  }
  return e == cudaSuccess ? KATTN_OK : KATTN_ERR_CUDA;
}

void set_workspace(DecodeParams& p, const WorkspaceLayout& w, void* workspace) {
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.err_word = reinterpret_cast<uint32_t*>(ws);
  p.item_count = reinterpret_cast<uint32_t*>(ws + 4);
  p.prefix = reinterpret_cast<int*>(ws + w.prefix_off);
  p.items = reinterpret_cast<int4*>(ws + w.items_off);
  p.qpack = ws + w.q_off;
  p.partials = reinterpret_cast<float*>(ws + w.partials_off);
}

// The paged layout's own argument rules, and its fields of p.
int check_paging(int max_pages, int page_rows, int cap_rows) {
  if (max_pages < 1 || page_rows < 1) return KATTN_ERR_INVALID_ARG;
  // a TMA block of 32 keys must lie inside one page
  if (page_rows < kBlockBk || (page_rows & (page_rows - 1)) != 0) return KATTN_ERR_UNSUPPORTED;
  if (cap_rows % page_rows != 0) return KATTN_ERR_INVALID_ARG;
  return KATTN_OK;
}

void set_paging(DecodeParams& p, const int32_t* block_table, int max_pages, int page_rows,
                int cap_rows) {
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.page_shift = __builtin_ctz((unsigned)page_rows);
  p.n_pages = cap_rows / page_rows;
}

// The append and the decode of kattn_decode_append / kattn_decode_paged_append,
// once the layout's own checks are done and p holds the layout: the append
// rides in the decode's query-packing launch (fast mode).
int run_append(DecodeParams& p, const float* k_new, const float* v_new, const int64_t* dst_rows,
               int n_new, int64_t row_stride_elems, int8_t* k, float* k_scale, int8_t* v,
               float* v_scale, int p_mode, float sm_scale, float* out, void* workspace,
               size_t workspace_bytes, void* stream) {
  if (p_mode < KATTN_P_F32 || p_mode > KATTN_P_E4M3_DIRECT) return KATTN_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return KATTN_ERR_INVALID_ARG;
  if (n_new < 0 || row_stride_elems < (int64_t)p.Hkv * kD) return KATTN_ERR_INVALID_ARG;
  if (n_new > 0 && (!k_new || !v_new || !dst_rows)) return KATTN_ERR_INVALID_ARG;
  if (n_new > 0 && (!aligned(k_new, 16) || !aligned(v_new, 16) || row_stride_elems % 4 != 0 ||
                    !aligned(dst_rows, 8)))
    return KATTN_ERR_MISALIGNED;
  if (p.B == 0) {                                 // nothing to decode: the append alone
    if (n_new == 0) return KATTN_OK;
    int e = kattn_quantize_kv_rows(k_new, n_new, p.Hkv, kD, row_stride_elems, dst_rows, k, k_scale,
                                   p.cap_rows, stream);
    if (e != KATTN_OK) return e;
    return kattn_quantize_kv_rows(v_new, n_new, p.Hkv, kD, row_stride_elems, dst_rows, v, v_scale,
                                  p.cap_rows, stream);
  }
  if (!v || !v_scale || !out) return KATTN_ERR_INVALID_ARG;
  if (!aligned(v, 16) || !aligned(v_scale, 4) || !aligned(out, 16)) return KATTN_ERR_MISALIGNED;
  const WorkspaceLayout w = workspace_layout(p.B, p.M, p.Hq, p.max_ctx);
  if ((int64_t)p.B * w.nsplit_max * p.Hkv > (int64_t)INT32_MAX / 4) return KATTN_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < w.total)
    return KATTN_ERR_WORKSPACE;
  set_workspace(p, w, workspace);
  p.k_new = k_new;
  p.v_new = v_new;
  p.dst_rows = dst_rows;
  p.n_new = n_new;
  p.new_stride = row_stride_elems;
  p.k_w = k;
  p.ks_w = k_scale;
  p.v_w = v;
  p.vs_w = v_scale;
  const cudaError_t e = launch_decode_fast(p, as_stream(stream));
  return e == cudaSuccess ? KATTN_OK : KATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* kattn_status_string(int status) {
  switch (status) {
    case KATTN_OK: return "KATTN_OK";
    case KATTN_ERR_INVALID_ARG: return "KATTN_ERR_INVALID_ARG";
    case KATTN_ERR_UNSUPPORTED: return "KATTN_ERR_UNSUPPORTED";
    case KATTN_ERR_MISALIGNED: return "KATTN_ERR_MISALIGNED";
    case KATTN_ERR_WORKSPACE: return "KATTN_ERR_WORKSPACE";
    case KATTN_ERR_CUDA: return "KATTN_ERR_CUDA";
    default: return "KATTN_UNKNOWN_STATUS";
  }
}

int kattn_get_tiling(int* split_C, int* round_block_Bk) {
  if (split_C) *split_C = kSpanC;
  if (round_block_Bk) *round_block_Bk = kBlockBk;
  return KATTN_OK;
}

size_t kattn_decode_workspace_size(int B, int M, int Hq, int max_ctx) {
  if (B < 1 || M < 1 || M > KATTN_MAX_M || Hq < 1 || max_ctx < 1) return 0;
  return workspace_layout(B, M, Hq, max_ctx).total;
}

int kattn_expf_constants(double* out68) {
  if (!out68) return KATTN_ERR_INVALID_ARG;
  const ExpfConsts& c = expf_constants();
  out68[0] = c.K;
  out68[1] = c.C2;
  out68[2] = c.C0;
  out68[3] = c.C1;
  for (int j = 0; j < 64; ++j) out68[4 + j] = c.T[j];
  return KATTN_OK;
}

int kattn_quantize_kv(const float* x, int n_rows, int n_kv, int d, int64_t row_stride_elems,
                      int8_t* out_q, float* out_scale, int64_t dst_row0, int cap_rows,
                      void* stream) {
  if (n_rows < 0 || n_kv < 1 || cap_rows < 1 || dst_row0 < 0) return KATTN_ERR_INVALID_ARG;
  if (d != KATTN_HEAD_DIM) return KATTN_ERR_UNSUPPORTED;
  if (dst_row0 + (int64_t)n_rows > (int64_t)cap_rows) return KATTN_ERR_INVALID_ARG;
  if (row_stride_elems < (int64_t)n_kv * d) return KATTN_ERR_INVALID_ARG;
  if (n_rows == 0) return KATTN_OK;
  if (!x || !out_q || !out_scale) return KATTN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || row_stride_elems % 4 != 0 || !aligned(out_q, 16) ||
      !aligned(out_scale, 4))
    return KATTN_ERR_MISALIGNED;
  cudaError_t e = launch_quantize_kv(x, n_rows, n_kv, row_stride_elems, out_q, out_scale,
                                     dst_row0, nullptr, cap_rows, as_stream(stream));
  return e == cudaSuccess ? KATTN_OK : KATTN_ERR_CUDA;
}

int kattn_quantize_kv_rows(const float* x, int n_rows, int n_kv, int d,
                           int64_t row_stride_elems, const int64_t* dst_rows, int8_t* out_q,
                           float* out_scale, int cap_rows, void* stream) {
  if (n_rows < 0 || n_kv < 1 || cap_rows < 1) return KATTN_ERR_INVALID_ARG;
  if (d != KATTN_HEAD_DIM) return KATTN_ERR_UNSUPPORTED;
  if (row_stride_elems < (int64_t)n_kv * d) return KATTN_ERR_INVALID_ARG;
  if (n_rows == 0) return KATTN_OK;
  if (!x || !dst_rows || !out_q || !out_scale) return KATTN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || row_stride_elems % 4 != 0 || !aligned(dst_rows, 8) ||
      !aligned(out_q, 16) || !aligned(out_scale, 4))
    return KATTN_ERR_MISALIGNED;
  cudaError_t e = launch_quantize_kv(x, n_rows, n_kv, row_stride_elems, out_q, out_scale, 0,
                                     dst_rows, cap_rows, as_stream(stream));
  return e == cudaSuccess ? KATTN_OK : KATTN_ERR_CUDA;
}

int kattn_decode(const float* q, const int8_t* k, const float* k_scale, const int8_t* v,
                 const float* v_scale, const int64_t* row_start, const int32_t* ctx_len,
                 int B, int M, int Hq, int Hkv, int d, int cap_rows, int max_ctx,
                 float sm_scale, int p_mode, int exact_mode, float* out, void* workspace,
                 size_t workspace_bytes, void* stream) {
  int st = check_common(q, k, k_scale, row_start, 8, ctx_len, B, M, Hq, Hkv, d, cap_rows, max_ctx);
  if (st != KATTN_OK) return st;
  DecodeParams p = make_params(q, k, k_scale, v, v_scale, row_start, ctx_len, B, M, Hq, Hkv,
                               cap_rows, max_ctx, sm_scale, p_mode, out);
  return run_decode(p, p_mode, exact_mode, sm_scale, v, v_scale, out, workspace, workspace_bytes,
                    stream);
}

int kattn_decode_paged(const float* q, const int8_t* k, const float* k_scale, const int8_t* v,
                       const float* v_scale, const int32_t* block_table, int max_pages,
                       int page_rows, const int32_t* ctx_len, int B, int M, int Hq, int Hkv,
                       int d, int cap_rows, int max_ctx, float sm_scale, int p_mode,
                       int exact_mode, float* out, void* workspace, size_t workspace_bytes,
                       void* stream) {
  int st = check_common(q, k, k_scale, block_table, 4, ctx_len, B, M, Hq, Hkv, d, cap_rows,
                        max_ctx);
  if (st != KATTN_OK) return st;
  st = check_paging(max_pages, page_rows, cap_rows);
  if (st != KATTN_OK) return st;
  DecodeParams p = make_params(q, k, k_scale, v, v_scale, nullptr, ctx_len, B, M, Hq, Hkv,
                               cap_rows, max_ctx, sm_scale, p_mode, out);
  set_paging(p, block_table, max_pages, page_rows, cap_rows);
  return run_decode(p, p_mode, exact_mode, sm_scale, v, v_scale, out, workspace, workspace_bytes,
                    stream);
}

int kattn_decode_append(const float* q, const float* k_new, const float* v_new,
                        const int64_t* dst_rows, int n_new, int64_t row_stride_elems, int8_t* k,
                        float* k_scale, int8_t* v, float* v_scale, const int64_t* row_start,
                        const int32_t* ctx_len, int B, int M, int Hq, int Hkv, int d,
                        int cap_rows, int max_ctx, float sm_scale, int p_mode, float* out,
                        void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_common(q, k, k_scale, row_start, 8, ctx_len, B, M, Hq, Hkv, d, cap_rows, max_ctx);
  if (st != KATTN_OK) return st;
  DecodeParams p = make_params(q, k, k_scale, v, v_scale, row_start, ctx_len, B, M, Hq, Hkv,
                               cap_rows, max_ctx, sm_scale, p_mode, out);
  return run_append(p, k_new, v_new, dst_rows, n_new, row_stride_elems, k, k_scale, v, v_scale,
                    p_mode, sm_scale, out, workspace, workspace_bytes, stream);
}

int kattn_decode_paged_append(const float* q, const float* k_new, const float* v_new,
                              const int64_t* dst_rows, int n_new, int64_t row_stride_elems,
                              int8_t* k, float* k_scale, int8_t* v, float* v_scale,
                              const int32_t* block_table, int max_pages, int page_rows,
                              const int32_t* ctx_len, int B, int M, int Hq, int Hkv, int d,
                              int cap_rows, int max_ctx, float sm_scale, int p_mode, float* out,
                              void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_common(q, k, k_scale, block_table, 4, ctx_len, B, M, Hq, Hkv, d, cap_rows,
                        max_ctx);
  if (st != KATTN_OK) return st;
  st = check_paging(max_pages, page_rows, cap_rows);
  if (st != KATTN_OK) return st;
  DecodeParams p = make_params(q, k, k_scale, v, v_scale, nullptr, ctx_len, B, M, Hq, Hkv,
                               cap_rows, max_ctx, sm_scale, p_mode, out);
  set_paging(p, block_table, max_pages, page_rows, cap_rows);
  return run_append(p, k_new, v_new, dst_rows, n_new, row_stride_elems, k, k_scale, v, v_scale,
                    p_mode, sm_scale, out, workspace, workspace_bytes, stream);
}

int kattn_qk_scores_debug(const float* q, const int8_t* k, const float* k_scale,
                          const int64_t* row_start, const int32_t* ctx_len, int B, int M,
                          int Hq, int Hkv, int d, int cap_rows, int max_ctx, int32_t* scores,
                          int8_t* q_i8, float* q_scale, void* stream) {
  int st = check_common(q, k, k_scale, row_start, 8, ctx_len, B, M, Hq, Hkv, d, cap_rows, max_ctx);
  if (st != KATTN_OK) return st;
  if (B == 0) return KATTN_OK;
  if (!scores) return KATTN_ERR_INVALID_ARG;
  if (!aligned(scores, 4) || (q_i8 && !aligned(q_i8, 16)) || (q_scale && !aligned(q_scale, 4)))
    return KATTN_ERR_MISALIGNED;
  DecodeParams p = make_params(q, k, k_scale, nullptr, nullptr, row_start, ctx_len, B, M, Hq,
                               Hkv, cap_rows, max_ctx, 0.0f, 0, nullptr);
  cudaError_t e = launch_qk_debug(p, scores, q_i8, q_scale, as_stream(stream));
  return e == cudaSuccess ? KATTN_OK : KATTN_ERR_CUDA;
}

int kattn_decode_launch_count(int B, int M, int Hq, int Hkv, int max_ctx) {
  if (B < 1 || M < 1 || M > KATTN_MAX_M || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_ctx < 1 ||
      (Hq / Hkv) * M > KATTN_MAX_ROWS || (int64_t)max_ctx + M - 1 > (int64_t)INT32_MAX / 2)
    return 0;
  const DecodeParams p = make_params(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                     nullptr, B, M, Hq, Hkv, 1, max_ctx, 0.0f, 0, nullptr);
  return decode_launch_count(p);
}

size_t kattn_shard_partials_size(int B, int M, int Hq, int Hkv, int win_per_shard) {
  if (B < 1 || M < 1 || M > KATTN_MAX_M || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 ||
      win_per_shard < 1)
    return 0;
  const int R = Hq / Hkv * M;
  if (R > KATTN_MAX_ROWS) return 0;
  return (size_t)B * (size_t)win_per_shard * (size_t)Hkv * (size_t)partial_stride(R) *
         sizeof(float);
}

int kattn_decode_shard(const float* q, const int8_t* k, const float* k_scale, const int8_t* v,
                       const float* v_scale, const int64_t* row_start, const int32_t* ctx_len,
                       int B, int M, int Hq, int Hkv, int d, int cap_rows, int max_ctx, int shard,
                       int win_per_shard, float sm_scale, int p_mode, float* partials,
                       void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_common(q, k, k_scale, row_start, 8, ctx_len, B, M, Hq, Hkv, d, cap_rows, max_ctx);
  if (st != KATTN_OK) return st;
  if (shard < 0 || win_per_shard < 1) return KATTN_ERR_INVALID_ARG;
  // key positions of the shard are int32 on the device
  if (((int64_t)shard + 1) * win_per_shard * kSplitC > (int64_t)INT32_MAX / 2)
    return KATTN_ERR_INVALID_ARG;
  if (p_mode < KATTN_P_F32 || p_mode > KATTN_P_E4M3_DIRECT) return KATTN_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return KATTN_ERR_INVALID_ARG;
  if (B == 0) return KATTN_OK;
  if (!v || !v_scale || !partials) return KATTN_ERR_INVALID_ARG;
  if (!aligned(v, 16) || !aligned(v_scale, 4) || !aligned(partials, 16))
    return KATTN_ERR_MISALIGNED;
  DecodeParams p = make_params(q, k, k_scale, v, v_scale, row_start, ctx_len, B, M, Hq, Hkv,
                               cap_rows, max_ctx, sm_scale, p_mode, nullptr);
  const WorkspaceLayout w = workspace_layout(B, M, Hq, max_ctx);
  if ((int64_t)B * w.nsplit_max * Hkv > (int64_t)INT32_MAX / 4) return KATTN_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < w.total)
    return KATTN_ERR_WORKSPACE;
  set_workspace(p, w, workspace);
  p.partials = partials;                          // the caller's array, not the workspace's
  p.shard_mode = 1;
  p.win_begin = shard * win_per_shard;
  p.part_ws = win_per_shard;
  const cudaError_t e = launch_decode_fast(p, as_stream(stream));
  return e == cudaSuccess ? KATTN_OK : KATTN_ERR_CUDA;
}

int kattn_merge_shards(const float* partials, const int32_t* ctx_len, int B, int M, int Hq,
                       int Hkv, int d, int max_ctx, int n_shards, int win_per_shard, float* out,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || M < 1 || Hq < 1 || Hkv < 1 || max_ctx < 1 || n_shards < 1 || win_per_shard < 1)
    return KATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || B > 65535 || Hkv > 65535) return KATTN_ERR_INVALID_ARG;
  if (d != KATTN_HEAD_DIM) return KATTN_ERR_UNSUPPORTED;
  if (M > KATTN_MAX_M || (Hq / Hkv) * M > KATTN_MAX_ROWS) return KATTN_ERR_UNSUPPORTED;
  if ((int64_t)max_ctx + M - 1 > (int64_t)INT32_MAX / 2 ||
      (int64_t)n_shards * win_per_shard > (int64_t)INT32_MAX / 2)
    return KATTN_ERR_INVALID_ARG;
  if (B == 0) return KATTN_OK;
  if (!partials || !ctx_len || !out) return KATTN_ERR_INVALID_ARG;
  if (!aligned(partials, 16) || !aligned(ctx_len, 4) || !aligned(out, 16))
    return KATTN_ERR_MISALIGNED;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < 256) return KATTN_ERR_WORKSPACE;
  DecodeParams p{};
  p.ctx_len = ctx_len;
  p.out = out;
  p.partials = const_cast<float*>(partials);
  p.err_word = static_cast<uint32_t*>(workspace);
  p.B = B;
  p.M = M;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.R = p.g * M;
  p.max_ctx = max_ctx;
  p.part_ws = win_per_shard;
  p.n_shards = n_shards;
  p.merge_all = 1;
  const cudaError_t e = launch_merge(p, as_stream(stream));
  return e == cudaSuccess ? KATTN_OK : KATTN_ERR_CUDA;
}

int kattn_hash_rows(const void* data, int64_t n_rows, int64_t row_bytes, int64_t row_stride_bytes,
                    uint64_t* hashes, void* stream) {
  if (n_rows < 0 || row_bytes < 0 || row_stride_bytes < row_bytes) return KATTN_ERR_INVALID_ARG;
  if (n_rows == 0) return KATTN_OK;
  if (!data || !hashes) return KATTN_ERR_INVALID_ARG;
  if (!aligned(hashes, 8)) return KATTN_ERR_MISALIGNED;
  const cudaError_t e = launch_hash_rows(data, n_rows, row_bytes, row_stride_bytes, hashes,
                                         as_stream(stream));
  return e == cudaSuccess ? KATTN_OK : KATTN_ERR_CUDA;
}

int kattn_get_device_status(void* workspace, size_t workspace_bytes, int* device_err,
                            void* stream) {
  if (!workspace || !device_err || workspace_bytes < 256) return KATTN_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return KATTN_ERR_WORKSPACE;
  uint32_t word = 0;
  cudaStream_t s = as_stream(stream);
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return KATTN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KATTN_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(word), s) != cudaSuccess) return KATTN_ERR_CUDA;
  *device_err = (int)word;
  return KATTN_OK;
}

}  // extern "C"
