/*
 * kattn.h -- C ABI for decode attention over an int8-quantized KV cache
 * on NVIDIA GB300 (sm_103a).
 *
 * The operation (sources cited by page title and section):
 *
 *   "Kestrel_VLLM - 18 · 投机解码位级对拍收口" (wsisp.com)
 *     §3.3  decode attention with an int8 query quantized per head, int32
 *           QK dot products against int8 K rows, online softmax over the
 *           tokens, sequential P.V; and the table-driven expf used by the
 *           bit-exact variant.
 *     §二   speculative batch verify: draft column j of an M-column batch
 *           must reproduce, byte for byte, an M=1 decode that saw the same
 *           tokens.
 *     §四   the per-layer cache fields: int8 K/V rows with one float scale
 *           per row (_k _ks _v _vs).
 *   "在 agent 时代如何快速验证 kernel 对精度的影响" (susun-blog.com)
 *     section "注意力权重：直接转 fp8 随上下文变差，先放大就和 bf16 差不多":
 *           blockwise online softmax where only the P that multiplies V is
 *           rounded (f32 / bf16 / fp8 e4m3 / x448 then e4m3), the row sum
 *           uses the unrounded P, and the output is divided by it at the end.
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller; the
 *     library never frees or retains them.  No entry point allocates
 *     device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it; arguments are
 *     validated on the host before anything is enqueued, and an invalid
 *     call enqueues nothing.
 *   - The return value is a kattn_status (0 = success, < 0 = error).
 *     KATTN_ERR_CUDA means a CUDA runtime call (launch or copy) failed;
 *     the CUDA error is left for the caller to query.
 *   - Layouts are dense row-major with the sizes given.  head_dim d must
 *     be 128.  Pointers to int8 or float arrays must be 16-byte aligned.
 *   - Values must be finite; behaviour for NaN or Inf inputs is undefined
 *     (no fault, unspecified output).
 */
#ifndef KATTN_H
#define KATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status -- */
enum kattn_status {
  KATTN_OK = 0,
  KATTN_ERR_INVALID_ARG = -1, /* null pointer, negative or inconsistent size */
  KATTN_ERR_UNSUPPORTED = -2, /* d != 128, M > KATTN_MAX_M, g*M > KATTN_MAX_ROWS */
  KATTN_ERR_MISALIGNED = -3,  /* a pointer or stride is not 16-byte aligned */
  KATTN_ERR_WORKSPACE = -4,   /* workspace missing, too small or unaligned */
  KATTN_ERR_CUDA = -5         /* a CUDA runtime call failed */
};

/* P rounding applied to the weights that multiply V (the row sum always uses
 * the unrounded weight): see the susun-blog page, section "注意力权重". */
enum kattn_p_mode {
  KATTN_P_F32 = 0,      /* keep float32 */
  KATTN_P_BF16 = 1,     /* round to bfloat16, nearest-even */
  KATTN_P_E4M3 = 2,     /* round to fp8 e4m3 (OCP), nearest-even, saturating */
  KATTN_P_E4M3_X448 = 3, /* e4m3(p * 448) / 448 */
  KATTN_P_E4M3_X256 = 4, /* e4m3(p * 256) / 256 (both scalings exact in float32) */
  /* e4m3 P fed straight to the tensor-core P.V (the same page's closing
   * question; fast mode only).  p~ = e4m3(p); the P.V operand of key t is the
   * float32 product p~ * v_scale_t rounded once to 11 significant bits
   * (f16 precision, nearest-even), and V enters exact as f16.  That drops the
   * low-part MMA the other modes use to carry p~ * v_scale at 22 bits. */
  KATTN_P_E4M3_DIRECT = 5
};

#define KATTN_HEAD_DIM 128 /* the only supported head_dim */
#define KATTN_MAX_M 8      /* draft columns per sequence */
#define KATTN_MAX_ROWS 64  /* g * M query rows per (sequence, kv head) */
#define KATTN_WINDOW_KEYS 512 /* keys per window of the fast path's fixed tiling
                                 (the unit of kattn_decode_shard's shards) */

/* Device error bits reported by kattn_get_device_status. */
#define KATTN_DEVERR_BAD_SEQUENCE 0x1u /* row_start / ctx_len out of range */
#define KATTN_DEVERR_TIMEOUT 0x2u      /* a bounded wait inside a kernel ran out
                                          (a K/V copy, or exact mode's hand-off
                                          between its thread groups); the
                                          affected outputs are not written (fast
                                          mode) or are NaN (exact mode) */
#define KATTN_DEVERR_BAD_PAGE 0x4u     /* kattn_decode_paged: a block-table entry
                                          outside [0, cap_rows / page_rows) */

/* Human-readable name of a status code (static storage, never NULL). */
const char* kattn_status_string(int status);

/* Fixed tiling of the fast decode path.
 * *split_C: keys per split.  The keys of every sequence are cut into splits
 *   at absolute positions [s*C, (s+1)*C); each split is reduced on its own
 *   (with its own running max) and the splits are merged in split order.  C
 *   is a compile-time constant, so the result for a query row depends only
 *   on its own keys -- never on the batch size, M, or other sequences (batch
 *   invariance, "Kestrel_VLLM - 18" §二).
 * *round_block_Bk: keys per online-softmax block inside a split; the running
 *   max that a rounded P is taken relative to is updated once per block.
 * Either pointer may be NULL.  Never fails. */
int kattn_get_tiling(int* split_C, int* round_block_Bk);

/* Bytes of workspace kattn_decode needs for these sizes (fast mode; exact
 * mode needs none).  max_ctx is the host-side upper bound on ctx_len.
 * Returns 0 for invalid sizes.  Before the FIRST call with a workspace, the
 * caller must zero it (e.g. cudaMemsetAsync): its first 256 bytes hold the
 * device error word, which only kattn_get_device_status clears; the rest
 * (work list, quantized queries, per-window partials) is written by every
 * call before it is read.  One workspace may be reused by any number of
 * calls that are ordered on the GPU.  Calls that share a workspace and
 * overlap on the GPU race and give undefined results. */
size_t kattn_decode_workspace_size(int B, int M, int Hq, int max_ctx);

/* Kernels one fast-mode kattn_decode or kattn_decode_append call launches for
 * these sizes: the query packing (with the append and, up to 2048 sequences,
 * the work list), the work list above 2048 sequences, the split-KV pass, and
 * the window merge when max_ctx + M - 1 spans more than one 512-key window.
 * 0 for invalid sizes. */
int kattn_decode_launch_count(int B, int M, int Hq, int Hkv, int max_ctx);

/* Quantize K or V rows into the int8 cache ("Kestrel_VLLM - 18" §四 fields
 * _k/_ks, _v/_vs).  For each row r < n_rows and kv head h < n_kv:
 *   scale = f32(max_i |x[r][h][i]|) / 127                (IEEE division)
 *   q[i]  = clamp(rint_half_even(x[r][h][i] / scale), -127, 127); scale 0 -> 0
 *   out_q[(h*cap_rows + dst_row0 + r)*d + i] = q[i]
 *   out_scale[h*cap_rows + dst_row0 + r]     = scale
 * x:       float32, row r of head h at x + r*row_stride_elems + h*d
 *          (row_stride_elems >= n_kv*d, a multiple of 4).
 * out_q:   int8 cache [n_kv][cap_rows][d];  out_scale: float32 [n_kv][cap_rows].
 * Requires 0 <= dst_row0 and dst_row0 + n_rows <= cap_rows.  n_rows == 0 is
 * a no-op.  Bitwise deterministic. */
int kattn_quantize_kv(const float* x, int n_rows, int n_kv, int d,
                      int64_t row_stride_elems, int8_t* out_q, float* out_scale,
                      int64_t dst_row0, int cap_rows, void* stream);

/* Append form of kattn_quantize_kv: row r of x is quantized into cache row
 * dst_rows[r] of every kv head (one launch for rows scattered over many
 * sequences, e.g. the draft tokens of a decode step).
 * dst_rows: int64 [n_rows] on the device.  Because it lives on the device it
 * is checked there: a row whose index is outside [0, cap_rows) is skipped and
 * nothing is written for it.  Two rows with the same index race.  Other
 * arguments, the formula, alignment and errors as in kattn_quantize_kv. */
int kattn_quantize_kv_rows(const float* x, int n_rows, int n_kv, int d,
                           int64_t row_stride_elems, const int64_t* dst_rows, int8_t* out_q,
                           float* out_scale, int cap_rows, void* stream);

/* Decode attention ("Kestrel_VLLM - 18" §3.3; the susun-blog page, section
 * "注意力权重").  For sequence b < B, draft column j < M, query head h < Hq
 * (kv head kh = h / g, g = Hq / Hkv):
 *   (q8, qs)  = absmax/127 int8 quantization of q[b][j][h][:]
 *   L         = ctx_len[b] + j      (column j sees the context and drafts 0..j)
 *   keys t < L are cache rows row_start[b] + t of head kh
 *   S_t       = sum_i q8[i] * k[kh][row_start[b]+t][i]          (exact int32)
 *   s_t       = ((float)S_t * (qs * k_scale[kh][row])) * sm_scale
 *   out[b][j][h][:] = sum_t softmax(s)_t * (v_scale[kh][row] * v[kh][row][:])
 *   with P rounded per p_mode before it multiplies V.
 * q:         float32 [B][M][Hq][d].
 * k, v:      int8 [Hkv][cap_rows][d];  k_scale, v_scale: float32 [Hkv][cap_rows].
 * row_start: int64 [B] (device); ctx_len: int32 [B] (device), each >= 1 and
 *            <= max_ctx, with row_start[b] + ctx_len[b] + M - 1 <= cap_rows.
 *            These two arrays live on the device, so they are checked on the
 *            device: a sequence that breaks the rule gets NaN outputs and sets
 *            KATTN_DEVERR_BAD_SEQUENCE in the workspace (exact mode: in the
 *            workspace if one is given); no memory outside the arrays is
 *            touched.
 * max_ctx:   host-side upper bound on ctx_len (sizes the grid).
 * sm_scale:  0 selects RN_f32(1/sqrt(d)).
 * p_mode:    a kattn_p_mode (KATTN_P_E4M3_DIRECT with exact_mode = 1 ->
 *            KATTN_ERR_INVALID_ARG: the exact scan has no tensor-core operand).
 * exact_mode = 0 (fast): split-KV over spans of C keys, merged in a fixed
 *   order; float32 accumulation; deterministic run to run, and the bytes of
 *   out[b][j][h] depend only on that row's own keys, so column j equals an
 *   M=1 call with ctx_len + j, in any batch.  Needs a workspace of
 *   kattn_decode_workspace_size(B, M, Hq, max_ctx) bytes, 256-byte aligned.
 *   Up to three kernels on `stream` (query packing and work list, the
 *   split-KV pass, the window merge), chained by programmatic dependent
 *   launch; the call is capturable in a CUDA graph once a first call on the
 *   device has run outside capture.
 *   B * ceil((max_ctx + M - 1) / 512) * Hkv above 2^29 -> KATTN_ERR_UNSUPPORTED.
 * exact_mode = 1: one token at a time in token order; every float32
 *   operation rounded separately (no contraction); exp by the table-driven
 *   method of "Kestrel_VLLM - 18" §3.3 (64-entry 2^(j/64) table, 3-term
 *   polynomial, double fused multiply-adds).  Bit-exact against the CPU
 *   oracle's sequential emulation.  workspace may be NULL; if given (at
 *   least 256 bytes, 256-byte aligned, zeroed before its first use) only its
 *   error word is used: KATTN_DEVERR_BAD_SEQUENCE, and KATTN_DEVERR_TIMEOUT
 *   when a bounded hand-off wait between the kernel's thread groups ran out
 *   (that row's output is then NaN).
 * out:       float32 [B][M][Hq][d]. */
int kattn_decode(const float* q, const int8_t* k, const float* k_scale,
                 const int8_t* v, const float* v_scale, const int64_t* row_start,
                 const int32_t* ctx_len, int B, int M, int Hq, int Hkv, int d,
                 int cap_rows, int max_ctx, float sm_scale, int p_mode,
                 int exact_mode, float* out, void* workspace,
                 size_t workspace_bytes, void* stream);

/* kattn_decode over a paged cache: the same computation, with key t of
 * sequence b at row
 *   block_table[b * max_pages + t / page_rows] * page_rows + t % page_rows
 * of head kh's plane of k, v, k_scale, v_scale (shapes as kattn_decode;
 * cap_rows = pages * page_rows).  Keys sit at the same positions of the
 * fixed tiling as in the contiguous layout, so out equals, byte for byte,
 * kattn_decode on a cache holding the same rows contiguously.
 * block_table: int32 [B][max_pages] on the device, 4-byte aligned.
 * page_rows:   32 * 2^k (a 32-key TMA block never crosses a page), dividing
 *              cap_rows; other powers of two or smaller pages ->
 *              KATTN_ERR_UNSUPPORTED.
 * Checked on the device: ctx_len[b] in [1, max_ctx] and
 *   ceil((ctx_len[b] + M - 1) / page_rows) <= max_pages, else NaN outputs
 *   and KATTN_DEVERR_BAD_SEQUENCE as in kattn_decode; a table entry read
 *   outside [0, cap_rows / page_rows) sets KATTN_DEVERR_BAD_PAGE (fast mode)
 *   and reads page 0 instead: the outputs of that sequence are then
 *   unspecified, and no access leaves the arrays.
 * Other arguments, modes, workspace and errors as kattn_decode. */
int kattn_decode_paged(const float* q, const int8_t* k, const float* k_scale, const int8_t* v,
                       const float* v_scale, const int32_t* block_table, int max_pages,
                       int page_rows, const int32_t* ctx_len, int B, int M, int Hq, int Hkv,
                       int d, int cap_rows, int max_ctx, float sm_scale, int p_mode,
                       int exact_mode, float* out, void* workspace, size_t workspace_bytes,
                       void* stream);

/* One decode step with its KV append: kattn_quantize_kv_rows of k_new into
 * (k, k_scale) and of v_new into (v, v_scale), then kattn_decode in fast mode
 * (exact_mode = 0), in fewer launches -- the append runs inside the decode's
 * query-packing launch, so the decode reads the rows it has just written.
 * k_new, v_new: float32 [n_new][Hkv][d], row r at + r*row_stride_elems;
 * dst_rows: int64 [n_new] on the device (out-of-range rows are skipped, as in
 * kattn_quantize_kv_rows).  For the new rows to be attended, the caller gives
 * them cache rows inside the sequences' visible ranges (e.g. the M draft rows
 * of each sequence, row_start[b] + ctx_len[b] - 1 + j).  The cache bytes and
 * `out` equal those of the separate calls, byte for byte.  Other arguments,
 * workspace and errors as kattn_decode; n_new = 0 is a plain decode. */
int kattn_decode_append(const float* q, const float* k_new, const float* v_new,
                        const int64_t* dst_rows, int n_new, int64_t row_stride_elems,
                        int8_t* k, float* k_scale, int8_t* v, float* v_scale,
                        const int64_t* row_start, const int32_t* ctx_len, int B, int M, int Hq,
                        int Hkv, int d, int cap_rows, int max_ctx, float sm_scale, int p_mode,
                        float* out, void* workspace, size_t workspace_bytes, void* stream);

/* kattn_decode_append over a paged cache: the step's K/V rows quantized into
 * the pool and kattn_decode_paged in fast mode, in the same launches as
 * kattn_decode_paged (the append rides in the query-packing launch).
 * dst_rows are PHYSICAL rows of the pool, as for kattn_quantize_kv_rows: the
 * caller maps key t of sequence b through its block table,
 *   block_table[b * max_pages + t / page_rows] * page_rows + t % page_rows,
 * and for the rows to be attended, t lies inside the keys a column sees
 * (e.g. the M draft keys ctx_len[b] - 1 + j).  Out-of-range rows are skipped
 * on the device.  The cache bytes and `out` equal, byte for byte, those of
 * kattn_quantize_kv_rows twice followed by kattn_decode_paged.  Paging
 * arguments as kattn_decode_paged; append arguments as kattn_decode_append. */
int kattn_decode_paged_append(const float* q, const float* k_new, const float* v_new,
                              const int64_t* dst_rows, int n_new, int64_t row_stride_elems,
                              int8_t* k, float* k_scale, int8_t* v, float* v_scale,
                              const int32_t* block_table, int max_pages, int page_rows,
                              const int32_t* ctx_len, int B, int M, int Hq, int Hkv, int d,
                              int cap_rows, int max_ctx, float sm_scale, int p_mode, float* out,
                              void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------ context parallel -- */
/* One sequence's keys spread over several GPUs (context parallelism): every
 * GPU reduces the 512-key windows it holds into window partials, the
 * partials are all-gathered, and kattn_merge_shards combines them in the
 * same fixed order as kattn_decode.  Each window's partial is computed
 * exactly as kattn_decode computes it, so the merged output equals, byte for
 * byte, kattn_decode (fast mode) on one cache holding every key.  The pages
 * fix only that the combine order must not depend on the batch
 * ("Kestrel_VLLM - 18", §二); the window tiling is kattn_get_tiling's.
 *
 * Shards: windows are cut at absolute key positions, 512 keys each (window w
 * holds keys [512w, 512w + 512) of a sequence's ctx_len + M - 1 keys).  Shard
 * s holds windows [s*Ws, (s+1)*Ws) of EVERY sequence, Ws = win_per_shard; a
 * merge needs n_shards*Ws >= ceil((ctx_len[b] + M - 1) / 512) for every b.
 *
 * Byte size of one shard's partials array, float32
 * [B][Ws][Hkv][stride], stride = g*M*(d+2) rounded up to a multiple of 4
 * (o[g*M][d], then m[g*M], then l[g*M]); 0 for invalid arguments. */
size_t kattn_shard_partials_size(int B, int M, int Hq, int Hkv, int win_per_shard);

/* The window partials of shard `shard` (fast mode).  This shard's cache holds
 * key t of sequence b, for t in [512*shard*Ws, min(512*(shard+1)*Ws,
 * ctx_len[b] + M - 1)), at row row_start[b] + t - 512*shard*Ws of every kv-head
 * plane of k, v, k_scale, v_scale (shapes as kattn_decode); sequences with no
 * key in the shard are skipped and row_start[b] is not read.  q, ctx_len
 * (the GLOBAL context lengths), M, heads, max_ctx, sm_scale and p_mode are the
 * same on every shard.  partials: float32 [B][Ws][Hkv][stride] (16-byte
 * aligned): the partial of the shard's window w of (b, kh) at [b][w - shard*Ws][kh];
 * entries for windows a sequence does not have are left untouched.
 * workspace: kattn_decode_workspace_size(B, M, Hq, max_ctx) bytes, as for
 * kattn_decode.  A sequence whose shard rows leave [0, cap_rows) or whose
 * ctx_len is outside [1, max_ctx] gets o = NaN, m = +inf, l = NaN in every
 * window of the shard, so its merged rows are NaN, and KATTN_DEVERR_BAD_SEQUENCE
 * in this workspace's error word.  Errors as kattn_decode; exact mode and the
 * paged layout are not offered here. */
int kattn_decode_shard(const float* q, const int8_t* k, const float* k_scale, const int8_t* v,
                       const float* v_scale, const int64_t* row_start, const int32_t* ctx_len,
                       int B, int M, int Hq, int Hkv, int d, int cap_rows, int max_ctx, int shard,
                       int win_per_shard, float sm_scale, int p_mode, float* partials,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Combination of the gathered partials into out: partials float32
 * [n_shards][B][Ws][Hkv][stride] (shard-major, as an all-gather of the
 * shards' arrays leaves them), ctx_len int32 [B] on the device, out float32
 * [B][M][Hq][d].  Row (b, j, h) combines the windows of its own ctx_len[b] + j
 * keys: m = max of the window maxima, weights e^(m_w - m), window sums in an
 * order fixed by the window count alone, then out = o / l.  workspace: at
 * least 256 bytes (only its error word is used; a decode workspace will do).
 * A sequence with ctx_len outside [1, max_ctx], or with more windows than
 * n_shards*Ws, gets NaN rows and KATTN_DEVERR_BAD_SEQUENCE. */
int kattn_merge_shards(const float* partials, const int32_t* ctx_len, int B, int M, int Hq,
                       int Hkv, int d, int max_ctx, int n_shards, int win_per_shard, float* out,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free form of kattn_decode in fast mode (exact_mode = 0).  The
 * pages have no counterpart to it: it exists for callers that cannot give the
 * library a workspace -- an engine whose device memory belongs to its own
 * arena, a serving loop that must not pay cudaMalloc's latency and implicit
 * synchronisation between steps, or a plugin interface that receives only
 * input and output buffers.  The caller passes inputs and outputs exactly as
 * for kattn_decode; the scratch (work list, quantized queries and per-window
 * partials) lives in one device array of KATTN_NOALLOC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until the process
 * exits.  The call allocates nothing and calls no allocating routine.
 *   - Limit: calls whose kattn_decode_workspace_size(B, M, Hq, max_ctx)
 *     exceeds KATTN_NOALLOC_SCRATCH_BYTES are rejected with
 *     KATTN_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device looks up the array's address on that device
 *     (with that device current); make that first call before any stream
 *     capture begins.  If the lookup fails the call returns KATTN_ERR_CUDA
 *     and the next call on that device tries the lookup again.
 *   - Each call clears the array's error word on `stream` (cudaMemsetAsync)
 *     before decoding; the array keeps the rest of the last call's contents.
 *   - All calls on a device share the one array: calls that overlap on the
 *     GPU (for example on two streams) race and give undefined results, so
 *     the caller must order them.
 *   - Device error bits are not reported (the array is private); sequences
 *     that break the row_start / ctx_len rule still get NaN outputs.
 * Arguments, results, determinism and errors otherwise as kattn_decode. */
#define KATTN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int kattn_decode_noalloc(const float* q, const int8_t* k, const float* k_scale,
                         const int8_t* v, const float* v_scale, const int64_t* row_start,
                         const int32_t* ctx_len, int B, int M, int Hq, int Hkv, int d,
                         int cap_rows, int max_ctx, float sm_scale, int p_mode, float* out,
                         void* stream);

/* Integer QK scores of the decode path, for parity checks ("Kestrel_VLLM -
 * 18" §3.3: int8 query quantization + int32 QK dot product).
 * scores: int32 [B][M][Hq][max_ctx + M - 1]; entry t of row (b, j, h) is
 *   written for t < ctx_len[b] + j and left untouched otherwise.
 * q_i8:   optional int8 [B][M][Hq][d] quantized queries (NULL to skip).
 * q_scale: optional float32 [B][M][Hq] query scales (NULL to skip).
 * Other arguments as in kattn_decode.  Sequences that break the row_start /
 * ctx_len rule are skipped (their scores are left untouched). */
int kattn_qk_scores_debug(const float* q, const int8_t* k, const float* k_scale,
                          const int64_t* row_start, const int32_t* ctx_len, int B,
                          int M, int Hq, int Hkv, int d, int cap_rows, int max_ctx,
                          int32_t* scores, int8_t* q_i8, float* q_scale, void* stream);

/* The constants exact mode uses for its table-driven exp ("Kestrel_VLLM - 18"
 * §3.3), as the library derived them on the host: out68[0..3] = K = RN(64/ln2),
 * C2 = RN(ln2/64), C0 = RN(1/6), C1 = 1/2; out68[4 + j] = RN(2^(j/64)) for
 * j < 64.  Host only; for parity checks.  Returns KATTN_ERR_INVALID_ARG if
 * out68 is NULL. */
int kattn_expf_constants(double* out68);

/* Row hashes for parity dumps ("Kestrel_VLLM - 18" §3.4: hash buffers on
 * both sides with the same FNV-1a 64, compare the lists, and the first
 * difference localises the divergence).  hashes[r] = FNV-1a 64 (offset basis
 * 14695981039346656037, prime 1099511628211) of the row_bytes bytes at
 * data + r * row_stride_bytes, in address order.  data, hashes: device
 * pointers (hashes 8-byte aligned, n_rows entries).  The library has no
 * counterpart in the pages' decode path; it is test tooling. */
int kattn_hash_rows(const void* data, int64_t n_rows, int64_t row_bytes, int64_t row_stride_bytes,
                    uint64_t* hashes, void* stream);

/* Read (and clear) the device error word of a decode workspace.  Copies 4
 * bytes to the host and waits for `stream`.  *device_err receives the
 * KATTN_DEVERR_* bits set by calls since the last read. */
int kattn_get_device_status(void* workspace, size_t workspace_bytes,
                            int* device_err, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KATTN_H */
