// The fast decode's launch chain: prepare_kernel (query packing, KV append,
// work list), list_kernel, the split-KV pass (decode_split.cuh) and
// merge_windows_kernel, and the host code that launches them.
#include "decode_split.cuh"

namespace kattn {
namespace {

// ------------------------------------------------------------------ prepare
// Blocks [0, q_blocks): one warp per packed query row (b, kv head, r < rpad):
// row r < R is query (column j = r / g, head kh * g + r % g) quantized per
// row, rows r >= R are zero.  The next a_blocks quantize the rows appended by
// kattn_decode_append into the cache, one warp per (row, kv head, K or V).
// The blocks after those write the work list (or, above kFusedListMaxB
// sequences, one block writes its prefix for list_kernel).
constexpr int kPrepWarps = 4;
constexpr int kFusedListMaxB = 2048;              // prepare writes the list itself up to here
constexpr int kListPerBlock = 1024;               // items per list block of prepare

__global__ void __launch_bounds__(kPrepWarps * 32) prepare_kernel(const DecodeParams p,
                                                                  int q_blocks, int a_blocks) {
  griddep_launch_dependents();                    // the decode grid may start its set-up
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if ((int)blockIdx.x >= q_blocks && (int)blockIdx.x < q_blocks + a_blocks) {
    // Appended rows: warp (r, kv head, K or V), as kattn_quantize_kv_rows.
    const int64_t idx = (int64_t)((int)blockIdx.x - q_blocks) * kPrepWarps + warp;
    if (idx >= (int64_t)p.n_new * p.Hkv * 2) return;
    const int which = (int)(idx & 1);
    const int64_t rh = idx >> 1;
    const int r = (int)(rh / p.Hkv), h = (int)(rh % p.Hkv);
    const int64_t row = p.dst_rows[r];
    if (row < 0 || row >= p.cap_rows) return;     // checked here: the index array is on the device
    const float* src = (which ? p.v_new : p.k_new) + (int64_t)r * p.new_stride + (int64_t)h * kD;
    warp_quantize_into_cache(src, which ? p.v_w : p.k_w, which ? p.vs_w : p.ks_w,
                             (int64_t)h * p.cap_rows + row);
    return;
  }
  if ((int)blockIdx.x < q_blocks) {
    const int64_t idx = (int64_t)blockIdx.x * kPrepWarps + warp;
    if (idx >= (int64_t)p.B * p.Hkv * p.rpad) return;
    const int r = (int)(idx % p.rpad);
    const int64_t bk = idx / p.rpad;
    const int kh = (int)(bk % p.Hkv), b = (int)(bk / p.Hkv);
    uint8_t* pack = p.qpack + bk * qpack_bytes(p.rpad);
    uint32_t w = 0;
    float s = 0.0f;
    if (r < p.R) {
      const int j = r / p.g, h = kh * p.g + r % p.g;
      const int64_t orow = (((int64_t)b * p.M + j) * p.Hq + h) * kD;
      if (sequence_valid(p, b)) {
        w = warp_quantize_row(p.q + orow, &s);
      } else {
        const float nan = __int_as_float(0x7fc00000);
        if (p.shard_mode) {
          // every window partial of the row: o = NaN, m = +inf, l = NaN, so
          // that a merge over the gathered shards yields NaN for the row
          for (int wl = 0; wl < p.part_ws; ++wl) {
            float* part = p.partials + (((size_t)b * p.part_ws + wl) * p.Hkv + kh) * partial_stride(p.R);
            reinterpret_cast<float4*>(part + (size_t)r * kD)[lane] = make_float4(nan, nan, nan, nan);
            if (lane == 0) {
              part[(size_t)p.R * kD + r] = INFINITY;
              part[(size_t)p.R * kD + p.R + r] = nan;
            }
          }
        } else {
          reinterpret_cast<float4*>(p.out + orow)[lane] = make_float4(nan, nan, nan, nan);
        }
        if (r == 0 && kh == 0 && lane == 0) atomicOr(p.err_word, KATTN_DEVERR_BAD_SEQUENCE);
      }
    }
    reinterpret_cast<uint32_t*>(pack + r * kD)[lane] = w;
    if (lane == 0) reinterpret_cast<float*>(pack + p.rpad * kD)[r] = s;
    return;
  }
  // prefix[b] = work items (windows x kv heads) of the valid sequences
  // before b.  Thread i takes a run of consecutive sequences, counts them,
  // the runs are scanned across the block, and each thread writes its run --
  // into shared memory (a list block: B <= kFusedListMaxB) or global memory
  // (the one prefix block for list_kernel).
  constexpr int kThreads = kPrepWarps * 32;
  __shared__ int s_warp[kPrepWarps];
  __shared__ int s_pre[kFusedListMaxB + 1];
  const bool fused = p.list_blocks > 0;
  int* pre = fused ? s_pre : p.prefix;
  auto items_of = [&](int b) -> int {
    return sequence_valid(p, b) ? local_windows(p, p.ctx_len[b]) * p.Hkv : 0;
  };
  const int per = (p.B + kThreads - 1) / kThreads;
  const int b_lo = min(p.B, tid * per), b_hi = min(p.B, b_lo + per);
  int run = 0;
  for (int b = b_lo; b < b_hi; ++b) run += items_of(b);
  int incl = run;                                 // inclusive scan over the block
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int base = incl - run;
#pragma unroll
  for (int w = 0; w < kPrepWarps; ++w)
    if (w < warp) base += s_warp[w];
  for (int b = b_lo; b < b_hi; ++b) {
    pre[b] = base;
    base += items_of(b);
  }
  if (tid == kThreads - 1) {                      // its run ends at B
    pre[p.B] = base;
    if (!fused || blockIdx.x == (unsigned)(q_blocks + a_blocks)) *p.item_count = (uint32_t)base;
  }
  if (!fused) return;
  // List block k writes items j = k * kThreads + tid, stepping by all list
  // blocks' threads: a thread finds its item's sequence by binary search in
  // the shared prefix.
  __syncthreads();
  const int total = s_pre[p.B];
  for (int j = ((int)blockIdx.x - q_blocks - a_blocks) * kThreads + tid; j < total;
       j += p.list_blocks * kThreads) {
    int lo = 0, hi = p.B;                         // s_pre[lo] <= j < s_pre[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pre[mid] <= j) lo = mid;
      else hi = mid;
    }
    const int i = j - s_pre[lo], w = i / p.Hkv, kh = i - w * p.Hkv;
    p.items[j] = make_int4(lo | (kh << 16), p.win_begin + w, kh * p.cap_rows + sequence_row0(p, lo),
                           p.ctx_len[lo]);
  }
}

// The work items, one per thread: a warp takes 32 consecutive items.  A
// 32-way search over prefix (every lane probes one entry per round) finds
// the sequence b0 of the warp's first item; the 32 items span at most 32
// sequences, so one more load of prefix[b0 + 1 .. b0 + 32] places each lane.
constexpr int kListThreads = 256;

__global__ void __launch_bounds__(kListThreads) list_kernel(const DecodeParams p) {
  griddep_wait();                                 // prefix and the count
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int total = (int)__ldcg(p.item_count);
  const int warps = gridDim.x * (kListThreads / 32);
  for (int j0 = (blockIdx.x * (kListThreads / 32) + (threadIdx.x >> 5)) * 32; j0 < total;
       j0 += warps * 32) {
    int lo = 0, hi = p.B, base = 0;               // prefix[lo] = base <= j0 < prefix[hi]
    while (hi - lo > 1) {
      const int step = (hi - lo + 31) >> 5;
      const int idx = lo + step * lane;
      const int v = (lane > 0 && idx < hi) ? __ldcg(p.prefix + idx) : base;
      const bool ok = lane == 0 || (idx < hi && v <= j0);
      const int last = 31 - __clz(__ballot_sync(0xffffffffu, ok));
      base = __shfl_sync(0xffffffffu, v, last);
      lo += step * last;
      hi = min(hi, lo + step);
    }
    // boundary i = prefix[lo + 1 + i]: the first item of sequence lo + 1 + i
    const int bi = lo + 1 + lane;
    const int bound = bi <= p.B ? __ldcg(p.prefix + bi) : INT_MAX;
    const int j = j0 + lane;
    int crossed = 0;                              // boundaries at or before item j
#pragma unroll 8
    for (int i = 0; i < 32; ++i) crossed += __shfl_sync(0xffffffffu, bound, i) <= j;
    const int b = lo + crossed;
    const int prev = __shfl_sync(0xffffffffu, bound, max(crossed - 1, 0));   // every lane shuffles
    const int first = crossed == 0 ? base : prev;
    if (j < total) {
      const int i = j - first, w = i / p.Hkv, kh = i - w * p.Hkv;
      p.items[j] = make_int4(b | (kh << 16), p.win_begin + w, kh * p.cap_rows + sequence_row0(p, b),
                             p.ctx_len[b]);
    }
  }
}

// ------------------------------------------------------------------- merge
// Combination of the 512-key windows of every row whose sequence has more
// than one window, in an order fixed by the row's own window count ns:
//   M  = max_s m_s,  w_s = e^(m_s - M)
//   slot k (window s goes to slot s mod 32) sums w_s o_s and w_s l_s over
//   its windows in order (first term a product, then fused adds);
//   O  = the slot sums of o added in slot order;
//   L  = the slot sums of l added by the butterfly of warp_sum (lane k = slot k);
//   out = O / L.
// Which warps do the work does not change a single rounding, so the same
// order serves many short rows (one warp per row, lane k = slot k, ns <= 64)
// and long or few rows (32 warps per row, warp k = slot k).
constexpr int kMergeSlots = 32;

template <int WPR>
__global__ void __launch_bounds__(WPR == 1 ? 256 : 32 * WPR, WPR == 1 ? 3 : 1)
merge_windows_kernel(const DecodeParams p) {
  constexpr int kRowsPerCta = WPR == 1 ? 8 : 1;
  __shared__ float sm_red[WPR == 1 ? 1 : kMergeSlots];
  __shared__ float sm_l[WPR == 1 ? 1 : kMergeSlots];
  __shared__ float4 sm_o[WPR == 1 ? 1 : kMergeSlots][32];
  griddep_wait();                                 // every partial is in place
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = p.R, gq = p.g;
  const int b = blockIdx.y;
  const int row = WPR == 1 ? (int)blockIdx.x * kRowsPerCta + warp : (int)blockIdx.x;   // kh * R + r
  if (row >= p.Hkv * R) return;
  const int kh = row / R, r = row - kh * R;
  const int j = r / gq, h = kh * gq + (r - j * gq);
  float4* dst = reinterpret_cast<float4*>(p.out + ((((int64_t)b * p.M + j) * p.Hq + h) * kD)) + lane;
  if (!sequence_valid(p, b)) {                  // decode: NaN rows already written
    if (p.merge_all && (WPR == 1 || warp == 0)) {
      const float nan = __int_as_float(0x7fc00000);
      *dst = make_float4(nan, nan, nan, nan);
      if (r == 0 && kh == 0 && lane == 0) atomicOr(p.err_word, KATTN_DEVERR_BAD_SEQUENCE);
    }
    return;
  }
  const int ctx = p.ctx_len[b];
  // a sequence of one window was written directly by the decode kernel
  if (!p.merge_all && nsplit_for(ctx + p.M - 1) == 1) return;
  const int ns = nsplit_for(ctx + r / gq);      // the windows this row sees
  const int pst = partial_stride(R);
  const size_t sstride = (size_t)p.Hkv * pst;   // floats from one window to the next
  const size_t shstride = (size_t)p.B * p.part_ws * sstride;   // and from one shard to the next
  const float* base = p.partials + ((size_t)b * p.part_ws * p.Hkv + kh) * pst;
  const float* mcol = base + (size_t)R * kD + r;
  const float* lcol = mcol + R;
  const float* ocol = base + (size_t)r * kD + 4 * lane;
  auto woff = [&](int s) -> size_t {            // window s of the row
    return p.n_shards == 1 ? (size_t)s * sstride
                           : (size_t)(s / p.part_ws) * shstride + (size_t)(s % p.part_ws) * sstride;
  };
  auto ldo = [&](int s) { return __ldcg(reinterpret_cast<const float4*>(ocol + woff(s))); };
  auto fma4 = [](float w, float4 v, float4 acc) {
    return make_float4(__fmaf_rn(w, v.x, acc.x), __fmaf_rn(w, v.y, acc.y), __fmaf_rn(w, v.z, acc.z),
                       __fmaf_rn(w, v.w, acc.w));
  };
  auto mul4 = [](float w, float4 v) {
    return make_float4(__fmul_rn(w, v.x), __fmul_rn(w, v.y), __fmul_rn(w, v.z), __fmul_rn(w, v.w));
  };
  auto add4 = [](float4 a, float4 v) {
    return make_float4(__fadd_rn(a.x, v.x), __fadd_rn(a.y, v.y), __fadd_rn(a.z, v.z), __fadd_rn(a.w, v.w));
  };

  float4 O;
  float L;
  if constexpr (WPR == 1) {
    // lane k: windows k and k + 32 (ns <= 64).  The first batch of o loads
    // goes out with the m and l loads, before the maximum is known.
    const int nk = min(ns, kMergeSlots);
    constexpr int kBatch = 4;                     // slots whose loads are in flight together
    float4 a[kBatch], c[kBatch];
    auto load_batch = [&](int k0) {
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (k0 + i < nk) a[i] = ldo(k0 + i);
        if (k0 + i + kMergeSlots < ns) c[i] = ldo(k0 + i + kMergeSlots);
      }
    };
    load_batch(0);
    const bool h0 = lane < ns, h1 = lane + kMergeSlots < ns;
    const float m0 = h0 ? __ldcg(mcol + woff(lane)) : -INFINITY;
    const float m1 = h1 ? __ldcg(mcol + woff(lane + kMergeSlots)) : -INFINITY;
    const float l0 = h0 ? __ldcg(lcol + woff(lane)) : 0.0f;
    const float l1 = h1 ? __ldcg(lcol + woff(lane + kMergeSlots)) : 0.0f;
    const float M = warp_max(fmaxf(m0, m1));
    const float w0 = h0 ? exp_diff(m0, M) : 0.0f, w1 = h1 ? exp_diff(m1, M) : 0.0f;
    L = warp_sum(h1 ? __fmaf_rn(w1, l1, __fmul_rn(w0, l0)) : __fmul_rn(w0, l0));
    O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < nk; k0 += kBatch) {
      if (k0 > 0) load_batch(k0);
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int k = k0 + i;
        if (k < nk) {
          float4 in = mul4(__shfl_sync(0xffffffffu, w0, k), a[i]);
          if (k + kMergeSlots < ns) in = fma4(__shfl_sync(0xffffffffu, w1, k), c[i], in);
          O = k == 0 ? in : add4(O, in);
        }
      }
    }
  } else {
    // warp k = slot k: windows k, k + 32, ...  The slot's first kPre windows
    // (m, l and o) are loaded at once, before the maximum is known.
    constexpr int kPre = 4;
    float4 vp[kPre];
    float mp[kPre], lp[kPre];
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
      const int s = warp + kMergeSlots * i;
      if (s < ns) {
        mp[i] = __ldcg(mcol + woff(s));
        lp[i] = __ldcg(lcol + woff(s));
        vp[i] = ldo(s);
      }
    }
    float mloc = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPre; ++i)
      if (warp + kMergeSlots * i < ns) mloc = fmaxf(mloc, mp[i]);
    for (int s = warp + kMergeSlots * kPre; s < ns; s += kMergeSlots) mloc = fmaxf(mloc, __ldcg(mcol + woff(s)));
    if (lane == 0) sm_red[warp] = mloc;
    __syncthreads();
    const float M = warp_max(sm_red[lane]);     // the 32 slot maxima (-inf for empty slots)
    float4 in = make_float4(0.f, 0.f, 0.f, 0.f);
    float il = 0.0f;
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
      if (warp + kMergeSlots * i < ns) {
        const float w = exp_diff(mp[i], M);
        if (i == 0) {
          in = mul4(w, vp[i]);
          il = __fmul_rn(w, lp[i]);
        } else {
          in = fma4(w, vp[i], in);
          il = __fmaf_rn(w, lp[i], il);
        }
      }
    }
#pragma unroll 4
    for (int s = warp + kMergeSlots * kPre; s < ns; s += kMergeSlots) {
      const float w = exp_diff(__ldcg(mcol + woff(s)), M);
      const float ls = __ldcg(lcol + woff(s));
      const float4 v = ldo(s);
      in = fma4(w, v, in);
      il = __fmaf_rn(w, ls, il);
    }
    sm_o[warp][lane] = in;
    if (lane == 0) sm_l[warp] = il;
    __syncthreads();
    if (warp != 0) return;
    L = warp_sum(sm_l[lane]);                   // empty slots hold 0
    O = sm_o[0][lane];
    for (int k = 1; k < kMergeSlots && k < ns; ++k) O = add4(O, sm_o[k][lane]);
  }
  *dst = make_float4(__fdiv_rn(O.x, L), __fdiv_rn(O.y, L), __fdiv_rn(O.z, L), __fdiv_rn(O.w, L));
}

// ------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// 2-D view [rows][128] of an int8 cache; kBlockBk-row boxes, 128-byte swizzle.
bool encode_cache_map(CUtensorMap* map, const int8_t* base, int64_t rows) {
  const auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD};
  const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)kBlockBk};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The split-KV pass over a contiguous cache, by the rows R of a CTA.  (The
// cache layout is a template parameter, so this kernel carries none of the
// paged lookups.)
cudaError_t launch_split_contiguous(const DecodeParams& p, const TmaMaps& maps,
                                    cudaStream_t stream) {
  if (p.R <= 8) return launch_modes<1, 1, false>(p, maps, stream);
  if (const int nrg = row_groups_for(p); nrg > 1) {      // rows in groups of 8, a CTA each
    DecodeParams pr = p;
    pr.row_groups = nrg;
    return launch_modes<1, 1, false>(pr, maps, stream);
  }
  if (p.R <= 16) return launch_modes<2, 1, false>(p, maps, stream);
  if (p.R <= 32) return launch_split_tc(p, maps, stream);   // P.V on tcgen05
  if (p.R <= 48) return launch_modes<3, 2, false>(p, maps, stream);
  return launch_modes<4, 2, false>(p, maps, stream);
}

}  // namespace

int decode_launch_count(const DecodeParams& p) {
  const bool merge = p.nsplit_max > 1 && !p.shard_mode;
  return 2 + (p.B > kFusedListMaxB ? 1 : 0) + (merge ? 1 : 0);
}

cudaError_t launch_decode_fast(const DecodeParams& p, cudaStream_t stream) {
  TmaMaps maps;
  const int64_t rows = (int64_t)p.Hkv * p.cap_rows;
  if (!encode_cache_map(&maps.k, p.k, rows) || !encode_cache_map(&maps.v, p.v, rows))
    return cudaErrorInvalidValue;
  // 1. packed queries and the work list (ordinary launch: it reads the
  //    caller's q, row_start and ctx_len)
  const int64_t qrows = (int64_t)p.B * p.Hkv * p.rpad;
  const int q_blocks = (int)((qrows + kPrepWarps - 1) / kPrepWarps);
  //    Up to kFusedListMaxB sequences its list blocks also write the work
  //    items; beyond, one block writes the prefix and list_kernel the items.
  const int64_t max_items = (int64_t)p.B * p.nsplit_max * p.Hkv;
  DecodeParams pp = p;
  pp.list_blocks =
      p.B <= kFusedListMaxB
          ? (int)std::min<int64_t>((max_items + kListPerBlock - 1) / kListPerBlock, 256)
          : 0;
  const int a_blocks = (int)(((int64_t)p.n_new * p.Hkv * 2 + kPrepWarps - 1) / kPrepWarps);
  prepare_kernel<<<q_blocks + a_blocks + (pp.list_blocks > 0 ? pp.list_blocks : 1), kPrepWarps * 32,
                   0, stream>>>(pp, q_blocks, a_blocks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (pp.list_blocks == 0) {
    const int list_blocks =
        (int)std::min<int64_t>((max_items + kListThreads - 1) / kListThreads, 1024);
    if ((e = launch_pdl(list_kernel, dim3((unsigned)list_blocks), dim3(kListThreads), 0, stream,
                        p)) != cudaSuccess)
      return e;
  }
  // 2. the split-KV pass
  e = p.block_table != nullptr ? launch_split_paged(p, maps, stream)
                               : launch_split_contiguous(p, maps, stream);
  if (e != cudaSuccess || p.nsplit_max <= 1 || p.shard_mode) return e;
  // 3. the window merge
  return launch_merge(p, stream);
}

// The window merge (the same arithmetic in both shapes), over the windows of
// at most n_shards * part_ws per row.  Estimated time = waves x dependent
// loads per row: one warp per row (24 rows per SM at once; a load round per 4
// windows) or 32 warps per row (one row per SM; a round per 128 windows), for
// rows of up to 64 windows.
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream) {
  const int nwin = p.n_shards * p.part_ws;
  const int rows_b = p.Hkv * p.R;                 // rows of one sequence
  const int64_t all_rows = (int64_t)rows_b * p.B;
  int sms = 0;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
      sms = 1;
  }
  const int64_t est_warp = (all_rows + 24LL * sms - 1) / (24LL * sms) * ((nwin + 3) / 4 + 2);
  const int64_t est_cta = (all_rows + sms - 1) / sms * ((nwin + 127) / 128 + 3);
  if (nwin <= 2 * kMergeSlots && est_warp <= est_cta)
    return launch_pdl(merge_windows_kernel<1>, dim3((unsigned)((rows_b + 7) / 8), (unsigned)p.B),
                      dim3(256), 0, stream, p);
  return launch_pdl(merge_windows_kernel<kMergeSlots>, dim3((unsigned)rows_b, (unsigned)p.B),
                    dim3(32 * kMergeSlots), 0, stream, p);
}

}  // namespace kattn
