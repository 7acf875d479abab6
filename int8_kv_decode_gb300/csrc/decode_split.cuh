// Fast decode over the int8 KV cache: split-KV on tensor cores, fixed-order merge.
//
// Four launches on the caller's stream, chained by programmatic dependent
// launch (a kernel starts while the previous one drains and waits on
// griddepcontrol before it reads that one's results):
//   1. prepare_kernel quantizes every query row once (int8 per row) into the
//      workspace and counts the work items of the valid sequences, one per
//      window of kSplitC = 512 keys and kv head (a prefix over sequences);
//      the rows of an invalid sequence become NaN and raise an error bit;
//   1b. list_kernel writes the work items, one thread each;
//   2. decode_fast_kernel: persistent CTAs (SM count x occupancy) take the
//      items x kv heads in a fixed stride.  In a CTA, warp kw reduces span kw
//      (kSpanC = 128 keys) of the window for all R = g*M query rows that read
//      the kv head -- the GQA group times the M draft columns -- so every K/V
//      byte is read from HBM once.  The four spans are merged in a fixed
//      pairwise order; a sequence of one window is finished here, otherwise
//      the window's (m, l, o) goes to the workspace.  With more than 8 rows
//      and few items (a small batch), each item is instead split into row
//      groups of 8 rows, one CTA each of the one-tile variant, which read the
//      same K/V blocks (all but the first from L2) and write their rows of
//      the same window partial;
//   3. merge_windows_kernel combines the windows of each row in order.
//
// Per warp and block of kBlockBk = 32 keys ("在 agent 时代如何快速验证 kernel
// 对精度的影响", section "注意力权重": blockwise online softmax, P rounded only
// where it multiplies V, row sum from the unrounded P):
//   * TMA (cp.async.bulk.tensor, 128-byte swizzle) streams the K and V rows of
//     the block into the warp's own ring of shared-memory stages; lane 0 is
//     the producer, one mbarrier per stage, every wait bounded.  The producer
//     runs ahead into the CTA's next work item, so HBM reads go on through
//     the merge of one window and the start of the next;
//   * QK on tensor cores: the int8 MMA (m16n8k32) when a warp holds one tile
//     of 8 query rows, else the f16 MMA (m16n8k16) over exactly converted
//     values; every partial sum is an integer below 2^24, so the f32 scores
//     equal the int32 dot products exactly.  Keys sit on the MMA's M side,
//     query rows on N (8 per n-tile);
//   * scores, the block max (warp shuffles), the online update of m and l, P
//     rounding and a = round_p(p) * v_scale in f32 registers;
//   * PV on tensor cores: mma.sync m16n8k16 f16 with V (int8, exact in f16)
//     on the A side and a = round_p(p) * v_scale split into f16 hi + lo on
//     the B side, accumulated in f32.  a is first scaled by a power of two
//     fixed per span and row (from the largest v_scale the row sees there),
//     so the split keeps float32-level accuracy; the power is undone,
//     exactly, in the merge.
//
// Batch invariance ("Kestrel_VLLM - 18" §二): the bytes of a query row depend
// only on its own keys: spans, blocks and windows sit at fixed key positions,
// a block with no visible key leaves a row untouched, each MMA output element
// depends only on its own row's operands, and every merge runs in a fixed
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <atomic>

#include "device_common.cuh"

namespace kattn {

struct TmaMaps {
  CUtensorMap k, v;
};

namespace {


constexpr int kRing = 2;                       // TMA stages per warp
constexpr int kBlockBytes = kBlockBk * kD;     // one K (or V) block: 4 KB
constexpr uint32_t kSpinLimit = 1u << 22;      // bounded mbarrier waits
static_assert(kBlockBk == 32, "the MMA layout below takes a block as two halves of 16 keys");
static_assert(kSpanC == 4 * kBlockBk, "span scales are held as 4 registers per lane");



template <int NR, int NG>
struct __align__(1024) SmemT {
  static constexpr int kRows = NG * NR * 8;                  // query rows of the CTA (rpad)
  static constexpr int kF = NR == 1 ? 1 : 0;                 // int8 QK: no f16 fragments

  uint8_t ring[kSpansPerCta][kRing][2][kBlockBytes];         // per span: [stage][K|V]
  float slot[NG][2][NR * 8 * kD];                            // span merge, fragment order
  uint8_t qbuf[kRows * (kD + 4)];                            // item's int8 rows, then scales
  uint2 qfrag[kF ? 1 : NG][kF ? 1 : NR][kF ? 1 : 8][kF ? 1 : 32];   // f16 query fragments
  uint64_t full[kSpansPerCta][kRing];                        // the stage's copy landed
  uint64_t empty[kSpansPerCta][kRing];                       // NG > 1: every group read it
  uint64_t qbar;
  // Per-span running max and row sum, double-buffered by item parity: warp 0
  // reads an item's values after the other warps have moved on to the next
  // item; a buffer comes back two items later, after a CTA barrier that
  // warp 0 reaches only once it is done reading.
  float wm[2][NG][kSpansPerCta][NR * 8];
  float wl[2][NG][kSpansPerCta][NR * 8];
  int fail[NG * kSpansPerCta];                               // per warp: a copy never arrived
  int brow[kSpansPerCta][2][kSpanC / kBlockBk];              // producer: block rows, by item parity
};

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t it = 0; it < kSpinLimit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// L2 policy for the K/V stream: read once, so its lines go first and the
// window partials written meanwhile stay in L2 for the merge.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
// With row groups the K/V of a window is read by several CTAs: keep it in L2
// at normal priority until they have all read it.
__device__ __forceinline__ uint64_t l2_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}

// kBlockBk rows x 128 bytes starting at row `row` of a 2-D cache view.
__device__ __forceinline__ void tma_load_block(void* dst, const CUtensorMap* map, int row,
                                               uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;\n" ::"r"(smem_u32(dst)),
      "l"(map), "r"(0), "r"(row), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// Two int8 bytes (chosen by `sel` from a word already XORed with 0x80808080)
// -> f16x2 of their exact values: byte ^ 0x80 becomes the low mantissa of
// 1024.0, then 1024 + 128 is subtracted.
__device__ __forceinline__ uint32_t i8pair_to_h2(uint32_t xored, uint32_t sel) {
  const uint32_t h = __byte_perm(xored, 0x64646464u, sel);
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), __half2(1152.0f, 1152.0f));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint2 b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y));
}

__device__ __forceinline__ void mma_i8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};\n"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Paired float32 arithmetic (one instruction for two lanes of a pair).
__device__ __forceinline__ unsigned long long f2_pack(float2 a) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(a.x), "f"(a.y));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r) {
  float2 a;
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(a.x), "=f"(a.y) : "l"(r));
  return a;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(r);
}

__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)), "l"(f2_pack(c)));
  return f2_unpack(r);
}

// x = hi + lo with hi = RN_f16(x) and lo = RN_f16(x - hi) (x - hi is exact in
// float32): 22 significant bits of each of two values, packed as f16x2.
__device__ __forceinline__ void split_f16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 r = f2_sub(make_float2(x0, x1), __half22float2(h));
  const __half2 l = __floats2half2_rn(r.x, r.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 2^x by the SFU in one instruction (ex2.approx.ftz: a result below 2^-126 is
// flushed to +0, 2^-inf = +0).  Every fast-mode kernel takes its weights from
// here, so the flush is the same for a row whatever kernel reduces it; a
// weight that small is below 1e-38 of the row's largest and moves no output.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// e^(x - m) for x <= m, m finite: the difference first (exact near the max,
// where the weights matter), then base 2.
__device__ __forceinline__ float exp_diff(float x, float m) {
  return fast_exp2(__fmul_rn(__fsub_rn(x, m), kLog2e));
}

// Weight of a partial with running max x in a merge whose max is m.
__device__ __forceinline__ float merge_weight(float x, float m) {
  return m == -INFINITY ? 0.0f : exp_diff(x, m);
}

template <int PM>
__device__ __forceinline__ float round_p_t(float p) {
  if constexpr (PM == KATTN_P_BF16) {
    return bf16_round(p);
  } else if constexpr (PM == KATTN_P_E4M3 || PM == KATTN_P_E4M3_DIRECT) {
    return e4m3_round(p);
  } else if constexpr (PM == KATTN_P_E4M3_X256) {
    return __fmul_rn(e4m3_round(__fmul_rn(p, 256.0f)), 1.0f / 256.0f);   // both exact
  } else if constexpr (PM == KATTN_P_E4M3_X448) {
    return __fmul_rn(e4m3_round(__fmul_rn(p, 448.0f)), 1.0f / 448.0f);
  } else {
    return p;
  }
}

// Online-softmax update of one 8-row n-tile over a 32-key block, for the two
// rows 2c, 2c + 1 a thread holds (e = 0, 1).  s0 / s1: the scores of the block's
// two 16-key halves in the MMA score layout ([0] key g row 2c, [1] key g row
// 2c+1, [2] key g+8 row 2c, [3] key g+8 row 2c+1); on return they hold the
// P.V operand values a = round_p(p) * v_scale * 2^E.  vs4[q]: v_scale of key
// g + 8q.  The two rows go through paired float32 operations, each element
// rounded as the scalar operation would be:
//   m' = max(m, block max);  alpha = e^(m - m');  p = e^(s - m')
//   l  = l * alpha + ((p_g + p_g8) + (p_16+g + p_24+g))   (one fused multiply-add)
// A row with no visible key yet (m' = -inf) is left untouched (alpha 1, p 0).
template <int PM>
__device__ __forceinline__ void softmax_tile(float (&s0)[4], float (&s1)[4], float (&m_run)[2],
                                             float (&l_run)[2], const float (&up)[2],
                                             const float (&vs4)[4], float (&alpha)[2],
                                             bool& rescale) {
  float mnew[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float bm = fmaxf(fmaxf(s0[e], s0[2 + e]), fmaxf(s1[e], s1[2 + e]));
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
    mnew[e] = fmaxf(m_run[e], bm);
  }
  const float2 mn = make_float2(mnew[0], mnew[1]);
  const float2 l2e = make_float2(kLog2e, kLog2e);
  const bool live0 = mnew[0] != -INFINITY, live1 = mnew[1] != -INFINITY;
  const float2 da = f2_mul(f2_sub(make_float2(m_run[0], m_run[1]), mn), l2e);
  alpha[0] = live0 ? fast_exp2(da.x) : 1.0f;
  alpha[1] = live1 ? fast_exp2(da.y) : 1.0f;
  rescale |= (alpha[0] != 1.0f) | (alpha[1] != 1.0f);
  m_run[0] = mnew[0];
  m_run[1] = mnew[1];
  float2 pk[2][2];                                // [half][key g | g + 8], rows (2c, 2c+1)
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float* sv = hf ? s1 : s0;
      const float2 d = f2_mul(f2_sub(make_float2(sv[2 * k], sv[2 * k + 1]), mn), l2e);
      pk[hf][k] = make_float2(live0 ? fast_exp2(d.x) : 0.0f, live1 ? fast_exp2(d.y) : 0.0f);
    }
  const float2 lsum = f2_add(f2_add(pk[0][0], pk[0][1]), f2_add(pk[1][0], pk[1][1]));
  const float2 lnew = f2_fma(make_float2(l_run[0], l_run[1]), make_float2(alpha[0], alpha[1]), lsum);
  l_run[0] = lnew.x;
  l_run[1] = lnew.y;
  const float2 up2 = make_float2(up[0], up[1]);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float v = vs4[2 * hf + k];
      const float2 a = f2_mul(f2_mul(make_float2(round_p_t<PM>(pk[hf][k].x), round_p_t<PM>(pk[hf][k].y)),
                                     make_float2(v, v)), up2);
      float* sv = hf ? s1 : s0;
      sv[2 * k] = a.x;
      sv[2 * k + 1] = a.y;
    }
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a block written by TMA
// with the 128-byte swizzle (chunk index XOR row mod 8; buffers 1 KB aligned).
__device__ __forceinline__ int swz(int row, int chunk) {
  return row * kD + ((chunk ^ (row & 7)) << 4);
}

// Programmatic dependent launch: wait until the preceding grid has finished
// and its writes are visible / let the next grid begin its launch.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Plain bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Named barriers of a warp group (ids 1.. ; 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int threads) {
  asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------------ work items
// Work item t of the decode grid is one (sequence b, window w, kv head kh):
// the items of sequence b are t in [prefix[b], prefix[b + 1]), windows in
// order, kv heads fastest.  list_kernel stores each as {b | kh << 16, w,
// kh * cap_rows + row_start[b], ctx_len[b]}: row is the cache row of key 0 of
// the sequence in the 2-D view [Hkv * cap_rows][128] (and the index of its
// scales); in the paged layout it is the plane's row 0 and key_row adds the
// key's row from the block table.  b < 0 marks "no item".
struct Item {
  int b, kh, w, row, ctx;
  int rg;               // row group: rows [8 rg, 8 rg + 8) of the item (row-group split)
};

__device__ __forceinline__ Item load_item(const DecodeParams& p, int t, int total) {
  Item it{-1, 0, 0, 0, 0, 0};
  if (t < total) {
    const int4 v = __ldcg(p.items + t);
    it = Item{v.x & 0xffff, (int)((unsigned)v.x >> 16), v.y, v.z, v.w, 0};
  }
  return it;
}

// Unit t of the decode grid when every work item is split into nrg row
// groups (nrg > 1: the one-tile kernel, 8 query rows per CTA): item t / nrg,
// row group t % nrg.  The row groups of an item are consecutive units, so
// CTAs that run side by side read the same K/V blocks, the later ones from L2.
__device__ __forceinline__ Item load_unit(const DecodeParams& p, int t, int total, int nrg) {
  if (nrg == 1) return load_item(p, t, total);
  const int i = t / nrg;
  Item it = load_item(p, i, total);
  it.rg = t - i * nrg;
  return it;
}

// A unit's work item as loaded, not yet taken apart: a kernel fetches the
// unit two items ahead and decodes it one item later, so that no warp waits
// on the load at an item boundary.
struct RawUnit {
  int4 v;
  int rg;
  bool valid;
};

__device__ __forceinline__ RawUnit fetch_unit(const DecodeParams& p, int t, int total, int nrg) {
  RawUnit r{make_int4(0, 0, 0, 0), 0, false};
  const int i = nrg == 1 ? t : t / nrg;
  if (i < total) {
    r.v = __ldcg(p.items + i);
    r.rg = t - i * nrg;
    r.valid = true;
  }
  return r;
}

__device__ __forceinline__ Item decode_unit(const RawUnit& r) {
  Item it{-1, 0, 0, 0, 0, 0};
  if (r.valid) it = Item{r.v.x & 0xffff, (int)((unsigned)r.v.x >> 16), r.v.y, r.v.z, r.v.w, r.rg};
  return it;
}

// Keys [s0, s1) of span kw of the item's window, its nb blocks, and the cache
// row of key s0 in the 2-D view [Hkv * cap_rows][128] (contiguous layout).
struct Span {
  int s0, s1, nb, row;
};

__device__ __forceinline__ Span span_of(const Item& it, int kw, int M) {
  Span s;
  const int Lmax = it.ctx + M - 1;
  const int k0 = it.w * kSplitC, k1 = min(k0 + kSplitC, Lmax);
  s.s0 = k0 + kw * kSpanC;
  s.s1 = min(s.s0 + kSpanC, k1);
  s.nb = s.s1 > s.s0 ? (s.s1 - s.s0 + kBlockBk - 1) / kBlockBk : 0;
  s.row = it.row + s.s0;
  return s;
}

// Scales of a span: lane l holds keys l, l+32, l+64, l+96 (0 past the span).
// PG: the paged layout, rows from the block table.
template <bool PG>
__device__ __forceinline__ void load_span_scales(const DecodeParams& p, const Item& it,
                                                 const Span& sp, int lane, float (&ks)[4],
                                                 float (&vs)[4]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int key = sp.s0 + lane + 32 * e;
    const bool in = it.b >= 0 && key < sp.s1;
    if constexpr (PG) {
      const int row = in ? it.row + paged_row(p, it.b, key) : 0;
      ks[e] = in ? __ldg(p.k_scale + row) : 0.0f;
      vs[e] = in ? __ldg(p.v_scale + row) : 0.0f;
    } else {
      ks[e] = in ? __ldg(p.k_scale + it.row + key) : 0.0f;
      vs[e] = in ? __ldg(p.v_scale + it.row + key) : 0.0f;
    }
  }
}

// ------------------------------------------------------------------ decode
// NR: 8-row n-tiles per warp group; NG: warp groups of kSpansPerCta warps;
// PM: the P rounding (a kattn_p_mode).  Warp kw of a group reduces span kw
// of the item's window for the group's rows, one block of kBlockBk = 32 keys
// at a time (two MMA halves of 16 keys).
//
// QK runs on the int8 MMA (raw K words straight from shared memory, no
// conversion) when a warp holds a single n-tile of query rows; with more
// n-tiles the slow int8 tensor rate would bind, so the f16 MMA on converted
// values is used.  Both give the same exact integer scores.
template <int NR, int NG, int PM, bool PG>
__global__ void __launch_bounds__(kSpansPerCta * 32 * NG, NR == 1 ? 3 : (NG == 1 ? 2 : 1))
decode_fast_kernel(const DecodeParams p, const __grid_constant__ TmaMaps maps) {
  using Smem = SmemT<NR, NG>;
  constexpr bool kQK8 = NR == 1;                  // QK on the int8 MMA (one n-tile)
  constexpr int RG = NR * 8;                      // rows per warp group
  constexpr int RP = Smem::kRows;                 // rows per CTA (the packed query rows)
  constexpr int kWarps = kSpansPerCta * NG;
  constexpr uint32_t kQBytes = RP * (kD + 4);
  extern __shared__ unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kw = warp % kSpansPerCta, grp = warp / kSpansPerCta;
  const int g = lane >> 2, c = lane & 3;
  const int gq = p.g, M = p.M, R = p.R;
  // Row groups (one-tile kernel only): an item's R rows are split over
  // nrg = ceil(R / 8) units of 8 rows, one CTA each.  The CTA then holds
  // rows [8 rg, 8 rg + 8) of the item, at rows 0..7 of its query buffer.
  constexpr bool kCanSplit = NR == 1 && NG == 1;
  const int nrg = kCanSplit ? p.row_groups : 1;
  const int qrow0 = grp * RG;                     // the group's first row in qbuf
  // Span kw's ring is filled by warp kw of group 0 and read by warp kw of
  // every group (the groups hold different query rows).
  uint64_t* full = sm.full[kw];
  uint64_t* empty = sm.empty[kw];
  const bool producer = grp == 0;
  // Per thread and item: the first row of the group (row0), the draft column
  // j of rows row0 + 8nr + 2c + e, and where those rows sit in out (head
  // kh * g + r % g; add kh * g * d and the sequence's offset).
  int row0 = qrow0;
  int jrow[NR][2], orow[NR][2];
  auto place_rows = [&](int rg) {
    row0 = qrow0 + 8 * rg;
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = row0 + nr * 8 + 2 * c + e;
        jrow[nr][e] = min(r / gq, M - 1);
        orow[nr][e] = ((r / gq) * p.Hq + r % gq) * kD + 16 * g;
      }
  };
  place_rows(0);

  if (lane == 0 && producer) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NG);
    }
  }
  if (lane == 0) {
    if (warp == 0) mbar_init(&sm.qbar, 1);
    sm.fail[warp] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  griddep_wait();                                 // the work list and the packed queries
  griddep_launch_dependents();

  const int total = (int)__ldcg(p.item_count);
  const int units = total * nrg;                  // below 2^31: checked on the host
  const int G = gridDim.x;
  int t = blockIdx.x;
  if (t >= units) return;
  Item it0 = load_unit(p, t, total, nrg), it1 = load_unit(p, t + G, total, nrg);
  RawUnit raw2 = fetch_unit(p, t + 2 * G, total, nrg);   // decoded one item later
  if (nrg > 1) place_rows(it0.rg);

  bool q_pending = false;                         // thread 0: a query copy in flight
  auto fetch_queries = [&](const Item& it) {      // thread 0
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    mbar_expect_tx(&sm.qbar, kQBytes);
    const uint8_t* pack = p.qpack + ((size_t)it.b * p.Hkv + it.kh) * qpack_bytes(p.rpad);
    if (kCanSplit && nrg > 1) {
      // the group's 8 int8 rows, then its 8 scales (the pack holds rpad rows)
      bulk_load(sm.qbuf, pack + (size_t)it.rg * 8 * kD, 8 * kD, &sm.qbar);
      bulk_load(sm.qbuf + 8 * kD, pack + (size_t)p.rpad * kD + it.rg * 8 * 4, 8 * 4, &sm.qbar);
    } else {
      bulk_load(sm.qbuf, pack, kQBytes, &sm.qbar);
    }
    q_pending = true;
  };
  if (tid == 0) fetch_queries(it0);

  // ---- producer: lane 0 issues, every lane keeps the same counters.  The
  // cursor runs over this item's blocks, then the next item's.
  Span psp = span_of(it0, kw, M);
  int pitem = 0, pblk = 0, ist = 0, inflight = 0;
  int par = 0;                                    // item parity: (m, l) and block-row buffers
  // Paged layout: the producer warp looks up the cache rows (2-D view) of its
  // span's blocks one item ahead, into the slot of the item's parity (lane e:
  // block e; a block never crosses a page).  At an item boundary it only
  // loads the next item's table entries (rows_ahead); they become rows when
  // the producer reaches that item (rows_finish), so no warp waits there.
  int pg_entry = 0, pg_key = 0, pg_n = 0, pg_slot = 0, pg_row = 0;
  bool pg_pending = false;
  auto rows_ahead = [&](const Item& it, int slot) {
    if constexpr (PG) {
      if (producer && it.b >= 0) {
        const Span s = span_of(it, kw, M);
        pg_key = s.s0 + lane * kBlockBk;
        if (lane < s.nb) pg_entry = page_entry(p, it.b, pg_key);
        pg_n = s.nb;
        pg_slot = slot;
        pg_row = it.row;
        pg_pending = true;
      }
    }
  };
  auto rows_finish = [&]() {
    if constexpr (PG) {
      if (pg_pending) {
        if (lane < pg_n) sm.brow[kw][pg_slot][lane] = pg_row + page_row_of(p, pg_entry, pg_key);
        __syncwarp();
        pg_pending = false;
      }
    }
  };
  rows_ahead(it0, 0);
  rows_finish();
  rows_ahead(it1, 1);
  rows_finish();
  uint32_t used = 0, eph = 0;                     // NG > 1: stages filled before; empty parities
  const uint64_t kv_policy = nrg > 1 ? l2_evict_normal() : l2_evict_first();
  // Returns false if a stage was never released (a bounded wait ran out).
  auto produce = [&]() -> bool {
    if (!producer) return true;
    while (inflight < kRing) {
      if (pblk < psp.nb) {
        if constexpr (NG > 1) {
          if ((used >> ist) & 1u) {               // wait until every group has read it
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[ist], (eph >> ist) & 1u)))
              return false;
            eph ^= 1u << ist;
          }
          used |= 1u << ist;
        }
        if (lane == 0) {
          asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
          mbar_expect_tx(&full[ist], 2 * kBlockBytes);
          const int row = PG ? sm.brow[kw][par ^ pitem][pblk] : psp.row + pblk * kBlockBk;
          tma_load_block(sm.ring[kw][ist][0], &maps.k, row, &full[ist], kv_policy);
          tma_load_block(sm.ring[kw][ist][1], &maps.v, row, &full[ist], kv_policy);
        }
        ++pblk;
        ++inflight;
        ist = ist + 1 == kRing ? 0 : ist + 1;
      } else if (pitem == 0 && it1.b >= 0) {
        rows_finish();                            // the next item's rows, loaded ahead
        pitem = 1;
        pblk = 0;
        psp = span_of(it1, kw, M);
      } else {
        break;
      }
    }
    return true;
  };
  bool prod_ok = produce();

  // ---- consumer state
  Span sp = span_of(it0, kw, M);
  float ksp[4], vsp[4], ksn[4], vsn[4];           // this item's / the next item's span scales
  load_span_scales<PG>(p, it0, sp, lane, ksp, vsp);
  load_span_scales<PG>(p, it1, span_of(it1, kw, M), lane, ksn, vsn);
  int cst = 0;                                    // ring stage of the next block to consume
  uint32_t cph = 0, qph = 0;                      // its mbarrier parity; the query barrier's

  for (;;) {
    // ---- the item's queries (packed by prepare_kernel)
    const bool q_ok = __all_sync(0xffffffffu, mbar_wait_bounded(&sm.qbar, qph));
    if (tid == 0 && q_ok) q_pending = false;
    // Thread (g, c) takes bytes [32c, 32c + 32) of row 8nr + g.  For the int8
    // MMA, step s covers d = 32c + 8s + 0..7 (words 2s, 2s + 1); for the f16
    // MMA, step s maps k = 2c,2c+1 -> d = 32c+4s+{0,1} and 2c+8,2c+9 ->
    // 32c+4s+{2,3}.  Either is a fixed permutation of d shared with the K
    // fragments, and the sums are integers, so both are exact.
    uint32_t qw8[8];
    if constexpr (kQK8) {
      const uint4* src = reinterpret_cast<const uint4*>(&sm.qbuf[(qrow0 + g) * kD + 32 * c]);
      const uint4 lo = src[0], hi = src[1];
      qw8[0] = lo.x; qw8[1] = lo.y; qw8[2] = lo.z; qw8[3] = lo.w;
      qw8[4] = hi.x; qw8[5] = hi.y; qw8[6] = hi.z; qw8[7] = hi.w;
    } else {
      if (kw < NR) {                              // warp kw builds n-tile kw of its group
        const uint4* src =
            reinterpret_cast<const uint4*>(&sm.qbuf[(qrow0 + kw * 8 + g) * kD + 32 * c]);
        const uint4 lo = src[0], hi = src[1];
        const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t w = wv[s] ^ 0x80808080u;
          sm.qfrag[grp][kw][s][lane] = make_uint2(i8pair_to_h2(w, 0x4140u), i8pair_to_h2(w, 0x4342u));
        }
      }
      __syncthreads();
    }
    float qs_row[NR][2];                          // scales of rows 8nr + 2c + e
    {
      const float* qsb = reinterpret_cast<const float*>(&sm.qbuf[RP * kD]);
#pragma unroll
      for (int nr = 0; nr < NR; ++nr)
#pragma unroll
        for (int e = 0; e < 2; ++e) qs_row[nr][e] = qsb[qrow0 + nr * 8 + 2 * c + e];
    }

    // Power of two 2^E per query row: over the keys of the span that the row
    // sees, max_k v_scale_k * 2^E lies in [2^14, 2^15), so a = round_p(p) *
    // v_scale * 2^E stays in the normal f16 range down to weights far below
    // the ones that matter; the row's o is held in units of 2^E.  E depends
    // only on the row's own keys (batch invariance).
    const int ctx = it0.ctx;
    float up_row[NR][2], down_row[NR][2];
    {
      const int kc = min(sp.s1, ctx);             // keys every row sees: [s0, kc)
      float vm = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (sp.s0 + lane + 32 * e < kc) vm = fmaxf(vm, vsp[e]);
      vm = warp_max(vm);
      float vt[kMaxM - 1];                        // scales of keys ctx + t (the draft tail)
#pragma unroll
      for (int t = 0; t < kMaxM - 1; ++t) vt[t] = 0.0f;
      if (sp.s1 > ctx) {                          // the span holds draft keys (uniform)
#pragma unroll
        for (int t = 0; t < kMaxM - 1; ++t) {
          const int rel = ctx + t - sp.s0;
          if (t < M - 1 && rel >= 0 && ctx + t < sp.s1) {
            const int e = rel >> 5;
            const float mine = e == 0 ? vsp[0] : e == 1 ? vsp[1] : e == 2 ? vsp[2] : vsp[3];
            vt[t] = __shfl_sync(0xffffffffu, mine, rel & 31);
          }
        }
      }
#pragma unroll
      for (int nr = 0; nr < NR; ++nr)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float vmax = vm;
#pragma unroll
          for (int t = 0; t < kMaxM - 1; ++t)
            if (t < jrow[nr][e]) vmax = fmaxf(vmax, vt[t]);
          const int bexp = min(max(268 - (int)((__float_as_uint(vmax) >> 23) & 0xffu), 1), 253);
          up_row[nr][e] = __uint_as_float((uint32_t)bexp << 23);
          down_row[nr][e] = __uint_as_float((uint32_t)(254 - bexp) << 23);
        }
    }

    // ---- per-thread row state: rows 8nr + 2c + e (e = 0, 1) of the group
    float m_run[NR][2], l_run[NR][2];
    int Lrow[NR][2];
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        m_run[nr][e] = -INFINITY;
        l_run[nr][e] = 0.0f;
        Lrow[nr][e] = ctx + jrow[nr][e];
      }
    float o[8][NR][4];
#pragma unroll
    for (int md = 0; md < 8; ++md)
#pragma unroll
      for (int nr = 0; nr < NR; ++nr)
#pragma unroll
        for (int u = 0; u < 4; ++u) o[md][nr][u] = 0.0f;

    bool failed = !q_ok || !prod_ok;
    prod_ok = true;
    const int nb = q_ok ? sp.nb : 0;
    for (int i = 0; i < nb; ++i) {
      const int t0 = sp.s0 + i * kBlockBk;
      // scales of keys 32i + g + 8q (q = 0..3): lane g + 8q, register i
      float ks4[4], vs4[4];
      {
        const float kse = i == 0 ? ksp[0] : i == 1 ? ksp[1] : i == 2 ? ksp[2] : ksp[3];
        const float vse = i == 0 ? vsp[0] : i == 1 ? vsp[1] : i == 2 ? vsp[2] : vsp[3];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          ks4[q] = __shfl_sync(0xffffffffu, kse, g + 8 * q);
          vs4[q] = __shfl_sync(0xffffffffu, vse, g + 8 * q);
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[cst], cph))) {
        failed = true;
        break;
      }
      const uint8_t* Kt = sm.ring[kw][cst][0];
      const uint8_t* Vt = sm.ring[kw][cst][1];
      // ---- QK for both 16-key halves hf.  sc[hf][nr]: [0] key 16hf+g row 2c,
      // [1] key 16hf+g row 2c+1, [2] key 16hf+g+8 row 2c, [3] key 16hf+g+8 row
      // 2c+1 (rows inside n-tile nr).
      float sc[2][NR][4];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int ra = 16 * hf + g, rb = ra + 8;
        const uint4 a_lo = lds128(Kt + swz(ra, 2 * c)), a_hi = lds128(Kt + swz(ra, 2 * c + 1));
        const uint4 b_lo = lds128(Kt + swz(rb, 2 * c)), b_hi = lds128(Kt + swz(rb, 2 * c + 1));
        const uint32_t wa[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
        const uint32_t wb[8] = {b_lo.x, b_lo.y, b_lo.z, b_lo.w, b_hi.x, b_hi.y, b_hi.z, b_hi.w};
        if constexpr (kQK8) {
          int iacc[4] = {0, 0, 0, 0}, iacc2[4] = {0, 0, 0, 0};
#pragma unroll
          for (int s = 0; s < 4; ++s)
            mma_i8((s & 1) ? iacc2 : iacc, wa[2 * s], wb[2 * s], wa[2 * s + 1], wb[2 * s + 1],
                   qw8[2 * s], qw8[2 * s + 1]);
#pragma unroll
          for (int u = 0; u < 4; ++u) sc[hf][0][u] = __int2float_rn(iacc[u] + iacc2[u]);
        } else {
          float sacc[NR][4], sacc2[NR][4];
#pragma unroll
          for (int nr = 0; nr < NR; ++nr)
#pragma unroll
            for (int u = 0; u < 4; ++u) sacc[nr][u] = sacc2[nr][u] = 0.0f;
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const uint32_t xa = wa[s] ^ 0x80808080u, xb = wb[s] ^ 0x80808080u;
            const uint32_t af[4] = {i8pair_to_h2(xa, 0x4140u), i8pair_to_h2(xb, 0x4140u),
                                    i8pair_to_h2(xa, 0x4342u), i8pair_to_h2(xb, 0x4342u)};
#pragma unroll
            for (int nr = 0; nr < NR; ++nr)
              mma_f16((s & 1) ? sacc2[nr] : sacc[nr], af, sm.qfrag[grp][nr][s][lane]);
          }
#pragma unroll
          for (int nr = 0; nr < NR; ++nr)
#pragma unroll
            for (int u = 0; u < 4; ++u) sc[hf][nr][u] = __fadd_rn(sacc[nr][u], sacc2[nr][u]);
        }
      }

      // ---- scores s = ((S * (qs * ks)) * sm_scale), rounded as written,
      // masked past each row's L (only the last block of a sequence has keys
      // some row does not see)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int nr = 0; nr < NR; ++nr)
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {            // k2: key g (0) or g + 8 (1)
            const float ksv = ks4[2 * hf + k2];
            const float2 qk = f2_mul(make_float2(qs_row[nr][0], qs_row[nr][1]), make_float2(ksv, ksv));
            float2 s2 = f2_mul(make_float2(sc[hf][nr][2 * k2], sc[hf][nr][2 * k2 + 1]), qk);
            s2 = f2_mul(s2, make_float2(p.sm_scale, p.sm_scale));
            sc[hf][nr][2 * k2] = s2.x;
            sc[hf][nr][2 * k2 + 1] = s2.y;
          }
      if (t0 + kBlockBk > ctx) {                    // ctx is the smallest L of any row
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int nr = 0; nr < NR; ++nr)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int key = t0 + 16 * hf + g + 8 * (u >> 1);
              if (key >= Lrow[nr][u & 1]) sc[hf][nr][u] = -INFINITY;
            }
      }

      // ---- online softmax update of rows 8nr + 2c + e over the 32-key block;
      // a = round_p(p) * v_scale is kept in the score layout (sc is done with)
      float alpha[NR][2];
      bool rescale = false;
#pragma unroll
      for (int nr = 0; nr < NR; ++nr)
        softmax_tile<PM>(sc[0][nr], sc[1][nr], m_run[nr], l_run[nr], up_row[nr], vs4, alpha[nr],
                         rescale);
      if (rescale) {
#pragma unroll
        for (int md = 0; md < 8; ++md)
#pragma unroll
          for (int nr = 0; nr < NR; ++nr) {
            const float2 a2 = make_float2(alpha[nr][0], alpha[nr][1]);
            const float2 lo = f2_mul(make_float2(o[md][nr][0], o[md][nr][1]), a2);
            const float2 hi = f2_mul(make_float2(o[md][nr][2], o[md][nr][3]), a2);
            o[md][nr][0] = lo.x; o[md][nr][1] = lo.y; o[md][nr][2] = hi.x; o[md][nr][3] = hi.y;
          }
      }

      // ---- PV, one 16-key half at a time, on the f16 MMA (m16n8k16)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        // B fragments (query rows on N): b0 = {a[key 2c][row g], a[key 2c+1][row g]},
        // b1 = {a[key 2c+8][row g], a[key 2c+9][row g]} (keys of the half), each
        // split into f16 hi + lo.  a[key x][row y] sits in lane
        // 4 * (x & 7) + (y >> 1), register (x >= 8 ? 2 : 0) + (y & 1) of the
        // score layout.
        uint2 bhi[NR], blo[NR];
        {
          const int srcA = 8 * c + (g >> 1), srcB = srcA + 4;
          const bool odd = g & 1;
#pragma unroll
          for (int nr = 0; nr < NR; ++nr) {
            float fA[4], fB[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              fA[u] = __shfl_sync(0xffffffffu, sc[hf][nr][u], srcA);
              fB[u] = __shfl_sync(0xffffffffu, sc[hf][nr][u], srcB);
            }
            split_f16x2(odd ? fA[1] : fA[0], odd ? fB[1] : fB[0], bhi[nr].x, blo[nr].x);
            split_f16x2(odd ? fA[3] : fA[2], odd ? fB[3] : fB[2], bhi[nr].y, blo[nr].y);
          }
        }
        // A = V^T (MMA rows = channels, cols = keys).  Thread (g, c) reads keys
        // 2c, 2c+1, 2c+8, 2c+9 of the half and channels 16g .. 16g+15; m-tile
        // md row g is d = 16g + 2md, row g + 8 is d + 1.  One byte permute
        // pairs the two keys of a channel, a second places each byte (XOR 0x80)
        // in the mantissa of 1024, and 1152 is subtracted: exact f16 values.
        const int kr = 16 * hf + 2 * c;
        const uint4 vw0 = lds128(Vt + swz(kr, g)), vw1 = lds128(Vt + swz(kr + 1, g));
        const uint4 vw2 = lds128(Vt + swz(kr + 8, g)), vw3 = lds128(Vt + swz(kr + 9, g));
        const uint32_t w0[4] = {vw0.x, vw0.y, vw0.z, vw0.w}, w1[4] = {vw1.x, vw1.y, vw1.z, vw1.w};
        const uint32_t w2[4] = {vw2.x, vw2.y, vw2.z, vw2.w}, w3[4] = {vw3.x, vw3.y, vw3.z, vw3.w};
#pragma unroll
        for (int md = 0; md < 8; ++md) {
          const int wi = md >> 1;
          const uint32_t sel = (md & 1) ? 0x7362u : 0x5140u;   // bytes j, j+1 of both words
          const uint32_t t01 = __byte_perm(w0[wi], w1[wi], sel) ^ 0x80808080u;
          const uint32_t t23 = __byte_perm(w2[wi], w3[wi], sel) ^ 0x80808080u;
          const uint32_t af[4] = {i8pair_to_h2(t01, 0x4140u), i8pair_to_h2(t01, 0x4342u),
                                  i8pair_to_h2(t23, 0x4140u), i8pair_to_h2(t23, 0x4342u)};
#pragma unroll
          for (int nr = 0; nr < NR; ++nr) {
            mma_f16(o[md][nr], af, bhi[nr]);
            if constexpr (PM != KATTN_P_E4M3_DIRECT) mma_f16(o[md][nr], af, blo[nr]);
          }
        }
      }

      __syncwarp();
      if constexpr (NG > 1) {
        if (lane == 0) mbar_arrive(&empty[cst]);  // this group is done with the stage
      }
      if (producer) --inflight;
      if (++cst == kRing) {
        cst = 0;
        cph ^= 1u;
      }
      if (!produce()) {                           // refill the stage just read
        failed = true;
        break;
      }
    }

    // ---- per-span row sums and maxima
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = l_run[nr][e];
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 16));
        if (g == 0) {
          sm.wl[par][grp][kw][nr * 8 + 2 * c + e] = v;
          sm.wm[par][grp][kw][nr * 8 + 2 * c + e] = m_run[nr][e];
        }
      }
    if (lane == 0 && failed) sm.fail[warp] = 1;
    __syncthreads();
    {
      int any_fail = 0;                           // uniform: read after the barrier
#pragma unroll
      for (int w = 0; w < kWarps; ++w) any_fail |= sm.fail[w];
      if (any_fail) {
        // A copy never arrived: flag it, give every copy still in flight a
        // bounded chance to land, then leave.
        if (lane == 0) {
          if (failed) atomicOr(p.err_word, KATTN_DEVERR_TIMEOUT);
          int s = cst;
          uint32_t ph = cph;
          for (int k = 0; k < inflight; ++k) {
            mbar_wait_bounded(&full[s], ph);
            if (++s == kRing) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (tid == 0 && q_pending) mbar_wait_bounded(&sm.qbar, qph);
        }
        return;
      }
    }
    // Every warp is done with this item's queries: fetch the next item's.
    if (tid == 0 && it1.b >= 0) fetch_queries(it1);

    // ---- merge of the window's 4 spans, in the fixed order
    //   o = (w0 o0 + w1 o1) + (w2 o2 + w3 o3),   w_s = e^(m_s - max_s m_s):
    // warps 1 and 3 write w o to their slot, warps 0 and 2 add theirs, warp 0
    // adds warp 2's sum and writes the result.  Slots hold a warp's
    // accumulator fragments in register order (conflict-free).
    float wt[NR][2], mwin[NR][2];
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int rr = nr * 8 + 2 * c + e;
        float m = sm.wm[par][grp][0][rr];
#pragma unroll
        for (int w = 1; w < kSpansPerCta; ++w) m = fmaxf(m, sm.wm[par][grp][w][rr]);
        mwin[nr][e] = m;
        wt[nr][e] = __fmul_rn(merge_weight(sm.wm[par][grp][kw][rr], m), down_row[nr][e]);
      }
    const int bar_pair = 1 + 2 * grp, bar_even = 2 + 2 * grp;
    float* slot = sm.slot[grp][kw >> 1];
    if (kw & 1) {
#pragma unroll
      for (int nr = 0; nr < NR; ++nr)
#pragma unroll
        for (int md = 0; md < 8; ++md)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            slot[((nr * 8 + md) * 4 + u) * 32 + lane] = __fmul_rn(o[md][nr][u], wt[nr][u & 1]);
      named_arrive(bar_pair, kSpansPerCta * 32);
    } else {
      named_sync(bar_pair, kSpansPerCta * 32);
#pragma unroll
      for (int nr = 0; nr < NR; ++nr)
#pragma unroll
        for (int md = 0; md < 8; ++md)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float& x = slot[((nr * 8 + md) * 4 + u) * 32 + lane];
            o[md][nr][u] = __fmaf_rn(o[md][nr][u], wt[nr][u & 1], x);
            if (kw == 2) x = o[md][nr][u];
          }
      named_sync(bar_even, 2 * 32);
      if (kw == 0) {
        const float* other = sm.slot[grp][1];
#pragma unroll
        for (int nr = 0; nr < NR; ++nr)
#pragma unroll
          for (int md = 0; md < 8; ++md)
#pragma unroll
            for (int u = 0; u < 4; ++u)
              o[md][nr][u] = __fadd_rn(o[md][nr][u], other[((nr * 8 + md) * 4 + u) * 32 + lane]);
        // the sequence is one window: out directly (shard mode: always a partial)
        const bool whole = !p.shard_mode && nsplit_for(ctx + M - 1) == 1;
        const int kh = it0.kh, b = it0.b;
        float* part = p.partials + (((size_t)b * p.part_ws + (it0.w - p.win_begin)) * p.Hkv + kh) *
                                       partial_stride(R);
#pragma unroll
        for (int nr = 0; nr < NR; ++nr)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int rr = nr * 8 + 2 * c + e, r = row0 + rr;
            if (r >= R) continue;
            float l = 0.0f;                       // window row sum, spans in order
#pragma unroll
            for (int w = 0; w < kSpansPerCta; ++w)
              l = __fmaf_rn(sm.wl[par][grp][w][rr], merge_weight(sm.wm[par][grp][w][rr], mwin[nr][e]), l);
            if (whole) {
              float* dst = p.out + ((int64_t)b * M * p.Hq + kh * gq) * kD + orow[nr][e];
#pragma unroll
              for (int md = 0; md < 8; ++md)
                *reinterpret_cast<float2*>(dst + 2 * md) =
                    make_float2(__fdiv_rn(o[md][nr][e], l), __fdiv_rn(o[md][nr][2 + e], l));
            } else {
              float* dst = part + (size_t)r * kD + 16 * g;
#pragma unroll
              for (int md = 0; md < 8; ++md)
                *reinterpret_cast<float2*>(dst + 2 * md) = make_float2(o[md][nr][e], o[md][nr][2 + e]);
              if (g == 0) {
                part[(size_t)R * kD + r] = mwin[nr][e];
                part[(size_t)R * kD + R + r] = l;
              }
            }
          }
      }
    }

    // ---- next item
    t += G;
    if (t >= units) break;
    it0 = it1;
    it1 = decode_unit(raw2);
    raw2 = fetch_unit(p, t + 2 * G, total, nrg);
    if (nrg > 1) place_rows(it0.rg);
    sp = span_of(it0, kw, M);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      ksp[e] = ksn[e];
      vsp[e] = vsn[e];
    }
    load_span_scales<PG>(p, it1, span_of(it1, kw, M), lane, ksn, vsn);
    qph ^= 1u;
    par ^= 1;
    rows_ahead(it1, par ^ 1);                     // the slot the producer has left
    if (pitem == 1) {
      pitem = 0;                                  // the producer is already on this item
    } else {
      psp = sp;                                   // it had nothing left to read ahead
      pblk = 0;
    }
    prod_ok = produce();
  }
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous one on the stream drains; it waits (griddepcontrol.wait)
// before it reads anything that one wrote.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr int kMaxDevices = 64;

template <int NR, int NG, int PM, bool PG>
cudaError_t launch_variant(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  const int smem = (int)sizeof(SmemT<NR, NG>) + 1024;   // + alignment slack
  constexpr int kThreads = kSpansPerCta * 32 * NG;
  const auto kern = decode_fast_kernel<NR, NG, PM, PG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // Persistent grid: every CTA the GPU holds at once (cached per device).
  static std::atomic<int> slots_cache[kMaxDevices];
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  int slots = (dev >= 0 && dev < kMaxDevices) ? slots_cache[dev].load() : 0;
  if (slots <= 0) {
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem)) !=
        cudaSuccess)
      return e;
    slots = sms * (per_sm > 0 ? per_sm : 1);
    if (dev >= 0 && dev < kMaxDevices) slots_cache[dev].store(slots);
  }
  const int64_t units = (int64_t)p.B * p.nsplit_max * p.Hkv * p.row_groups;   // an upper bound
  const int grid = (int)(units < slots ? units : slots);
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), (size_t)smem, stream, p, maps);
}

// Row groups.  With more than 8 query rows per (sequence, kv head), the rows
// of a work item can be split into groups of 8, each reduced by its own CTA
// of the one-tile kernel (int8 QK, the M = 1 per-row arithmetic, so the bytes
// of every row are unchanged); the K/V of the item is then read from L2 by
// all but the first group.  That pays where the grouped kernels would leave
// the GPU short of work: a small batch, with about as many items as CTA slots
// (speculative verify).  With many items the grouped kernels, which read
// each K/V block once into shared memory for all rows, are kept.
constexpr int64_t kRowGroupMaxItems = 4096;       // upper bound on items for the split

inline int row_groups_for(const DecodeParams& p) {
  if (p.R <= 8) return 1;
  const int64_t items = (int64_t)p.B * p.nsplit_max * p.Hkv;
  const int nrg = (p.R + 7) / 8;
  if (items > kRowGroupMaxItems || items * nrg > (int64_t)INT32_MAX / 4) return 1;
  return nrg;
}

template <int NR, int NG, bool PG>
cudaError_t launch_modes(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  switch (p.p_mode) {
    case KATTN_P_BF16: return launch_variant<NR, NG, KATTN_P_BF16, PG>(p, maps, stream);
    case KATTN_P_E4M3: return launch_variant<NR, NG, KATTN_P_E4M3, PG>(p, maps, stream);
    case KATTN_P_E4M3_X448: return launch_variant<NR, NG, KATTN_P_E4M3_X448, PG>(p, maps, stream);
    case KATTN_P_E4M3_X256: return launch_variant<NR, NG, KATTN_P_E4M3_X256, PG>(p, maps, stream);
    case KATTN_P_E4M3_DIRECT:
      return launch_variant<NR, NG, KATTN_P_E4M3_DIRECT, PG>(p, maps, stream);
    default: return launch_variant<NR, NG, KATTN_P_F32, PG>(p, maps, stream);
  }
}

}  // namespace

// The split-KV pass over a paged cache (decode_fast_paged.cu): the same
// kernel instantiated with PG = true, built in a translation unit of its own.
cudaError_t launch_split_paged(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream);

// The split-KV pass for 17..32 query rows per (sequence, kv head) with P.V on
// the fifth-generation tensor cores (decode_tc.cu), contiguous or paged cache.
cudaError_t launch_split_tc(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream);

}  // namespace kattn
