// Fast decode over the int8 KV cache: split-KV on tensor cores, fixed-order merge.
//
// Work decomposition (all positions absolute within the sequence, fixed at
// compile time):
//   * keys are cut into spans of kSpanC = 128; one warp reduces one span with
//     its own running max, kBlockBk = 16 keys at a time ("在 agent 时代如何快速
//     验证 kernel 对精度的影响", section "注意力权重": blockwise online softmax,
//     P rounded only where it multiplies V, row sum from the unrounded P);
//   * a CTA (grid (nsplit, Hkv, B)) owns a window of 4 consecutive spans of
//     one (sequence, kv head) for all R = g*M query rows that read that kv
//     head -- the GQA group times the M draft columns -- so every K/V byte is
//     read from HBM once; its 4 warps merge their spans at the end;
//   * the last CTA of a (sequence, kv head) -- found with an acq_rel ticket,
//     nothing ever waits for another CTA -- merges the windows in order and
//     divides by the row sum.
//
// Per warp and block of 16 keys:
//   * TMA (cp.async.bulk.tensor, 128-byte swizzle) streams the K and V rows of
//     the block into the warp's own ring of shared-memory stages; lane 0 is
//     the producer, one mbarrier per stage, every wait bounded;
//   * QK on tensor cores: mma.sync m16n8k16 f16 with f32 accumulation over the
//     int8 values (exact in f16); every partial sum is an integer below 2^24,
//     so the f32 scores equal the int32 dot products exactly.  Keys sit on the
//     MMA's M side, query rows on N (8 per n-tile);
//   * scores, the block max (warp shuffles), the online update of m and l, P
//     rounding and a = round_p(p) * v_scale in f32 registers;
//   * PV on tensor cores: mma.sync m16n8k8 tf32 with V (int8, exact in tf32)
//     on the A side and a split into tf32 hi + lo on the B side, accumulated
//     in f32; the split keeps float32-level accuracy with no data-dependent
//     scaling.
//
// Batch invariance ("Kestrel_VLLM - 18" §二): the bytes of a query row depend
// only on its own keys: spans, blocks and windows sit at fixed key positions,
// a block with no visible key leaves a row untouched, each MMA output element
// depends only on its own row's operands, and every merge runs in a fixed
// order that does not depend on R, M, B or the grid.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "device_common.cuh"

namespace kattn {
namespace {

#ifndef KATTN_STAGES
#define KATTN_STAGES 3
#endif
constexpr int kRing = KATTN_STAGES;            // TMA stages per warp
constexpr int kBlockBytes = kBlockBk * kD;     // one K (or V) block: 2 KB
constexpr uint32_t kSpinLimit = 1u << 22;      // bounded mbarrier waits
static_assert(kBlockBk == 16, "the MMA layout below assumes 16 keys per block");

struct TmaMaps {
  CUtensorMap k, v;
};

template <int NR, int NG>
struct __align__(1024) SmemT {
  uint8_t ring[NG * kSpansPerCta][kRing][2][kBlockBytes];  // per warp: [stage][K|V]
  uint64_t full[NG * kSpansPerCta][kRing];
  uint2 qfrag[NG][NR][8][32];                   // query B fragments in lane order
  float qs[NG * NR * 8];
  float wm[NG][kSpansPerCta][NR * 8];           // per-span running max
  float wl[NG][kSpansPerCta][NR * 8];           // per-span row sum
  int fail;
  int last;
};

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
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

// kBlockBk rows x 128 bytes starting at row `row` of a 2-D cache view.
__device__ __forceinline__ void tma_load_block(void* dst, const CUtensorMap* map, int row,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(smem_u32(dst)),
      "l"(map), "r"(0), "r"(row), "r"(smem_u32(bar))
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

// Byte i of a word already XORed with 0x80808080 -> exact float32 of the int8
// value: the byte becomes the low mantissa of 2^23, then 2^23 + 128 is subtracted.
__device__ __forceinline__ float i8_to_f32(uint32_t xored, int i) {
  const uint32_t f = __byte_perm(xored, 0x4B000000u, 0x7540u | (uint32_t)i);
  return __fsub_rn(__uint_as_float(f), 8388736.0f);
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint2 b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// e^(x - m) for x <= m, m finite: the difference first (exact near the max,
// where the weights matter), then base 2.  exp2f(-inf) = 0.
__device__ __forceinline__ float exp_diff(float x, float m) {
  return exp2f(__fmul_rn(__fsub_rn(x, m), kLog2e));
}

// Weight of a partial with running max x in a merge whose max is m.
__device__ __forceinline__ float merge_weight(float x, float m) {
  return m == -INFINITY ? 0.0f : exp_diff(x, m);
}

__device__ __forceinline__ float round_p_fast(float p, int mode) {
  switch (mode) {
    case KATTN_P_BF16: return bf16_round(p);
    case KATTN_P_E4M3: return e4m3_round(p);
    case KATTN_P_E4M3_X448: return __fmul_rn(e4m3_round(__fmul_rn(p, 448.0f)), 1.0f / 448.0f);
    default: return p;
  }
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a block written by TMA
// with the 128-byte swizzle (chunk index XOR row mod 8; buffers 1 KB aligned).
__device__ __forceinline__ int swz(int row, int chunk) {
  return row * kD + ((chunk ^ (row & 7)) << 4);
}

// ------------------------------------------------------------------ kernel
// NR: 8-row n-tiles per warp group; NG: warp groups of kSpansPerCta warps.
// Warp kw of a group reduces span kw of the window for the group's rows.
template <int NR, int NG>
__global__ void __launch_bounds__(kSpansPerCta * 32 * NG)
decode_fast_kernel(const DecodeParams p, const __grid_constant__ TmaMaps maps) {
  using Smem = SmemT<NR, NG>;
  extern __shared__ unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  constexpr int RG = NR * 8;                     // rows per warp group
  constexpr int kThreads = kSpansPerCta * 32 * NG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kw = warp % kSpansPerCta, grp = warp / kSpansPerCta;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int R = p.R, gq = p.g;
  const int row0 = grp * RG;

  const int64_t rs = p.row_start[b];
  const int ctx = p.ctx_len[b];
  if (!sequence_ok(rs, ctx, p.M, p.cap_rows, p.max_ctx)) {
    if (split == 0) {
      for (int i = tid; i < R * kD; i += kThreads) {
        const int r = i / kD, j = r / gq, h = kh * gq + r % gq;
        p.out[(((int64_t)b * p.M + j) * p.Hq + h) * kD + i % kD] = __int_as_float(0x7fc00000);
      }
      if (tid == 0 && kh == 0) atomicOr(p.err_word, KATTN_DEVERR_BAD_SEQUENCE);
    }
    return;
  }
  const int Lmax = ctx + p.M - 1;
  const int nsplit = nsplit_for(Lmax);
  if (split >= nsplit) return;
  const int k0 = split * kSplitC;
  const int k1 = min(k0 + kSplitC, Lmax);
  // this warp's span [s0, s1) and its blocks
  const int s0 = k0 + kw * kSpanC;
  const int s1 = min(s0 + kSpanC, k1);
  const int nb = s1 > s0 ? (s1 - s0 + kBlockBk - 1) / kBlockBk : 0;
  const int tma_row0 = (int)((int64_t)kh * p.cap_rows + rs + s0);
  uint64_t* full = sm.full[warp];

  // ---- per-warp barriers and the first TMA loads (lane 0 is the producer)
  int issued = 0;                                 // meaningful in lane 0 only
  if (lane == 0) {
    for (int s = 0; s < kRing; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    for (int s = 0; s < kRing && s < nb; ++s) {
      mbar_expect_tx(&full[s], 2 * kBlockBytes);
      tma_load_block(sm.ring[warp][s][0], &maps.k, tma_row0 + s * kBlockBk, &full[s]);
      tma_load_block(sm.ring[warp][s][1], &maps.v, tma_row0 + s * kBlockBk, &full[s]);
      ++issued;
    }
  }
  if (tid == 0) sm.fail = 0;

  // ---- queries: warp 0 of each group quantizes the group's rows and stores
  // their f16 B fragments.  Thread (g, c) covers row 8nr + g, bytes
  // [32c, 32c + 32); the logical k index of step s maps to d as
  // 2c,2c+1 -> 32c+4s+{0,1} and 2c+8,2c+9 -> 32c+4s+{2,3}, a fixed
  // permutation of d shared with the K fragments (integer sums, so exact).
  if (kw == 0) {
#pragma unroll
    for (int nr = 0; nr < NR; ++nr) {
      const int r = row0 + nr * 8 + g;
      float4 x[8];
      float amax = 0.0f;
      if (r < R) {
        const int j = r / gq, h = kh * gq + r % gq;
        const float4* src = reinterpret_cast<const float4*>(
            p.q + (((int64_t)b * p.M + j) * p.Hq + h) * kD + 32 * c);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          x[u] = src[u];
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x[u].x), fabsf(x[u].y)),
                                   fmaxf(fabsf(x[u].z), fabsf(x[u].w))));
        }
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const float qsc = quant_scale(amax);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t w = pack_i8x4(quant_one(x[s].x, qsc), quant_one(x[s].y, qsc),
                                     quant_one(x[s].z, qsc), quant_one(x[s].w, qsc)) ^
                           0x80808080u;
        sm.qfrag[grp][nr][s][lane] =
            make_uint2(i8pair_to_h2(w, 0x4140u), i8pair_to_h2(w, 0x4342u));
      }
      if (c == 0) sm.qs[row0 + nr * 8 + g] = qsc;
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
      Lrow[nr][e] = ctx + (row0 + nr * 8 + 2 * c + e) / gq;
    }
  float o[8][NR][4];
#pragma unroll
  for (int md = 0; md < 8; ++md)
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int u = 0; u < 4; ++u) o[md][nr][u] = 0.0f;

  // Scales of this thread's keys g and g + 8 of a block.
  const float* ksb = p.k_scale + (int64_t)kh * p.cap_rows + rs;
  const float* vsb = p.v_scale + (int64_t)kh * p.cap_rows + rs;
  float ks_cur[2], vs_cur[2], ks_nxt[2], vs_nxt[2];
  {
    const bool va = s0 + g < s1, vb = s0 + g + 8 < s1;
    ks_cur[0] = va ? __ldg(ksb + s0 + g) : 0.0f;
    ks_cur[1] = vb ? __ldg(ksb + s0 + g + 8) : 0.0f;
    vs_cur[0] = va ? __ldg(vsb + s0 + g) : 0.0f;
    vs_cur[1] = vb ? __ldg(vsb + s0 + g + 8) : 0.0f;
  }
  __syncthreads();                                // query fragments and barriers ready

  float qs_row[NR][2];
#pragma unroll
  for (int nr = 0; nr < NR; ++nr)
#pragma unroll
    for (int e = 0; e < 2; ++e) qs_row[nr][e] = sm.qs[row0 + nr * 8 + 2 * c + e];

  int fail_blk = -1;
  for (int i = 0; i < nb; ++i) {
    const int st = i % kRing;
    const int t0 = s0 + i * kBlockBk;
    {  // next block's scales, one block ahead
      const int tn = t0 + kBlockBk;
      const bool va = tn + g < s1, vb = tn + g + 8 < s1;
      ks_nxt[0] = va ? __ldg(ksb + tn + g) : 0.0f;
      ks_nxt[1] = vb ? __ldg(ksb + tn + g + 8) : 0.0f;
      vs_nxt[0] = va ? __ldg(vsb + tn + g) : 0.0f;
      vs_nxt[1] = vb ? __ldg(vsb + tn + g + 8) : 0.0f;
    }
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[st], (uint32_t)((i / kRing) & 1)))) {
      fail_blk = i;
      break;
    }
    const uint8_t* Kt = sm.ring[warp][st][0];
    const uint8_t* Vt = sm.ring[warp][st][1];

    // ---- QK: A = K rows g and g + 8 of the block, f16.  Even and odd k-steps
    // accumulate separately (shorter chains); both hold exact integers below
    // 2^24, so their sum is exact.
    float sacc[NR][4], sacc2[NR][4];
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int u = 0; u < 4; ++u) sacc[nr][u] = sacc2[nr][u] = 0.0f;
    {
      const uint4 a_lo = lds128(Kt + swz(g, 2 * c)), a_hi = lds128(Kt + swz(g, 2 * c + 1));
      const uint4 b_lo = lds128(Kt + swz(g + 8, 2 * c)), b_hi = lds128(Kt + swz(g + 8, 2 * c + 1));
      const uint32_t wa[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
      const uint32_t wb[8] = {b_lo.x, b_lo.y, b_lo.z, b_lo.w, b_hi.x, b_hi.y, b_hi.z, b_hi.w};
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
        for (int u = 0; u < 4; ++u) sacc[nr][u] = __fadd_rn(sacc[nr][u], sacc2[nr][u]);
    }

    // ---- scores.  sacc[nr]: [0] key g row 2c, [1] key g row 2c+1,
    // [2] key g+8 row 2c, [3] key g+8 row 2c+1 (rows inside n-tile nr).
    float sc[NR][4];
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = u & 1, key = t0 + g + ((u < 2) ? 0 : 8);
        const float ksv = (u < 2) ? ks_cur[0] : ks_cur[1];
        const float s =
            __fmul_rn(__fmul_rn(sacc[nr][u], __fmul_rn(qs_row[nr][e], ksv)), p.sm_scale);
        sc[nr][u] = (key < Lrow[nr][e]) ? s : -INFINITY;
      }

    // ---- online softmax update of rows 8nr + 2c + e (block max by shuffles)
    float alpha[NR][2], pv[NR][4];
    bool rescale = false;
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float bm = fmaxf(sc[nr][e], sc[nr][2 + e]);
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        const float mnew = fmaxf(m_run[nr][e], bm);
        float a, p0, p1;
        if (mnew == -INFINITY) {                  // no visible key yet: row untouched
          a = 1.0f;
          p0 = p1 = 0.0f;
        } else {
          a = exp_diff(m_run[nr][e], mnew);
          p0 = exp_diff(sc[nr][e], mnew);
          p1 = exp_diff(sc[nr][2 + e], mnew);
        }
        alpha[nr][e] = a;
        rescale |= (a != 1.0f);
        m_run[nr][e] = mnew;
        l_run[nr][e] = __fmaf_rn(l_run[nr][e], a, __fadd_rn(p0, p1));
        pv[nr][e] = __fmul_rn(round_p_fast(p0, p.p_mode), vs_cur[0]);
        pv[nr][2 + e] = __fmul_rn(round_p_fast(p1, p.p_mode), vs_cur[1]);
      }
    if (rescale) {
#pragma unroll
      for (int md = 0; md < 8; ++md)
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) {
          o[md][nr][0] = __fmul_rn(o[md][nr][0], alpha[nr][0]);
          o[md][nr][1] = __fmul_rn(o[md][nr][1], alpha[nr][1]);
          o[md][nr][2] = __fmul_rn(o[md][nr][2], alpha[nr][0]);
          o[md][nr][3] = __fmul_rn(o[md][nr][3], alpha[nr][1]);
        }
    }

    // ---- PV B fragments (tf32, query rows on N): for k-step h,
    // b0 = P[key 2c + 8h][row g], b1 = P[key 2c + 1 + 8h][row g].
    // P[key x][row y] sits in lane 4 * (x & 7) + (y >> 1), register
    // (x >= 8 ? 2 : 0) + (y & 1) of the score layout.
    uint32_t bhi[NR][2][2], blo[NR][2][2];
    {
      const int srcA = 8 * c + (g >> 1), srcB = srcA + 4;
      const bool odd = g & 1;
#pragma unroll
      for (int nr = 0; nr < NR; ++nr) {
        float fA[4], fB[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          fA[u] = __shfl_sync(0xffffffffu, pv[nr][u], srcA);
          fB[u] = __shfl_sync(0xffffffffu, pv[nr][u], srcB);
        }
        const float vv[2][2] = {{odd ? fA[1] : fA[0], odd ? fB[1] : fB[0]},
                                {odd ? fA[3] : fA[2], odd ? fB[3] : fB[2]}};
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint32_t hi = to_tf32(vv[h][q]);
            bhi[nr][h][q] = hi;
            blo[nr][h][q] = to_tf32(__fsub_rn(vv[h][q], __uint_as_float(hi)));
          }
      }
    }

    // ---- PV: A = V^T (MMA rows = channels, cols = keys).  Thread (g, c)
    // reads keys 2c, 2c+1, 2c+8, 2c+9 of the block and channels 16g..16g+15;
    // m-tile md row g is d = 16g + 2md, row g + 8 is d + 1.
    {
      uint4 vw[4];
      vw[0] = lds128(Vt + swz(2 * c, g));
      vw[1] = lds128(Vt + swz(2 * c + 1, g));
      vw[2] = lds128(Vt + swz(2 * c + 8, g));
      vw[3] = lds128(Vt + swz(2 * c + 9, g));
      uint32_t x[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[k][0] = vw[k].x ^ 0x80808080u;
        x[k][1] = vw[k].y ^ 0x80808080u;
        x[k][2] = vw[k].z ^ 0x80808080u;
        x[k][3] = vw[k].w ^ 0x80808080u;
      }
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        const int wi = md >> 1, bi = 2 * (md & 1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t af[4] = {__float_as_uint(i8_to_f32(x[2 * h][wi], bi)),
                                  __float_as_uint(i8_to_f32(x[2 * h][wi], bi + 1)),
                                  __float_as_uint(i8_to_f32(x[2 * h + 1][wi], bi)),
                                  __float_as_uint(i8_to_f32(x[2 * h + 1][wi], bi + 1))};
#pragma unroll
          for (int nr = 0; nr < NR; ++nr) {
            mma_tf32(o[md][nr], af, bhi[nr][h][0], bhi[nr][h][1]);
            mma_tf32(o[md][nr], af, blo[nr][h][0], blo[nr][h][1]);
          }
        }
      }
    }
    ks_cur[0] = ks_nxt[0];
    ks_cur[1] = ks_nxt[1];
    vs_cur[0] = vs_nxt[0];
    vs_cur[1] = vs_nxt[1];

    // ---- refill the stage just read with block i + kRing
    __syncwarp();
    if (lane == 0 && i + kRing < nb) {
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      mbar_expect_tx(&full[st], 2 * kBlockBytes);
      tma_load_block(sm.ring[warp][st][0], &maps.k, tma_row0 + (i + kRing) * kBlockBk, &full[st]);
      tma_load_block(sm.ring[warp][st][1], &maps.v, tma_row0 + (i + kRing) * kBlockBk, &full[st]);
      ++issued;
    }
  }

  if (fail_blk >= 0 && lane == 0) {
    // A block never arrived: flag it and give the copies still in flight a
    // bounded chance to land before the CTA leaves.
    sm.fail = 1;
    atomicOr(p.err_word, KATTN_DEVERR_TIMEOUT);
    for (int i = fail_blk; i < issued; ++i)
      mbar_wait_bounded(&full[i % kRing], (uint32_t)((i / kRing) & 1));
  }

  // ---- per-span row sums and maxima, then the merge of the 4 spans
#pragma unroll
  for (int nr = 0; nr < NR; ++nr)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = l_run[nr][e];
      v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
      v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 8));
      v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 16));
      if (g == 0) {
        sm.wl[grp][kw][nr * 8 + 2 * c + e] = v;
        sm.wm[grp][kw][nr * 8 + 2 * c + e] = m_run[nr][e];
      }
    }
  __syncthreads();
  if (sm.fail) return;                            // uniform: read after the barrier

  // Window max and span weights for this thread's rows.
  float wmax[NR][2], wt[NR][2];
#pragma unroll
  for (int nr = 0; nr < NR; ++nr)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int rr = nr * 8 + 2 * c + e;
      float m = sm.wm[grp][0][rr];
#pragma unroll
      for (int w = 1; w < kSpansPerCta; ++w) m = fmaxf(m, sm.wm[grp][w][rr]);
      wmax[nr][e] = m;
      wt[nr][e] = merge_weight(sm.wm[grp][kw][rr], m);
    }
  float* O = reinterpret_cast<float*>(&sm.ring[0][0][0][0]);   // [NG * RG][kD]; ring idle
#pragma unroll
  for (int w = 0; w < kSpansPerCta; ++w) {
    if (kw == w) {
#pragma unroll
      for (int md = 0; md < 8; ++md)
#pragma unroll
        for (int nr = 0; nr < NR; ++nr)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int rr = row0 + nr * 8 + 2 * c + (u & 1);
            float* dst = O + rr * kD + 16 * g + 2 * md + (u >> 1);
            const float v = __fmul_rn(o[md][nr][u], wt[nr][u & 1]);
            *dst = (w == 0) ? v : __fadd_rn(*dst, v);
          }
    }
    __syncthreads();
  }
  // merged row max and row sum of the window, for all rows (smem)
  if (kw == 0 && g == 0) {
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int rr = nr * 8 + 2 * c + e;
        float l = 0.0f;
#pragma unroll
        for (int w = 0; w < kSpansPerCta; ++w)
          l = __fmaf_rn(sm.wl[grp][w][rr], merge_weight(sm.wm[grp][w][rr], wmax[nr][e]), l);
        sm.wl[grp][0][rr] = l;
        sm.wm[grp][0][rr] = wmax[nr][e];
      }
  }
  __syncthreads();

  const int64_t out_b = (int64_t)b * p.M;
  if (nsplit == 1) {
    for (int i = tid; i < R * kD; i += kThreads) {
      const int r = i / kD, j = r / gq, h = kh * gq + r % gq;
      p.out[((out_b + j) * p.Hq + h) * kD + i % kD] = __fdiv_rn(O[i], sm.wl[r / RG][0][r % RG]);
    }
    return;
  }

  const size_t pstride = (size_t)R * (kD + 2);
  float* part = p.partials + (((size_t)b * p.nsplit_max + split) * p.Hkv + kh) * pstride;
  for (int i = tid; i < R * kD; i += kThreads) part[i] = O[i];
  if (tid < R) {
    part[(size_t)R * kD + tid] = sm.wm[tid / RG][0][tid % RG];
    part[(size_t)R * kD + R + tid] = sm.wl[tid / RG][0][tid % RG];
  }
  __syncthreads();
  if (tid == 0) {
    // Release this CTA's partial and learn whether it was the last one; the
    // acquire half makes the other windows' partials visible to the merge.
    unsigned int* ticket = p.tickets + (size_t)b * p.Hkv + kh;
    unsigned int prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;\n"
                 : "=r"(prev)
                 : "l"(ticket)
                 : "memory");
    const int is_last = prev == (unsigned int)(nsplit - 1);
    if (is_last) atomicExch(ticket, 0u);          // leave the counter at zero
    sm.last = is_last;
  }
  __syncthreads();
  if (!sm.last) return;

  // Merge the windows in order: M* = max m_s, w_s = e^(m_s - M*),
  // out = sum w o / sum w l.
  const float* part0 = p.partials + ((size_t)b * p.nsplit_max * p.Hkv + kh) * pstride;
  const size_t sstride = (size_t)p.Hkv * pstride;
  for (int i = tid; i < R * kD; i += kThreads) {
    const int r = i / kD, d = i % kD;
    const int ns = nsplit_for(ctx + r / gq);
    float mstar = -INFINITY;
    for (int s = 0; s < ns; ++s)
      mstar = fmaxf(mstar, __ldcg(part0 + s * sstride + (size_t)R * kD + r));
    float lt = 0.0f, ot = 0.0f;
    for (int s = 0; s < ns; ++s) {
      const float* ps = part0 + s * sstride;
      const float w = exp_diff(__ldcg(ps + (size_t)R * kD + r), mstar);
      lt = __fmaf_rn(w, __ldcg(ps + (size_t)R * kD + R + r), lt);
      ot = __fmaf_rn(w, __ldcg(ps + (size_t)r * kD + d), ot);
    }
    const int j = r / gq, h = kh * gq + r % gq;
    p.out[((out_b + j) * p.Hq + h) * kD + d] = __fdiv_rn(ot, lt);
  }
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

template <int NR, int NG>
cudaError_t launch_variant(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  const int smem = (int)sizeof(SmemT<NR, NG>) + 1024;   // + alignment slack
  const auto kern = decode_fast_kernel<NR, NG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)p.nsplit_max, (unsigned)p.Hkv, (unsigned)p.B);
  kern<<<grid, kSpansPerCta * 32 * NG, smem, stream>>>(p, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_fast(const DecodeParams& p, cudaStream_t stream) {
  TmaMaps maps;
  const int64_t rows = (int64_t)p.Hkv * p.cap_rows;
  if (!encode_cache_map(&maps.k, p.k, rows) || !encode_cache_map(&maps.v, p.v, rows))
    return cudaErrorInvalidValue;
  if (p.R <= 8) return launch_variant<1, 1>(p, maps, stream);
  if (p.R <= 16) return launch_variant<2, 1>(p, maps, stream);
  if (p.R <= 32) return launch_variant<4, 1>(p, maps, stream);
  return launch_variant<4, 2>(p, maps, stream);
}

}  // namespace kattn
