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
constexpr int kBlockBytes = kBlockBk * kD;     // one K (or V) block: 4 KB
constexpr uint32_t kSpinLimit = 1u << 22;      // bounded mbarrier waits
static_assert(kBlockBk == 32, "the MMA layout below takes a block as two halves of 16 keys");
static_assert(kSpanC == 4 * kBlockBk, "span scales are held as 4 registers per lane");

struct TmaMaps {
  CUtensorMap k, v;
};

template <int NR, int NG>
struct __align__(1024) SmemT {
  uint8_t ring[NG * kSpansPerCta][kRing][2][kBlockBytes];  // per warp: [stage][K|V]
  uint64_t full[NG * kSpansPerCta][kRing];
  uint2 qfrag[NG][NR][8][32];                   // query f16 B fragments in lane order
  int8_t q8[NG * NR * 8][kD];                   // quantized query rows
  float qs[NG * NR * 8];
  float wm[NG][kSpansPerCta][NR * 8];           // per-span running max
  float wl[NG][kSpansPerCta][NR * 8];           // per-span row sum
  int fail[NG * kSpansPerCta];                  // per warp: a block never arrived
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

// Bytes i and i+1 of a word already XORed with 0x80808080 -> the exact
// float32 values of the two int8 values (bit patterns), one paired subtract.
__device__ __forceinline__ uint2 i8pair_to_f32pair(uint32_t xored, int i) {
  const uint32_t f0 = __byte_perm(xored, 0x4B000000u, 0x7540u | (uint32_t)i);
  const uint32_t f1 = __byte_perm(xored, 0x4B000000u, 0x7540u | (uint32_t)(i + 1));
  const float2 v = f2_sub(make_float2(__uint_as_float(f0), __uint_as_float(f1)),
                          make_float2(8388736.0f, 8388736.0f));   // 2^23 + 128
  return make_uint2(__float_as_uint(v.x), __float_as_uint(v.y));
}

// 2^x by the SFU (ex2.approx; subnormal results kept, 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;\n" : "=f"(y) : "f"(x));
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
  } else if constexpr (PM == KATTN_P_E4M3) {
    return e4m3_round(p);
  } else if constexpr (PM == KATTN_P_E4M3_X448) {
    return __fmul_rn(e4m3_round(__fmul_rn(p, 448.0f)), 1.0f / 448.0f);
  } else {
    return p;
  }
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a block written by TMA
// with the 128-byte swizzle (chunk index XOR row mod 8; buffers 1 KB aligned).
__device__ __forceinline__ int swz(int row, int chunk) {
  return row * kD + ((chunk ^ (row & 7)) << 4);
}

// ------------------------------------------------------------------ kernel
// NR: 8-row n-tiles per warp group; NG: warp groups of kSpansPerCta warps;
// PM: the P rounding (a kattn_p_mode).  Warp kw of a group reduces span kw of
// the window for the group's rows, one block of kBlockBk = 32 keys at a time
// (two MMA halves of 16 keys).
//
// QK runs on the int8 MMA (raw K words straight from shared memory, no
// conversion) when a warp holds a single n-tile of query rows; with more
// n-tiles the slow int8 tensor rate would bind, so the f16 MMA on converted
// values is used.  Both give the same exact integer scores.
#ifndef KATTN_QK_INT8
#define KATTN_QK_INT8 1
#endif
template <int NR, int NG, int PM>
__global__ void __launch_bounds__(kSpansPerCta * 32 * NG)
decode_fast_kernel(const DecodeParams p, const __grid_constant__ TmaMaps maps) {
  using Smem = SmemT<NR, NG>;
  constexpr bool kQK8 = KATTN_QK_INT8 && NR == 1;
  extern __shared__ unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  constexpr int RG = NR * 8;                     // rows per warp group
  constexpr int kWarps = kSpansPerCta * NG;
  constexpr int kThreads = kWarps * 32;
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

  // Scales of this warp's span: lane l holds keys l, l+32, l+64, l+96 (one
  // load each, issued now so they land while the first blocks stream in).
  const float* ksb = p.k_scale + (int64_t)kh * p.cap_rows + rs;
  const float* vsb = p.v_scale + (int64_t)kh * p.cap_rows + rs;
  float ksp[4], vsp[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int key = s0 + lane + 32 * e;
    ksp[e] = key < s1 ? __ldg(ksb + key) : 0.0f;
    vsp[e] = key < s1 ? __ldg(vsb + key) : 0.0f;
  }

  // ---- queries, quantized once per CTA: warp w takes rows w, w + kWarps, ...
  // (lane l: channels 4l .. 4l+3); bytes and scales go to shared memory.
  for (int r = warp; r < NG * RG; r += kWarps) {
    uint32_t w = 0;
    float qsc = 0.0f;
    if (r < R) {
      const int j = r / gq, h = kh * gq + r % gq;
      w = warp_quantize_row(p.q + (((int64_t)b * p.M + j) * p.Hq + h) * kD, &qsc);
    }
    reinterpret_cast<uint32_t*>(sm.q8[r])[lane] = w;
    if (lane == 0) sm.qs[r] = qsc;
  }
  __syncthreads();                                // query bytes and every warp's mbarriers ready

  // Thread (g, c) takes bytes [32c, 32c + 32) of row 8nr + g.  For the int8
  // MMA, step s covers d = 32c + 8s + 0..7 (words 2s, 2s + 1); for the f16
  // MMA, step s maps k = 2c,2c+1 -> d = 32c+4s+{0,1} and 2c+8,2c+9 ->
  // 32c+4s+{2,3}.  Either is a fixed permutation of d shared with the K
  // fragments, and the sums are integers, so both are exact.
  uint32_t qw8[8];
  if constexpr (kQK8) {
    const uint4* src = reinterpret_cast<const uint4*>(&sm.q8[row0 + g][32 * c]);
    const uint4 lo = src[0], hi = src[1];
    qw8[0] = lo.x; qw8[1] = lo.y; qw8[2] = lo.z; qw8[3] = lo.w;
    qw8[4] = hi.x; qw8[5] = hi.y; qw8[6] = hi.z; qw8[7] = hi.w;
  } else {
    if (kw < NR) {                                // warp kw builds n-tile kw of its group
      const uint4* src = reinterpret_cast<const uint4*>(&sm.q8[row0 + kw * 8 + g][32 * c]);
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
  float qs_row[NR][2];                            // scales of rows 8nr + 2c + e
#pragma unroll
  for (int nr = 0; nr < NR; ++nr)
#pragma unroll
    for (int e = 0; e < 2; ++e) qs_row[nr][e] = sm.qs[row0 + nr * 8 + 2 * c + e];

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

  int fail_blk = -1;
  int st = 0;                                     // ring stage of block i
  uint32_t ph = 0;                                // its mbarrier phase parity
  for (int i = 0; i < nb; ++i) {
    const int t0 = s0 + i * kBlockBk;
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
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[st], ph))) {
      fail_blk = i;
      break;
    }
    const uint8_t* Kt = sm.ring[warp][st][0];
    const uint8_t* Vt = sm.ring[warp][st][1];

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

    // ---- scores s = ((S * (qs * ks)) * sm_scale), masked past each row's L
    const bool all_visible = t0 + kBlockBk <= ctx;   // ctx is the smallest L of any row
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
          const int key = t0 + 16 * hf + g + 8 * k2;
          sc[hf][nr][2 * k2] = (all_visible || key < Lrow[nr][0]) ? s2.x : -INFINITY;
          sc[hf][nr][2 * k2 + 1] = (all_visible || key < Lrow[nr][1]) ? s2.y : -INFINITY;
        }

    // ---- online softmax update of rows 8nr + 2c + e over the 32-key block
    float alpha[NR][2];
    bool rescale = false;
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float bm = fmaxf(fmaxf(sc[0][nr][e], sc[0][nr][2 + e]), fmaxf(sc[1][nr][e], sc[1][nr][2 + e]));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        const float mnew = fmaxf(m_run[nr][e], bm);
        float a = 1.0f, pk[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
        if (mnew != -INFINITY) {                  // else: no visible key yet, row untouched
          a = exp_diff(m_run[nr][e], mnew);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            pk[hf][0] = exp_diff(sc[hf][nr][e], mnew);
            pk[hf][1] = exp_diff(sc[hf][nr][2 + e], mnew);
          }
        }
        alpha[nr][e] = a;
        rescale |= (a != 1.0f);
        m_run[nr][e] = mnew;
        l_run[nr][e] = __fmaf_rn(l_run[nr][e], a,
                                 __fadd_rn(__fadd_rn(pk[0][0], pk[0][1]), __fadd_rn(pk[1][0], pk[1][1])));
        // a = round_p(p) * v_scale, kept in the score layout (sc is done with)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          sc[hf][nr][e] = __fmul_rn(round_p_t<PM>(pk[hf][0]), vs4[2 * hf]);
          sc[hf][nr][2 + e] = __fmul_rn(round_p_t<PM>(pk[hf][1]), vs4[2 * hf + 1]);
        }
      }
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

    // ---- PV, one 16-key half at a time
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      // B fragments (tf32, query rows on N): for k-step h, b0 = P[key 2c+8h][row g],
      // b1 = P[key 2c+1+8h][row g].  P[key x][row y] sits in lane
      // 4 * (x & 7) + (y >> 1), register (x >= 8 ? 2 : 0) + (y & 1) of the
      // score layout.
      uint32_t bhi[NR][2][2], blo[NR][2][2];
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
          const float vv[2][2] = {{odd ? fA[1] : fA[0], odd ? fB[1] : fB[0]},
                                  {odd ? fA[3] : fA[2], odd ? fB[3] : fB[2]}};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t h0 = to_tf32(vv[h][0]), h1 = to_tf32(vv[h][1]);
            const float2 rest = f2_sub(make_float2(vv[h][0], vv[h][1]),
                                       make_float2(__uint_as_float(h0), __uint_as_float(h1)));
            bhi[nr][h][0] = h0;
            bhi[nr][h][1] = h1;
            blo[nr][h][0] = to_tf32(rest.x);
            blo[nr][h][1] = to_tf32(rest.y);
          }
        }
      }
      // A = V^T (MMA rows = channels, cols = keys).  Thread (g, c) reads keys
      // 2c, 2c+1, 2c+8, 2c+9 of the half and channels 16g .. 16g+15; m-tile
      // md row g is d = 16g + 2md, row g + 8 is d + 1.
      const int kr = 16 * hf + 2 * c;
      const uint4 vw0 = lds128(Vt + swz(kr, g)), vw1 = lds128(Vt + swz(kr + 1, g));
      const uint4 vw2 = lds128(Vt + swz(kr + 8, g)), vw3 = lds128(Vt + swz(kr + 9, g));
      const uint32_t x[4][4] = {
          {vw0.x ^ 0x80808080u, vw0.y ^ 0x80808080u, vw0.z ^ 0x80808080u, vw0.w ^ 0x80808080u},
          {vw1.x ^ 0x80808080u, vw1.y ^ 0x80808080u, vw1.z ^ 0x80808080u, vw1.w ^ 0x80808080u},
          {vw2.x ^ 0x80808080u, vw2.y ^ 0x80808080u, vw2.z ^ 0x80808080u, vw2.w ^ 0x80808080u},
          {vw3.x ^ 0x80808080u, vw3.y ^ 0x80808080u, vw3.z ^ 0x80808080u, vw3.w ^ 0x80808080u}};
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        const int wi = md >> 1, bi = 2 * (md & 1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint2 p01 = i8pair_to_f32pair(x[2 * h][wi], bi);       // key 2c+8h, d, d+1
          const uint2 p23 = i8pair_to_f32pair(x[2 * h + 1][wi], bi);   // key 2c+1+8h
          const uint32_t af[4] = {p01.x, p01.y, p23.x, p23.y};
#pragma unroll
          for (int nr = 0; nr < NR; ++nr) {
            mma_tf32(o[md][nr], af, bhi[nr][h][0], bhi[nr][h][1]);
            mma_tf32(o[md][nr], af, blo[nr][h][0], blo[nr][h][1]);
          }
        }
      }
    }

    // ---- refill the stage just read with block i + kRing
    __syncwarp();
    if (lane == 0 && i + kRing < nb) {
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      mbar_expect_tx(&full[st], 2 * kBlockBytes);
      tma_load_block(sm.ring[warp][st][0], &maps.k, tma_row0 + (i + kRing) * kBlockBk, &full[st]);
      tma_load_block(sm.ring[warp][st][1], &maps.v, tma_row0 + (i + kRing) * kBlockBk, &full[st]);
      ++issued;
    }
    if (++st == kRing) {
      st = 0;
      ph ^= 1u;
    }
  }

  if (lane == 0) {
    sm.fail[warp] = fail_blk >= 0;
    if (fail_blk >= 0) {
      // A block never arrived: flag it and give the copies still in flight a
      // bounded chance to land before the CTA leaves.
      atomicOr(p.err_word, KATTN_DEVERR_TIMEOUT);
      for (int i = fail_blk; i < issued; ++i)
        mbar_wait_bounded(&full[i % kRing], (uint32_t)((i / kRing) & 1));
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
        sm.wl[grp][kw][nr * 8 + 2 * c + e] = v;
        sm.wm[grp][kw][nr * 8 + 2 * c + e] = m_run[nr][e];
      }
    }
  __syncthreads();
  {
    int any_fail = 0;                             // uniform: read after the barrier
#pragma unroll
    for (int w = 0; w < kWarps; ++w) any_fail |= sm.fail[w];
    if (any_fail) return;
  }

  // ---- merge the window's 4 spans in span order: each warp writes its o,
  // weighted by e^(m_span - m_window), to its own slot; one barrier; then
  // every (row, d) sums the slots in order.  The TMA ring is idle now and
  // holds the slots: [kSpansPerCta][NG * RG][kD].
  float* slots = reinterpret_cast<float*>(&sm.ring[0][0][0][0]);
  constexpr int kSlot = NG * RG * kD;
  static_assert(sizeof(sm.ring) >= kSpansPerCta * kSlot * sizeof(float),
                "the idle TMA ring must hold one slot per span");
#pragma unroll
  for (int nr = 0; nr < NR; ++nr) {
    float wt[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int rr = nr * 8 + 2 * c + e;
      float m = sm.wm[grp][0][rr];
#pragma unroll
      for (int w = 1; w < kSpansPerCta; ++w) m = fmaxf(m, sm.wm[grp][w][rr]);
      wt[e] = merge_weight(sm.wm[grp][kw][rr], m);
    }
#pragma unroll
    for (int md = 0; md < 8; ++md)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int rr = row0 + nr * 8 + 2 * c + (u & 1);
        slots[kw * kSlot + rr * kD + 16 * g + 2 * md + (u >> 1)] = __fmul_rn(o[md][nr][u], wt[u & 1]);
      }
  }
  __syncthreads();

  const int64_t out_b = (int64_t)b * p.M;
  const size_t pstride = (size_t)R * (kD + 2);
  float* part = p.partials + (((size_t)b * p.nsplit_max + split) * p.Hkv + kh) * pstride;
  for (int i = tid; i < R * kD; i += kThreads) {
    const int r = i / kD, gi = r / RG, rr = r % RG;
    float m = sm.wm[gi][0][rr];
#pragma unroll
    for (int w = 1; w < kSpansPerCta; ++w) m = fmaxf(m, sm.wm[gi][w][rr]);
    float l = 0.0f, ov = 0.0f;
#pragma unroll
    for (int w = 0; w < kSpansPerCta; ++w) {
      l = __fmaf_rn(sm.wl[gi][w][rr], merge_weight(sm.wm[gi][w][rr], m), l);
      ov = (w == 0) ? slots[i] : __fadd_rn(ov, slots[w * kSlot + i]);
    }
    if (nsplit == 1) {                            // the whole sequence: final output
      const int j = r / gq, h = kh * gq + r % gq;
      p.out[((out_b + j) * p.Hq + h) * kD + i % kD] = __fdiv_rn(ov, l);
    } else {                                      // this window's partial (m, l, o)
      part[i] = ov;
      if (i % kD == 0) {
        part[(size_t)R * kD + r] = m;
        part[(size_t)R * kD + R + r] = l;
      }
    }
  }
}

// Merge of the 512-key windows of every (sequence, kv head) with more than one
// window: M* = max_s m_s, w_s = e^(m_s - M*), out = sum_s w_s o_s / sum_s w_s l_s.
// One CTA of 4 warps per (row, kv head, sequence), launched right after
// decode_fast_kernel on the same stream (so every partial is in place).
// Lane l covers channels 4l .. 4l+3; warp w takes windows s = w, w+4, ...
// and sums them in window order; the 4 warp sums are added in warp order.
// M* and l are block reductions in a fixed order.  Every step depends only
// on the row's own windows, never on the batch.
constexpr int kMergeWarps = 4;

__global__ void __launch_bounds__(kMergeWarps * 32) merge_windows_kernel(const DecodeParams p) {
  __shared__ float red[kMergeWarps];
  __shared__ float4 part_o[kMergeWarps][32];
  const int r = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = p.R, gq = p.g;
  const int64_t rs = p.row_start[b];
  const int ctx = p.ctx_len[b];
  if (!sequence_ok(rs, ctx, p.M, p.cap_rows, p.max_ctx)) return;   // NaN rows already written
  if (nsplit_for(ctx + p.M - 1) == 1) return;   // written directly by the decode kernel
  const int ns = nsplit_for(ctx + r / gq);      // windows this row sees
  const size_t pstride = (size_t)R * (kD + 2);
  const size_t sstride = (size_t)p.Hkv * pstride;
  const float* part0 = p.partials + ((size_t)b * p.nsplit_max * p.Hkv + kh) * pstride;
  const float* mcol = part0 + (size_t)R * kD + r;   // m of window s at mcol + s * sstride
  const float* lcol = mcol + R;

  // M*: thread t takes windows t, t + 128, ...; then warp and block maxima.
  float mloc = -INFINITY;
  for (int s = tid; s < ns; s += kMergeWarps * 32) mloc = fmaxf(mloc, __ldcg(mcol + s * sstride));
  mloc = warp_max(mloc);
  if (lane == 0) red[warp] = mloc;
  __syncthreads();
  float mstar = red[0];
#pragma unroll
  for (int w = 1; w < kMergeWarps; ++w) mstar = fmaxf(mstar, red[w]);
  __syncthreads();

  // l = sum_s w_s l_s: per-thread sums in window order, then warp butterflies,
  // then warps in order.
  float lloc = 0.0f;
  for (int s = tid; s < ns; s += kMergeWarps * 32)
    lloc = __fmaf_rn(exp_diff(__ldcg(mcol + s * sstride), mstar), __ldcg(lcol + s * sstride), lloc);
  lloc = warp_sum(lloc);
  if (lane == 0) red[warp] = lloc;

  // o: warp w sums windows w, w + 4, ... in order (float4 per lane).
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* ocol = part0 + (size_t)r * kD + 4 * lane;
#pragma unroll 4
  for (int s = warp; s < ns; s += kMergeWarps) {
    const float w = exp_diff(__ldcg(mcol + s * sstride), mstar);
    const float4 v = __ldcg(reinterpret_cast<const float4*>(ocol + s * sstride));
    acc.x = __fmaf_rn(w, v.x, acc.x);
    acc.y = __fmaf_rn(w, v.y, acc.y);
    acc.z = __fmaf_rn(w, v.z, acc.z);
    acc.w = __fmaf_rn(w, v.w, acc.w);
  }
  part_o[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float l = red[0];
    float4 o = part_o[0][lane];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) {
      l = __fadd_rn(l, red[w]);
      const float4 v = part_o[w][lane];
      o.x = __fadd_rn(o.x, v.x);
      o.y = __fadd_rn(o.y, v.y);
      o.z = __fadd_rn(o.z, v.z);
      o.w = __fadd_rn(o.w, v.w);
    }
    const int j = r / gq, h = kh * gq + r % gq;
    float4* dst = reinterpret_cast<float4*>(p.out + ((((int64_t)b * p.M + j) * p.Hq + h) * kD)) + lane;
    *dst = make_float4(__fdiv_rn(o.x, l), __fdiv_rn(o.y, l), __fdiv_rn(o.z, l), __fdiv_rn(o.w, l));
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

template <int NR, int NG, int PM>
cudaError_t launch_variant(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  const int smem = (int)sizeof(SmemT<NR, NG>) + 1024;   // + alignment slack
  const auto kern = decode_fast_kernel<NR, NG, PM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)p.nsplit_max, (unsigned)p.Hkv, (unsigned)p.B);
  kern<<<grid, kSpansPerCta * 32 * NG, smem, stream>>>(p, maps);
  return cudaGetLastError();
}

template <int NR, int NG>
cudaError_t launch_rows(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  switch (p.p_mode) {
    case KATTN_P_BF16: return launch_variant<NR, NG, KATTN_P_BF16>(p, maps, stream);
    case KATTN_P_E4M3: return launch_variant<NR, NG, KATTN_P_E4M3>(p, maps, stream);
    case KATTN_P_E4M3_X448: return launch_variant<NR, NG, KATTN_P_E4M3_X448>(p, maps, stream);
    default: return launch_variant<NR, NG, KATTN_P_F32>(p, maps, stream);
  }
}

}  // namespace

cudaError_t launch_decode_fast(const DecodeParams& p, cudaStream_t stream) {
  TmaMaps maps;
  const int64_t rows = (int64_t)p.Hkv * p.cap_rows;
  if (!encode_cache_map(&maps.k, p.k, rows) || !encode_cache_map(&maps.v, p.v, rows))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (p.R <= 8) e = launch_rows<1, 1>(p, maps, stream);
  else if (p.R <= 16) e = launch_rows<2, 1>(p, maps, stream);
  else if (p.R <= 32) e = launch_rows<4, 1>(p, maps, stream);
  else e = launch_rows<4, 2>(p, maps, stream);
  if (e != cudaSuccess || p.nsplit_max <= 1) return e;
  merge_windows_kernel<<<dim3((unsigned)p.R, (unsigned)p.Hkv, (unsigned)p.B), kMergeWarps * 32, 0,
                         stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kattn
