// Fast decode over the int8 KV cache: split-KV with a fixed-order merge.
//
// Grid (nsplit_max, Hkv, B): CTA (s, kh, b) owns keys [s*C, (s+1)*C) of
// sequence b for every query row that reads kv head kh -- the g heads of the
// GQA group times the M draft columns (R = g*M rows), so each K/V byte is
// read from HBM once.  Inside the split, blocks of Bk keys are processed in
// order with an online softmax ("在 agent 时代如何快速验证 kernel 对精度的影响",
// section "注意力权重": running max per block, P rounded only where it
// multiplies V, row sum from the unrounded P).  The last CTA of a
// (sequence, kv head) to finish -- found with an atomic ticket, no waiting --
// merges the splits in split order and divides by the row sum.
//
// Batch invariance ("Kestrel_VLLM - 18" §二): the bytes of a query row depend
// only on its own keys.  Splits and blocks sit at fixed key positions; a
// block with no visible key for a row leaves that row untouched; every
// floating-point step of a row is an explicit single-rounding intrinsic in
// a fixed order that does not depend on R, M or B.
#include "device_common.cuh"

namespace kattn {
namespace {

constexpr int kThreads = 128;

struct SmemFast {
  int8_t kt[2][kTileBk * kD];      // K blocks, 16-byte chunks XOR-swizzled by row
  int8_t vt[2][kTileBk * kD];      // V blocks, same swizzle
  float ks[2][kTileBk];
  float vs[2][kTileBk];
  uint32_t q8[kMaxRows][kD / 4];   // quantized queries
  float qs[kMaxRows];
  float S[kMaxRows][kTileBk];      // scores of the block
  float PT[kMaxRows][kTileBk];     // round_p(p) * v_scale
  float alpha[kMaxRows];
  float m[kMaxRows];               // running max of the scores
  float l[kMaxRows];               // running row sum
  int Lr[kMaxRows];                // keys visible to the row
  int last;
};

// Byte offset of (row t, byte i) inside a swizzled 64x128 block.
__device__ __forceinline__ int swz(int t, int i) {
  return t * kD + ((((i >> 4) ^ (t & 7))) << 4) + (i & 15);
}

// e^(x - m) for x <= m.  The difference is taken first (exact when x is near
// m, where the weights matter), then scaled to base 2.  exp2f(-inf) = 0.
__device__ __forceinline__ float exp_diff(float x, float m) {
  return exp2f(__fmul_rn(__fsub_rn(x, m), kLog2e));
}

__device__ __forceinline__ float round_p_fast(float p, int mode) {
  switch (mode) {
    case KATTN_P_BF16: return bf16_round(p);
    case KATTN_P_E4M3: return e4m3_round(p);
    case KATTN_P_E4M3_X448: return __fmul_rn(e4m3_round(__fmul_rn(p, 448.0f)), 1.0f / 448.0f);
    default: return p;
  }
}

__device__ __forceinline__ void load_block(SmemFast& sm, int buf, const int8_t* kbase,
                                           const int8_t* vbase, const float* ksb,
                                           const float* vsb, int t0, int nvalid) {
  const int tid = threadIdx.x;
  // 64 rows x 8 chunks each for K and V: 4 chunks per thread per tensor.
#pragma unroll
  for (int it = 0; it < (kTileBk * kD / 16) / kThreads; ++it) {
    const int idx = it * kThreads + tid;
    const int t = idx >> 3, c = idx & 7;
    const bool ok = t < nvalid;
    const int64_t src = (int64_t)(ok ? t0 + t : t0) * kD + c * 16;
    const int dst = t * kD + ((c ^ (t & 7)) << 4);
    cp_async16(&sm.kt[buf][dst], kbase + src, ok ? 16 : 0);
    cp_async16(&sm.vt[buf][dst], vbase + src, ok ? 16 : 0);
  }
  if (tid < kTileBk) {
    const bool ok = tid < nvalid;
    cp_async4(&sm.ks[buf][tid], ksb + (ok ? t0 + tid : t0), ok ? 4 : 0);
  } else {
    const int t = tid - kTileBk;
    const bool ok = t < nvalid;
    cp_async4(&sm.vs[buf][t], vsb + (ok ? t0 + t : t0), ok ? 4 : 0);
  }
  cp_async_commit();
}

template <int RPAD>
__global__ void __launch_bounds__(kThreads)
decode_fast_kernel(DecodeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SmemFast& sm = *reinterpret_cast<SmemFast*>(smem_raw);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int R = p.R, g = p.g;

  const int64_t rs = p.row_start[b];
  const int ctx = p.ctx_len[b];
  if (!sequence_ok(rs, ctx, p.M, p.cap_rows, p.max_ctx)) {
    if (split == 0) {
      for (int r = 0; r < R; ++r) {
        const int j = r / g, h = kh * g + r % g;
        p.out[(((int64_t)b * p.M + j) * p.Hq + h) * kD + tid] = __int_as_float(0x7fc00000);
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

  const int8_t* kbase = p.k + ((int64_t)kh * p.cap_rows + rs) * kD;
  const int8_t* vbase = p.v + ((int64_t)kh * p.cap_rows + rs) * kD;
  const float* ksb = p.k_scale + (int64_t)kh * p.cap_rows + rs;
  const float* vsb = p.v_scale + (int64_t)kh * p.cap_rows + rs;

  // Prefetch the first block while the queries are quantized.
  load_block(sm, 0, kbase, vbase, ksb, vsb, k0, min(kTileBk, k1 - k0));

  for (int r = warp; r < R; r += kThreads / 32) {
    const int j = r / g, h = kh * g + r % g;
    float qsv;
    sm.q8[r][lane] = warp_quantize_row(p.q + (((int64_t)b * p.M + j) * p.Hq + h) * kD, &qsv);
    if (lane == 0) {
      sm.qs[r] = qsv;
      sm.m[r] = -INFINITY;
      sm.l[r] = 0.0f;
      sm.Lr[r] = ctx + j;
    }
  }

  float o[RPAD];
#pragma unroll
  for (int r = 0; r < RPAD; ++r) o[r] = 0.0f;

  const int nblk = (k1 - k0 + kTileBk - 1) / kTileBk;
  for (int blk = 0; blk < nblk; ++blk) {
    const int buf = blk & 1;
    const int t0 = k0 + blk * kTileBk;
    if (blk + 1 < nblk) {
      const int tn = t0 + kTileBk;
      load_block(sm, buf ^ 1, kbase, vbase, ksb, vsb, tn, min(kTileBk, k1 - tn));
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    // ---- QK: thread owns key kt and rows r = rsel, rsel + 2, ...
    {
      const int kt = tid & (kTileBk - 1);
      const int rsel = tid >> 6;
      int4 kr[kD / 16];
#pragma unroll
      for (int c = 0; c < kD / 16; ++c)
        kr[c] = *reinterpret_cast<const int4*>(&sm.kt[buf][kt * kD + ((c ^ (kt & 7)) << 4)]);
      const float ksv = sm.ks[buf][kt];
      const int tabs = t0 + kt;
      for (int r = rsel; r < R; r += 2) {
        int acc = 0;
#pragma unroll
        for (int c = 0; c < kD / 16; ++c) {
          const int4 qq = *reinterpret_cast<const int4*>(&sm.q8[r][4 * c]);
          acc = __dp4a(kr[c].x, qq.x, acc);
          acc = __dp4a(kr[c].y, qq.y, acc);
          acc = __dp4a(kr[c].z, qq.z, acc);
          acc = __dp4a(kr[c].w, qq.w, acc);
        }
        const float s = __fmul_rn(__fmul_rn((float)acc, __fmul_rn(sm.qs[r], ksv)), p.sm_scale);
        sm.S[r][kt] = tabs < sm.Lr[r] ? s : -INFINITY;
      }
    }
    __syncthreads();

    // ---- online softmax per row (one warp per row)
    for (int r = warp; r < R; r += kThreads / 32) {
      const float s0 = sm.S[r][lane], s1 = sm.S[r][lane + 32];
      const float bmax = warp_max(fmaxf(s0, s1));
      if (bmax == -INFINITY) {            // no visible key: row untouched
        sm.PT[r][lane] = 0.0f;
        sm.PT[r][lane + 32] = 0.0f;
        if (lane == 0) sm.alpha[r] = 1.0f;
        continue;
      }
      const float mold = sm.m[r];
      const float mnew = fmaxf(mold, bmax);
      const float a = exp_diff(mold, mnew);
      const float p0 = exp_diff(s0, mnew);
      const float p1 = exp_diff(s1, mnew);
      const float sum = warp_sum(__fadd_rn(p0, p1));
      sm.PT[r][lane] = __fmul_rn(round_p_fast(p0, p.p_mode), sm.vs[buf][lane]);
      sm.PT[r][lane + 32] = __fmul_rn(round_p_fast(p1, p.p_mode), sm.vs[buf][lane + 32]);
      if (lane == 0) {
        sm.alpha[r] = a;
        sm.m[r] = mnew;
        sm.l[r] = __fmaf_rn(sm.l[r], a, sum);
      }
    }
    __syncthreads();

    // ---- P.V: thread owns channel d = tid for all rows
    {
      const int d = tid;
#pragma unroll
      for (int r = 0; r < RPAD; ++r)
        if (r < R) o[r] = __fmul_rn(o[r], sm.alpha[r]);
      for (int t = 0; t < kTileBk; t += 4) {
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = (float)sm.vt[buf][swz(t + u, d)];
#pragma unroll
        for (int r = 0; r < RPAD; ++r) {
          if (r < R) {
            const float4 pw = *reinterpret_cast<const float4*>(&sm.PT[r][t]);
            o[r] = __fmaf_rn(pw.x, v[0], o[r]);
            o[r] = __fmaf_rn(pw.y, v[1], o[r]);
            o[r] = __fmaf_rn(pw.z, v[2], o[r]);
            o[r] = __fmaf_rn(pw.w, v[3], o[r]);
          }
        }
      }
    }
    __syncthreads();
  }

  // ---- finish: one split -> write o / l; else publish a partial and merge
  const int64_t out_b = (int64_t)b * p.M;
  if (nsplit == 1) {
#pragma unroll
    for (int r = 0; r < RPAD; ++r) {
      if (r < R) {
        const int j = r / g, h = kh * g + r % g;
        p.out[((out_b + j) * p.Hq + h) * kD + tid] = __fdiv_rn(o[r], sm.l[r]);
      }
    }
    return;
  }
  const size_t pstride = (size_t)R * (kD + 2);
  float* part = p.partials + (((size_t)b * p.nsplit_max + split) * p.Hkv + kh) * pstride;
#pragma unroll
  for (int r = 0; r < RPAD; ++r)
    if (r < R) part[(size_t)r * kD + tid] = o[r];
  if (tid < R) {
    part[(size_t)R * kD + tid] = sm.m[tid];
    part[(size_t)R * kD + R + tid] = sm.l[tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    unsigned int* ticket = p.tickets + (size_t)b * p.Hkv + kh;
    const unsigned int prev = atomicAdd(ticket, 1u);
    const int is_last = prev == (unsigned int)(nsplit - 1);
    if (is_last) atomicExch(ticket, 0u);   // leave the counter at zero
    sm.last = is_last;
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();

  // Merge in split order: M* = max m_s, w_s = e^(m_s - M*), out = sum w o / sum w l.
  const float* part0 = p.partials + ((size_t)b * p.nsplit_max * p.Hkv + kh) * pstride;
  const size_t sstride = (size_t)p.Hkv * pstride;
  for (int r = 0; r < R; ++r) {
    const int ns = nsplit_for(sm.Lr[r]);
    float mstar = -INFINITY;
    for (int s = 0; s < ns; ++s) mstar = fmaxf(mstar, __ldcg(part0 + s * sstride + (size_t)R * kD + r));
    float lt = 0.0f, ot = 0.0f;
    for (int s = 0; s < ns; ++s) {
      const float* ps = part0 + s * sstride;
      const float w = exp_diff(__ldcg(ps + (size_t)R * kD + r), mstar);
      lt = __fmaf_rn(w, __ldcg(ps + (size_t)R * kD + R + r), lt);
      ot = __fmaf_rn(w, __ldcg(ps + (size_t)r * kD + tid), ot);
    }
    const int j = r / g, h = kh * g + r % g;
    p.out[((out_b + j) * p.Hq + h) * kD + tid] = __fdiv_rn(ot, lt);
  }
}

template <int RPAD>
cudaError_t launch_rpad(const DecodeParams& p, cudaStream_t stream) {
  const int smem = (int)sizeof(SmemFast);
  cudaError_t e = cudaFuncSetAttribute(decode_fast_kernel<RPAD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.nsplit_max, (unsigned)p.Hkv, (unsigned)p.B);
  decode_fast_kernel<RPAD><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_fast(const DecodeParams& p, cudaStream_t stream) {
  if (p.R <= 8) return launch_rpad<8>(p, stream);
  if (p.R <= 16) return launch_rpad<16>(p, stream);
  if (p.R <= 32) return launch_rpad<32>(p, stream);
  return launch_rpad<64>(p, stream);
}

}  // namespace kattn
