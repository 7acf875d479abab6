// exact_mode decode: the sequential online-softmax scan of "Kestrel_VLLM - 18"
// §3.3, reproduced operation for operation.
//
// Per query row, one token at a time in token order, each float32 operation
// rounded on its own (this file is compiled with --fmad=false and spells the
// operations with __f*_rn intrinsics):
//   vdeq = f32(v8) * vs;  m' = max(m, s);  a = expf_tang(m - m');
//   p = expf_tang(s - m');  l = l*a + p;  o_i = o_i*a + round_p(p)*vdeq_i
// and finally out_i = o_i / l.
//
// Only the l and o chains are inherently serial.  The scores, the running
// max (a prefix max, which is exact in any order) and every exp are computed
// in parallel per chunk of 128 keys by one group of threads, while a second
// group walks the previous chunk's chains (thread i: channel i), reading the
// chunk's V rows from shared memory.
#include "device_common.cuh"

namespace kattn {
namespace {

constexpr int kChunk = 128;
constexpr int kSub = 32;                          // keys per step of the serial scan

// f32 of a signed byte, exactly: the offset-binary byte u = v + 128 placed in
// the low mantissa bits of 1.5 * 2^23 gives 12582912 + u; subtracting
// 12582912 + 128 leaves v (both operands and the difference are integers
// below 2^24, so nothing rounds).
__device__ __forceinline__ float i8_to_f32(uint8_t byte) {
  const uint32_t u = (uint32_t)(byte ^ 0x80u);
  return __fsub_rn(__uint_as_float(0x4B400000u | u), 12583040.0f);
}

// Table-driven float32 exp (P. T. P. Tang, ACM TOMS 1989; the variant the
// page describes in §3.3): x = (64m + j + r/C2)/K, exp(x) = 2^m 2^(j/64) e^r,
// e^r - 1 ~ r + r^2/2 + r^3/6 evaluated with double fused multiply-adds, one
// rounding to float at the end.
__device__ __forceinline__ float expf_tang(float xf, const ExpfConsts& c) {
  if (xf > 88.7228394f) return __double2float_rn(exp((double)xf));  // overflow side
  if (xf < -104.0f) return 0.0f;                                   // deep underflow
  const double x = (double)xf;
  const int n = __double2int_rn(__dmul_rn(x, c.K));   // nearest, ties to even
  const double r = __fma_rn(-(double)n, c.C2, x);     // reduced argument
  const int m = n >> 6;                               // floor(n / 64)
  const double tj = c.T[n & 63];
  const double r2 = __dmul_rn(r, r);
  const double poly = __fma_rn(__fma_rn(r, c.C0, c.C1), r2, r);   // r + r^2/2 + r^3/6
  const double mant = __fma_rn(tj, poly, tj);                      // 2^(j/64) e^r
  const double two_m = __longlong_as_double((long long)(m + 1023) << 52);
  return __double2float_rn(__dmul_rn(two_m, mant));
}

__device__ __forceinline__ float round_p_exact(float p, int mode) {
  switch (mode) {
    case KATTN_P_BF16: return bf16_round(p);
    case KATTN_P_E4M3: return e4m3_round(p);
    case KATTN_P_E4M3_X448: return __fdiv_rn(e4m3_round(__fmul_rn(p, 448.0f)), 448.0f);
    case KATTN_P_E4M3_X256: return __fmul_rn(e4m3_round(__fmul_rn(p, 256.0f)), 1.0f / 256.0f);
    default: return p;
  }
}

// ------------------------------------------------------------ sync helpers
// Bounded waits: after this many polls a hand-off wait gives up, the row is
// NaN and KATTN_DEVERR_TIMEOUT is set.  The library is built with the default;
// a test-only build of this file (build.py, build_exact_timeout_variant) sets
// it to 0 so that every wait runs out at once and the give-up path is
// exercised without any wait that could block.
#ifndef KATTN_EXACT_SPIN_LIMIT
#define KATTN_EXACT_SPIN_LIMIT (1u << 22)
#endif
constexpr uint32_t kExactSpin = KATTN_EXACT_SPIN_LIMIT;

__device__ __forceinline__ void ex_mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void ex_mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ bool ex_mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t it = 0; it < kExactSpin; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    if (ok) return true;
  }
  return false;
}
// Barrier among the 128 threads of one group (ids 1 and 2; 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int id) {
  asm volatile("bar.sync %0, 128;\n" ::"r"(id) : "memory");
}

// Shared memory of one row's CTA.  A chunk's K and V rows are staged by
// cp.async one chunk ahead (three stages); the 16-byte pieces of a K row sit at
// piece c ^ (key & 7) so that the per-key dot products read without bank
// conflicts.  tok holds, per key of a stage: round_p(p), v_scale, alpha, p.
constexpr int kStages = 3;                        // K/V stages: the chains may be a chunk behind

struct ExactSmem {
  int8_t k[kStages][kChunk][kD];
  int8_t v[kStages][kChunk][kD];
  float4 tok[2][kChunk];
  ExpfConsts c;
  uint64_t full[2];                               // chunk c's tok (and V) are ready: full[c & 1]
  uint64_t empty[2];                              // the chains are done with chunk c: empty[c & 1]
  int row[kStages][kChunk];                       // plane rows of the stage's keys
  uint32_t q8[kD / 4];
  float red[kChunk / 32];
  float carry;
  int ok_p, ok_c;                                 // group-wide outcome of a bounded wait
};

// One CTA of 256 threads per query row, in two groups that overlap chunks:
//   producers (threads 128..255, one per key of a chunk): stage chunk c + 1,
//     then chunk c's scores, prefix max and exps -> tok[c & 1];
//   chains (threads 0..127, one per channel): walk chunk c's o and l chains
//     while the producers work on chunk c + 1.
// A stage is handed over through full / empty mbarriers; one thread of each
// group waits (bounded) and the group learns the outcome at a group barrier.
__global__ void __launch_bounds__(2 * kChunk)
decode_exact_kernel(DecodeParams p, ExpfConsts consts) {
  extern __shared__ __align__(16) unsigned char exact_smem[];
  ExactSmem& sm = *reinterpret_cast<ExactSmem*>(exact_smem);

  const int tid = threadIdx.x;
  const bool producer = tid >= kChunk;
  const int gt = producer ? tid - kChunk : tid;   // key (producers) or channel (chains)
  const int lane = gt & 31, gwarp = gt >> 5;
  const int h = blockIdx.x % p.Hq;
  const int j = (blockIdx.x / p.Hq) % p.M;
  const int b = blockIdx.x / (p.Hq * p.M);
  const int kh = h / p.g;
  const int64_t qrow = ((int64_t)b * p.M + j) * p.Hq + h;
  float* orow = p.out + qrow * kD;

  if (!sequence_valid(p, b)) {
    if (!producer) orow[gt] = __int_as_float(0x7fc00000);
    if (tid == 0 && p.err_word != nullptr) atomicOr(p.err_word, KATTN_DEVERR_BAD_SEQUENCE);
    return;
  }
  const int L = p.ctx_len[b] + j;
  const int rs = sequence_row0(p, b);
  const int nchunks = (L + kChunk - 1) / kChunk;

  for (int i = tid; i < (int)(sizeof(ExpfConsts) / sizeof(double)); i += 2 * kChunk)
    reinterpret_cast<double*>(&sm.c)[i] = reinterpret_cast<const double*>(&consts)[i];
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      ex_mbar_init(&sm.full[s], 1);
      ex_mbar_init(&sm.empty[s], 1);
    }
    sm.carry = -INFINITY;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  // Key t is row `row` of head kh's plane: rs + t, or from the block table.
  const int64_t plane = (int64_t)kh * p.cap_rows;
  const int8_t* kbase = p.k + plane * kD;
  const int8_t* vbase = p.v + plane * kD;
  const float* ksb = p.k_scale + plane;
  const float* vsb = p.v_scale + plane;

  if (producer) {
    // ---------------------------------------------------------- producers
    float ks_next = 0.0f, vs_next = 0.0f;
    auto stage_rows = [&](int t0, int st) {
      const int t = t0 + gt;
      int row = -1;
      if (t < L) {
        row = p.block_table == nullptr ? rs + t : paged_row(p, b, t);
        ks_next = ksb[row];
        vs_next = vsb[row];
      }
      sm.row[st][gt] = row;
    };
    auto issue = [&](int t0, int st) {            // after a group barrier publishes the rows
      const int n = min(kChunk, L - t0);
#pragma unroll
      for (int i = 0; i < kD / 16; ++i) {
        const int idx = i * kChunk + gt;
        const int u = idx >> 3, c16 = idx & 7;
        if (u < n) {
          const int64_t off = (int64_t)sm.row[st][u] * kD + c16 * 16;
          cp_async16(&sm.k[st][u][(c16 ^ (u & 7)) * 16], kbase + off, 16);
          cp_async16(&sm.v[st][u][c16 * 16], vbase + off, 16);
        }
      }
      cp_async_commit();
    };
    stage_rows(0, 0);
    group_sync(1);
    issue(0, 0);

    // int8 query: absmax over the 128 channels, then one IEEE division each.
    const float x = p.q[qrow * kD + gt];
    float amax = warp_max(fabsf(x));
    if (lane == 0) sm.red[gwarp] = amax;
    group_sync(1);
    amax = fmaxf(fmaxf(sm.red[0], sm.red[1]), fmaxf(sm.red[2], sm.red[3]));
    const float qs = quant_scale(amax);
    reinterpret_cast<int8_t*>(sm.q8)[gt] = (int8_t)quant_one(x, qs);
    group_sync(1);                                // q8 complete; red free again

    for (int c = 0; c < nchunks; ++c) {
      const int st = c % kStages, tb = c & 1, t0 = c * kChunk, t = t0 + gt;
      const bool live = t < L;
      const int n = min(kChunk, L - t0);
      const float ks_cur = ks_next, vs_cur = vs_next;
      // The chains must be done with chunk c - 2: its K/V stage takes chunk
      // c + 1 now, and its tok buffer takes chunk c.
      if (c >= 2) {
        if (gt == 0) {
          sm.ok_p = ex_mbar_wait(&sm.empty[tb], ((c - 2) >> 1) & 1);
          if (!sm.ok_p && p.err_word != nullptr) atomicOr(p.err_word, KATTN_DEVERR_TIMEOUT);
        }
        group_sync(1);
        if (!sm.ok_p) break;                      // the copies in flight drain below
      }
      if (c + 1 < nchunks) {
        stage_rows(t0 + kChunk, (c + 1) % kStages);
        group_sync(1);
        issue(t0 + kChunk, (c + 1) % kStages);
      } else {
        cp_async_commit();                        // an empty group keeps the count
      }
      cp_async_wait<1>();                         // this chunk's copies (own) landed
      group_sync(1);                              // ... and the whole group's

      float s = -INFINITY;
      if (live) {
        const int4* krow = reinterpret_cast<const int4*>(sm.k[st][gt]);
        int acc = 0;
#pragma unroll
        for (int cc = 0; cc < kD / 16; ++cc) {
          const int4 kv = krow[cc ^ (gt & 7)];
          acc = __dp4a((int)kv.x, (int)sm.q8[4 * cc + 0], acc);
          acc = __dp4a((int)kv.y, (int)sm.q8[4 * cc + 1], acc);
          acc = __dp4a((int)kv.z, (int)sm.q8[4 * cc + 2], acc);
          acc = __dp4a((int)kv.w, (int)sm.q8[4 * cc + 3], acc);
        }
        s = __fmul_rn(__fmul_rn((float)acc, __fmul_rn(qs, ks_cur)), p.sm_scale);
      }
      // Inclusive prefix max over the chunk, seeded with the running max.
      float pm = s;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o2 = __shfl_up_sync(0xffffffffu, pm, off);
        if (lane >= off) pm = fmaxf(pm, o2);
      }
      if (lane == 31) sm.red[gwarp] = pm;
      const float carry = sm.carry;
      group_sync(1);
      for (int w = 0; w < gwarp; ++w) pm = fmaxf(pm, sm.red[w]);
      pm = fmaxf(pm, carry);
      // Running max before this key: the previous lane's inclusive max, or for
      // a warp's first lane the max of the carry and all earlier warps.
      float prev = __shfl_up_sync(0xffffffffu, pm, 1);
      if (lane == 0) {
        float pw = carry;
        for (int w = 0; w < gwarp; ++w) pw = fmaxf(pw, sm.red[w]);
        prev = pw;
      }
      if (live) {
        // expf_tang(0) is exactly 1: skip the double-precision steps when the
        // running max did not move.
        const float a = prev == pm ? 1.0f : expf_tang(__fsub_rn(prev, pm), sm.c);
        const float pp = s == pm ? 1.0f : expf_tang(__fsub_rn(s, pm), sm.c);
        sm.tok[tb][gt] = make_float4(round_p_exact(pp, p.p_mode), vs_cur, a, pp);
      }
      group_sync(1);                              // tok complete; red and carry reads done
      if (gt == n - 1) sm.carry = pm;
      if (gt == 0) ex_mbar_arrive(&sm.full[tb]);
    }
    cp_async_wait<0>();
    return;
  }

  // ---------------------------------------------------------------- chains
  float o = 0.0f, l = 0.0f;
  bool ok = true;
  for (int c = 0; c < nchunks; ++c) {
    const int st = c % kStages, tb = c & 1, n = min(kChunk, L - c * kChunk);
    if (gt == 0) {
      sm.ok_c = ex_mbar_wait(&sm.full[tb], (c >> 1) & 1);
      if (!sm.ok_c && p.err_word != nullptr) atomicOr(p.err_word, KATTN_DEVERR_TIMEOUT);
    }
    group_sync(2);
    if (!sm.ok_c) {
      ok = false;
      break;
    }
    // 32 keys at a time: first every key's term round_p(p) * (f32(v8) * vs)
    // (independent of one another), then the two chains, key by key.
    const uint8_t* vcol = reinterpret_cast<const uint8_t*>(&sm.v[st][0][gt]);
    const float2* tk2 = reinterpret_cast<const float2*>(sm.tok[tb]);
    for (int u0 = 0; u0 < n; u0 += kSub) {
      float term[kSub];
#pragma unroll
      for (int i = 0; i < kSub; ++i) {
        const float2 pv = tk2[2 * (u0 + i)];      // round_p(p), v_scale
        term[i] = __fmul_rn(pv.x, __fmul_rn(i8_to_f32(vcol[(u0 + i) * kD]), pv.y));
      }
      if (u0 + kSub <= n) {
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
          const float2 ap = tk2[2 * (u0 + i) + 1];   // alpha, p
          o = __fadd_rn(__fmul_rn(o, ap.x), term[i]);
          l = __fadd_rn(__fmul_rn(l, ap.x), ap.y);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
          if (u0 + i < n) {
            const float2 ap = tk2[2 * (u0 + i) + 1];
            o = __fadd_rn(__fmul_rn(o, ap.x), term[i]);
            l = __fadd_rn(__fmul_rn(l, ap.x), ap.y);
          }
        }
      }
    }
    group_sync(2);                                // every chain is done with chunk c
    if (gt == 0) ex_mbar_arrive(&sm.empty[tb]);
  }
  orow[gt] = ok ? __fdiv_rn(o, l) : __int_as_float(0x7fc00000);
}

}  // namespace

cudaError_t launch_decode_exact(const DecodeParams& p, const ExpfConsts& c,
                                cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.M * p.Hq;
  const int smem = (int)sizeof(ExactSmem);
  cudaError_t e = cudaFuncSetAttribute(decode_exact_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  decode_exact_kernel<<<(unsigned)rows, 2 * kChunk, smem, stream>>>(p, c);
  return cudaGetLastError();
}

}  // namespace kattn
