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
// in parallel per chunk of 128 keys, by two producer groups on alternate
// chunks, while the consumers walk the earlier chunks' chains (thread i:
// channel i; one warp the row sum), reading each chunk's V laid out by
// channel in shared memory.
#include "device_common.cuh"

namespace kattn {
namespace {

constexpr int kChunk = 128;
constexpr int kSub = 32;                          // keys per step of the serial scan
constexpr int kProducersBar = 128;                // threads of one producer group
constexpr int kConsumersBar = 160;                // chains (128) and the row-sum warp

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
// Barrier among the threads of one group: producer group 0 (id 1), the
// consumers (id 2) or producer group 1 (id 3); 0 is __syncthreads.
__device__ __forceinline__ void group_sync(int id) {
  if (id == 2) asm volatile("bar.sync 2, %0;\n" ::"n"(kConsumersBar) : "memory");
  else asm volatile("bar.sync %0, %1;\n" ::"r"(id), "n"(kProducersBar) : "memory");
}

// Shared memory of one row's CTA.  The chunks of 128 keys alternate between
// two producer groups; group g stages its chunks' K and V rows into its own
// stage g by cp.async, one of its chunks ahead; the 16-byte pieces of a K row
// sit at piece c ^ (key & 7) so that the per-key dot products read without
// bank conflicts.  The producers then lay the chunk's V out by channel (vt: the
// offset-binary bytes v + 128 of one channel for the chunk's 128 keys, 16-key
// piece j at piece j ^ ((channel / 4) mod 8), so that both the transposing
// stores and the chain threads' 16-byte loads spread over all bank groups).
constexpr int kChainThreads = kD;                 // one per channel
constexpr int kSumThreads = 32;                   // the warp that walks the row sum
constexpr int kConsumers = kChainThreads + kSumThreads;
constexpr int kProducers = kChunk;                // one per key of a chunk, per group
constexpr int kExactThreads = kConsumers + 2 * kProducers;
constexpr int kSubs = kChunk / kSub;

struct ExactSmem {
  int8_t k[2][kChunk][kD];                        // [group]
  uint8_t v[2][kChunk][kD];                       // [group], as the cache holds them
  uint8_t vt[2][kD][kChunk];                      // [c & 1] by channel, offset binary
  float2 pv[2][kChunk];                           // per key: round_p(p), v_scale
  float2 ap[2][kChunk];                           // per key: alpha, p
  int same[2][kSubs];                             // every alpha of the 32 keys is exactly 1
  ExpfConsts c;
  uint64_t full[2];                               // chunk c's pv, ap, same, vt are ready: full[c & 1]
  uint64_t empty[2];                              // the chains are done with chunk c: empty[c & 1]
  uint64_t carried[2];                            // carried[c & 1]: carry[c & 3] holds the running
                                                  // max through chunk c
  int row[2][kChunk];                             // [group] plane rows of the stage's keys
  uint32_t q8[kD / 4];
  float red[2][kChunk / 32];                      // [group] per-warp maxima
  float carry[4];                                 // four slots: chunk c's is read at chunk c + 1
                                                  // and rewritten at chunk c + 4
  float qs;                                       // the query's int8 scale
  float lsum;                                     // the row sum, for the final division
  int ok_carry[2], ok_empty[2], ok_c;             // group-wide outcomes of bounded waits
};

// One CTA of 416 threads per query row, in three groups that overlap chunks:
//   producers, two groups of 128 threads (one per key of a chunk): group g
//     takes chunks c = g, g + 2, ...: chunk c's scores and prefix max; once the
//     running max through chunk c - 1 has come from the other group (and its
//     own through chunk c has gone back), its exps; once the consumers are
//     done with chunk c - 2, its pv, ap and V by channel -> [c & 1]; then it
//     stages chunk c + 2;
//   consumers: the chains (128 threads, one per channel) walk chunk c's o
//     chain and one warp its l chain, while the producers work on later chunks.
// Chunks are handed over through full / empty mbarriers, running maxima
// through carried; one thread of a group waits (bounded) and the group
// learns the outcome at a group barrier.
//
// Where every alpha of a run of 32 keys is exactly 1 (the running max did not
// move), the chain steps o = o * alpha + term and l = l * alpha + p are taken
// as o = o + term and l = l + p: multiplying by 1 is exact, so the bits are
// the same and each step is one rounding shorter.
__global__ void __launch_bounds__(kExactThreads, 2)
decode_exact_kernel(DecodeParams p, ExpfConsts consts) {
  extern __shared__ __align__(16) unsigned char exact_smem[];
  ExactSmem& sm = *reinterpret_cast<ExactSmem*>(exact_smem);

  const int tid = threadIdx.x;
  const bool producer = tid >= kConsumers;
  const int h = blockIdx.x % p.Hq;
  const int j = (blockIdx.x / p.Hq) % p.M;
  const int b = blockIdx.x / (p.Hq * p.M);
  const int kh = h / p.g;
  const int64_t qrow = ((int64_t)b * p.M + j) * p.Hq + h;
  float* orow = p.out + qrow * kD;

  if (!sequence_valid(p, b)) {
    if (tid < kChainThreads) orow[tid] = __int_as_float(0x7fc00000);
    if (tid == 0 && p.err_word != nullptr) atomicOr(p.err_word, KATTN_DEVERR_BAD_SEQUENCE);
    return;
  }
  const int L = p.ctx_len[b] + j;
  const int rs = sequence_row0(p, b);
  const int nchunks = (L + kChunk - 1) / kChunk;

  for (int i = tid; i < (int)(sizeof(ExpfConsts) / sizeof(double)); i += kExactThreads)
    reinterpret_cast<double*>(&sm.c)[i] = reinterpret_cast<const double*>(&consts)[i];
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      ex_mbar_init(&sm.full[s], 1);
      ex_mbar_init(&sm.empty[s], 1);
      ex_mbar_init(&sm.carried[s], 1);
    }
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
    const int grp = (tid - kConsumers) / kProducers;   // group: chunks c with c % 2 == grp
    const int gt = tid - kConsumers - grp * kProducers;   // key of the chunk
    const int lane = gt & 31, gwarp = gt >> 5;
    const int bar = grp == 0 ? 1 : 3;
    float ks_next = 0.0f, vs_next = 0.0f;
    auto stage_rows = [&](int t0) {
      const int t = t0 + gt;
      int row = -1;
      if (t < L) {
        row = p.block_table == nullptr ? rs + t : paged_row(p, b, t);
        ks_next = ksb[row];
        vs_next = vsb[row];
      }
      sm.row[grp][gt] = row;
    };
    auto issue = [&](int t0) {                    // after a group barrier publishes the rows
      const int n = min(kChunk, L - t0);
#pragma unroll
      for (int i = 0; i < kD / 16; ++i) {
        const int idx = i * kChunk + gt;
        const int u = idx >> 3, c16 = idx & 7;
        if (u < n) {
          const int64_t off = (int64_t)sm.row[grp][u] * kD + c16 * 16;
          cp_async16(&sm.k[grp][u][(c16 ^ (u & 7)) * 16], kbase + off, 16);
          cp_async16(&sm.v[grp][u][c16 * 16], vbase + off, 16);
        }
      }
      cp_async_commit();
    };
    if (grp < nchunks) {
      stage_rows(grp * kChunk);
      group_sync(bar);
      issue(grp * kChunk);
    }

    // int8 query (group 0): absmax over the 128 channels, then one IEEE
    // division each.  Both groups wait for it at the CTA's barrier 4.
    if (grp == 0) {
      const float x = p.q[qrow * kD + gt];
      float amax = warp_max(fabsf(x));
      if (lane == 0) sm.red[0][gwarp] = amax;
      group_sync(bar);
      amax = fmaxf(fmaxf(sm.red[0][0], sm.red[0][1]), fmaxf(sm.red[0][2], sm.red[0][3]));
      reinterpret_cast<int8_t*>(sm.q8)[gt] = (int8_t)quant_one(x, quant_scale(amax));
      if (gt == 0) sm.qs = quant_scale(amax);
    }
    asm volatile("bar.sync 4, %0;\n" ::"n"(2 * kProducers) : "memory");
    const float qs = sm.qs;

    for (int c = grp; c < nchunks; c += 2) {
      const int tb = c & 1, t0 = c * kChunk, t = t0 + gt;
      const bool live = t < L;
      const int n = min(kChunk, L - t0);
      const float ks_cur = ks_next, vs_cur = vs_next;
      cp_async_wait<0>();                         // this chunk's copies (own) landed
      group_sync(bar);                            // ... and the whole group's

      float s = -INFINITY;
      if (live) {
        // four partial sums (integers: any order gives the same total)
        const int4* krow = reinterpret_cast<const int4*>(sm.k[grp][gt]);
        const uint4* qw = reinterpret_cast<const uint4*>(sm.q8);
        int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
        for (int cc = 0; cc < kD / 16; ++cc) {
          const int4 kv = krow[cc ^ (gt & 7)];
          const uint4 q4 = qw[cc];
          a0 = __dp4a((int)kv.x, (int)q4.x, a0);
          a1 = __dp4a((int)kv.y, (int)q4.y, a1);
          a2 = __dp4a((int)kv.z, (int)q4.z, a2);
          a3 = __dp4a((int)kv.w, (int)q4.w, a3);
        }
        const int acc = (a0 + a1) + (a2 + a3);
        s = __fmul_rn(__fmul_rn((float)acc, __fmul_rn(qs, ks_cur)), p.sm_scale);
      }
      // Inclusive prefix max within the chunk (the running max joins below).
      float pm = s;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o2 = __shfl_up_sync(0xffffffffu, pm, off);
        if (lane >= off) pm = fmaxf(pm, o2);
      }
      if (lane == 31) sm.red[grp][gwarp] = pm;
      // The running max through chunk c - 1, from the other group.
      if (c >= 1 && gt == 0) {
        sm.ok_carry[grp] = ex_mbar_wait(&sm.carried[(c - 1) & 1], ((c - 1) >> 1) & 1);
        if (!sm.ok_carry[grp] && p.err_word != nullptr) atomicOr(p.err_word, KATTN_DEVERR_TIMEOUT);
      }
      group_sync(bar);                            // red written; the carry's outcome
      if (c >= 1 && !sm.ok_carry[grp]) break;     // the copies in flight drain below
      const float carry = c >= 1 ? sm.carry[(c - 1) & 3] : -INFINITY;
      float pw = -INFINITY;                       // maximum of the earlier warps of the chunk
      for (int w = 0; w < gwarp; ++w) pw = fmaxf(pw, sm.red[grp][w]);
      pm = fmaxf(pm, pw);
      // Running max before this key: the previous lane's inclusive max, or for
      // a warp's first lane the max of the carry and all earlier warps.
      float prev = __shfl_up_sync(0xffffffffu, pm, 1);
      if (lane == 0) prev = pw;
      prev = fmaxf(prev, carry);
      pm = fmaxf(pm, carry);
      if (gt == n - 1) {                          // the running max through chunk c
        sm.carry[c & 3] = pm;
        ex_mbar_arrive(&sm.carried[tb]);
      }
      // expf_tang(0) is exactly 1: skip the double-precision steps when the
      // running max did not move.
      float a = 1.0f, pp = 0.0f;
      if (live) {
        a = prev == pm ? 1.0f : expf_tang(__fsub_rn(prev, pm), sm.c);
        pp = s == pm ? 1.0f : expf_tang(__fsub_rn(s, pm), sm.c);
      }
      // warp gwarp holds keys 32 gwarp .. + 31: its run of alphas
      const bool same = __all_sync(0xffffffffu, a == 1.0f);
      // The consumers must be done with chunk c - 2: its vt, pv, ap buffers
      // take chunk c.
      if (c >= 2 && gt == 0) {
        sm.ok_empty[grp] = ex_mbar_wait(&sm.empty[tb], ((c - 2) >> 1) & 1);
        if (!sm.ok_empty[grp] && p.err_word != nullptr) atomicOr(p.err_word, KATTN_DEVERR_TIMEOUT);
      }
      group_sync(bar);                            // red reads done; the release's outcome
      if (c >= 2 && !sm.ok_empty[grp]) break;
      if (live) {
        sm.pv[tb][gt] = make_float2(round_p_exact(pp, p.p_mode), vs_cur);
        sm.ap[tb][gt] = make_float2(a, pp);
      }
      if (lane == 0) sm.same[tb][gwarp] = same ? 1 : 0;
      // Chunk c's V by channel: thread (kb = gwarp, g4 = lane) transposes keys
      // 32 kb .. + 31 of channels 4 g4 .. + 3, in 4 x 4 byte blocks.
      {
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 32; ++k)
          w[k] = *reinterpret_cast<const uint32_t*>(&sm.v[grp][32 * gwarp + k][4 * lane]);
        uint32_t ot[4][8];                        // [channel i][keys 4q .. 4q + 3]
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t t01 = __byte_perm(w[4 * q], w[4 * q + 1], 0x5140);
          const uint32_t t23 = __byte_perm(w[4 * q + 2], w[4 * q + 3], 0x5140);
          const uint32_t u01 = __byte_perm(w[4 * q], w[4 * q + 1], 0x7362);
          const uint32_t u23 = __byte_perm(w[4 * q + 2], w[4 * q + 3], 0x7362);
          ot[0][q] = __byte_perm(t01, t23, 0x5410) ^ 0x80808080u;
          ot[1][q] = __byte_perm(t01, t23, 0x7632) ^ 0x80808080u;
          ot[2][q] = __byte_perm(u01, u23, 0x5410) ^ 0x80808080u;
          ot[3][q] = __byte_perm(u01, u23, 0x7632) ^ 0x80808080u;
        }
        const int sw = lane & 7;                  // (channel / 4) mod 8
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int piece = (2 * gwarp + hh) ^ sw;
            *reinterpret_cast<uint4*>(&sm.vt[tb][4 * lane + i][16 * piece]) =
                make_uint4(ot[i][4 * hh], ot[i][4 * hh + 1], ot[i][4 * hh + 2], ot[i][4 * hh + 3]);
          }
      }
      group_sync(bar);                            // chunk c published; stage grp read
      if (gt == 0) ex_mbar_arrive(&sm.full[tb]);
      // Stage this group's next chunk, c + 2, into its stage.
      if (c + 2 < nchunks) {
        stage_rows(t0 + 2 * kChunk);
        group_sync(bar);
        issue(t0 + 2 * kChunk);
      }
    }
    cp_async_wait<0>();
    return;
  }

  // -------------------------------------------------------------- consumers
  const bool chain = tid < kChainThreads;         // else the row-sum warp
  const int ch = tid;                             // chains: the channel
  const int sw = (ch >> 2) & 7;
  float acc = 0.0f;                               // o (chains) or l (row-sum warp)
  bool ok = true;
  for (int c = 0; c < nchunks; ++c) {
    const int tb = c & 1, n = min(kChunk, L - c * kChunk);
    if (tid == 0) {
      sm.ok_c = ex_mbar_wait(&sm.full[tb], (c >> 1) & 1);
      if (!sm.ok_c && p.err_word != nullptr) atomicOr(p.err_word, KATTN_DEVERR_TIMEOUT);
    }
    group_sync(2);
    if (!sm.ok_c) {
      ok = false;
      break;
    }
    const float2* pvb = sm.pv[tb];
    const float2* apb = sm.ap[tb];
    for (int sb = 0; sb * kSub < n; ++sb) {
      const int u0 = sb * kSub;
      const bool full_run = u0 + kSub <= n;
      const bool same = sm.same[tb][sb] != 0;
      if (chain) {
        // this channel's 32 bytes: keys u0 .. u0 + 31, byte i of word i / 4
        const uint4 va = *reinterpret_cast<const uint4*>(&sm.vt[tb][ch][16 * ((2 * sb) ^ sw)]);
        const uint4 vb = *reinterpret_cast<const uint4*>(&sm.vt[tb][ch][16 * ((2 * sb + 1) ^ sw)]);
        const uint32_t vw[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
        // every key's term round_p(p) * (f32(v8) * vs) first (independent of
        // one another): the offset-binary byte u in the low mantissa bits of
        // 1.5 * 2^23 gives 12582912 + u, minus 12582912 + 128 leaves v exactly
        float term[kSub];
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
          const float2 pvv = pvb[u0 + i];
          const float vf = __fsub_rn(__uint_as_float(__byte_perm(vw[i >> 2], 0x4B400000u, 0x7640u | (i & 3))),
                                     12583040.0f);
          term[i] = __fmul_rn(pvv.x, __fmul_rn(vf, pvv.y));
        }
        if (full_run && same) {
#pragma unroll
          for (int i = 0; i < kSub; ++i) acc = __fadd_rn(acc, term[i]);
        } else if (full_run) {
#pragma unroll
          for (int i = 0; i < kSub; ++i) acc = __fadd_rn(__fmul_rn(acc, apb[u0 + i].x), term[i]);
        } else {
#pragma unroll
          for (int i = 0; i < kSub; ++i)
            if (u0 + i < n) acc = __fadd_rn(__fmul_rn(acc, apb[u0 + i].x), term[i]);
        }
      } else {
        if (full_run && same) {
#pragma unroll
          for (int i = 0; i < kSub; ++i) acc = __fadd_rn(acc, apb[u0 + i].y);
        } else if (full_run) {
#pragma unroll
          for (int i = 0; i < kSub; ++i) {
            const float2 x2 = apb[u0 + i];
            acc = __fadd_rn(__fmul_rn(acc, x2.x), x2.y);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kSub; ++i)
            if (u0 + i < n) {
              const float2 x2 = apb[u0 + i];
              acc = __fadd_rn(__fmul_rn(acc, x2.x), x2.y);
            }
        }
      }
    }
    group_sync(2);                                // every chain is done with chunk c
    if (tid == 0) ex_mbar_arrive(&sm.empty[tb]);
  }
  if (tid == kChainThreads) sm.lsum = acc;
  group_sync(2);
  if (chain) orow[ch] = ok ? __fdiv_rn(acc, sm.lsum) : __int_as_float(0x7fc00000);
}

}  // namespace

cudaError_t launch_decode_exact(const DecodeParams& p, const ExpfConsts& c,
                                cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.M * p.Hq;
  const int smem = (int)sizeof(ExactSmem);
  cudaError_t e = cudaFuncSetAttribute(decode_exact_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  decode_exact_kernel<<<(unsigned)rows, kExactThreads, smem, stream>>>(p, c);
  return cudaGetLastError();
}

}  // namespace kattn
