// The split-KV pass for 17..32 query rows per (sequence, kv head) with warps
// that own spans and P.V on the fifth-generation tensor cores.
//
// Each row gets the arithmetic of the M = 1 kernel (decode_split.cuh) in the
// same order -- the int8 QK on mma.sync, the same online softmax per 32-key
// block with the maximum reset at every 128-key span, the same P.V operands
// (V exact in f16, a = round_p(p) * v_scale * 2^E split into f16 hi + lo) and
// the same order of 16-key MMA steps per span (hi then lo of the first half
// of a block, then of the second) -- so every row equals the M = 1 kernel's
// bytes and batch invariance holds.  tcgen05 kind::f16 with an f32
// accumulator adds such a step exactly as mma.sync m16n8k16 does.
//
// Layout.  One CTA of 8 warps per work item (sequence, 512-key window, kv
// head), persistent over the work list, 2 CTAs per SM.  Warp w reduces span
// kw = w % 4 of the window for the rows of its group grp = w / 4 (rows
// 16 grp .. 16 grp + 15, two 8-row n-tiles), one 32-key block at a time, as
// the M = 1 kernel does for its 8 rows; so the per-key work that does not
// depend on the rows (K and V loads, the V conversion, waits and loop
// control) is shared by 16 rows instead of 8.  The 4 spans advance together
// in steps: step i is block i of every span.  Per step:
//   * each warp computes its rows' scores (int8 MMA), softmax and P operand
//     words, and converts half of its span's V block (16 keys, 128 channels)
//     into the transposed f16 operand;
//   * the accumulators D_s[d][row] (span s, tensor-memory lanes = channels,
//     columns 32 s .. 32 s + 31 = rows) of rows whose running max moved are
//     rescaled by alpha -- by all 8 warps, since a warp reaches only its own
//     quarter of the lanes (warps q and q + 4 split the spans);
//   * one thread issues the step's MMAs, four per span
//       D_s += Vt_s[d][key] * P_s[row][key]   (M = 128, N = 32, K = 16)
//     and commits them to an mbarrier that the next step's operand writes
//     wait on.
// K blocks stream through a 2-stage TMA ring per span and V blocks through a
// 1-stage ring per span (a V block is converted as soon as it is read, which
// frees its stage early).  At the window's end the spans are merged per row in
// the M = 1 kernel's order.  PG: the paged cache, block rows from the table.
#include "tcgen05_common.cuh"

namespace kattn {
namespace {

constexpr int kWRows = 32;                          // rows per CTA (R in 17..32)
constexpr int kWGroups = 2;                         // warp groups over the rows
constexpr int kWNR = kWRows / 8 / kWGroups;         // 8-row n-tiles per warp: 2
constexpr int kWWarps = kSpansPerCta * kWGroups;    // 8
constexpr int kWThreads = 32 * kWWarps;
constexpr int kWStages = 2;                         // K stages per span
constexpr int kWCols = kSpansPerCta * kWRows;       // tensor-memory columns: 128
constexpr int kWCtasPerSm = 2;                      // shared memory and registers
static_assert(kWRows == kTcN, "the instruction descriptor's N");
static_assert(kWNR == 2 && kWGroups == 2, "a group converts one 16-key half of a V block");

struct __align__(1024) TcwSmem {
  uint8_t kring[kSpansPerCta][kWStages][kBlockBytes];   // K blocks (TMA, 128-byte swizzle)
  uint8_t vring[kSpansPerCta][kBlockBytes];             // the span's next V block (same)
  // MMA operands of the step in flight (no swizzle, K-major, 16 keys per
  // half; element (row, key) at op_off(row, key)).
  uint8_t vt[kSpansPerCta][2][128 * 16 * 2];            // [span][half] V transposed
  uint8_t pb[kSpansPerCta][2][2][kWRows * 16 * 2];      // [span][half][hi | lo] P
  uint8_t qbuf[kWRows * (kD + 4)];                      // the item's int8 rows, then scales
  uint64_t kfull[kSpansPerCta][kWStages], kempty[kSpansPerCta][kWStages];
  uint64_t vfull[kSpansPerCta], vempty[kSpansPerCta];
  uint64_t qbar, mbar;
  __align__(16) float alpha[kSpansPerCta][kWRows];      // the step's alpha per span and row
  // a row's max moved this step, by step parity: a warp may write step
  // i + 1's flags while a slower one still reads step i's
  int moved[2][kSpansPerCta][kWGroups];
  float wm[kSpansPerCta][kWRows], wl[kSpansPerCta][kWRows], wd[kSpansPerCta][kWRows];
  int brow[kSpansPerCta][2][kSpanC / kBlockBk];         // paged: block rows, by item parity
  float scale[2][kSpansPerCta][2][kSpanC];              // [item parity][span][k | v] scales
  Item item[2];                                         // the current and next items, by parity
  int fail[kWWarps];                                    // a wait ran out (per warp)
  uint32_t tmem;
};

template <int PM, bool PG>
__global__ void __launch_bounds__(kWThreads, kWCtasPerSm)
decode_tcw_kernel(const DecodeParams p, const __grid_constant__ TmaMaps maps) {
  extern __shared__ unsigned char smem_raw[];
  TcwSmem& sm = *reinterpret_cast<TcwSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t kQBytes = kWRows * (kD + 4);
  constexpr int NR = kWNR;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kw = warp % kSpansPerCta, grp = warp / kSpansPerCta;
  const int g = lane >> 2, c = lane & 3;
  const int gq = p.g, M = p.M, R = p.R;
  const int row0 = 16 * grp;                      // the warp's first row
  const bool producer = grp == 0;                 // warp kw of group 0 fills span kw's rings
  const uint32_t tlane = (uint32_t)(32 * kw) << 16;   // the tensor-memory lanes this warp reaches
  int jrow[NR][2];
#pragma unroll
  for (int nr = 0; nr < NR; ++nr)
#pragma unroll
    for (int e = 0; e < 2; ++e) jrow[nr][e] = min((row0 + 8 * nr + 2 * c + e) / gq, M - 1);

  const int G = gridDim.x;
  int t = blockIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kSpansPerCta; ++s) {
      for (int st = 0; st < kWStages; ++st) {
        mbar_init(&sm.kfull[s][st], 1);
        mbar_init(&sm.kempty[s][st], kWGroups);
      }
      mbar_init(&sm.vfull[s], 1);
      mbar_init(&sm.vempty[s], kWGroups);
    }
    mbar_init(&sm.qbar, 1);
    mbar_init(&sm.mbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (lane == 0) sm.fail[warp] = 0;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                 ::"r"(smem_u32(&sm.tmem)), "r"(kWCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  griddep_wait();                                 // the work list and the packed queries
  griddep_launch_dependents();
  const int total = (int)__ldcg(p.item_count);
  // The item descriptors live in shared memory, slot = item parity: the
  // current item's and the next one's (thread 0 loads them).
  if (tid == 0) {
    sm.item[0] = load_item(p, t, total);
    sm.item[1] = load_item(p, t + G, total);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const uint64_t kv_policy = l2_evict_first();
  int par = 0;                                    // parity of the current item
  Item it0 = sm.item[0];

  bool q_pending = false;                         // thread 0: a query copy in flight
  auto fetch_queries = [&](const Item& it) {      // thread 0
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    mbar_expect_tx(&sm.qbar, kQBytes);
    bulk_load(sm.qbuf, p.qpack + ((size_t)it.b * p.Hkv + it.kh) * qpack_bytes(p.rpad), kQBytes,
              &sm.qbar);
    q_pending = true;
  };
  if (tid == 0 && it0.b >= 0) fetch_queries(it0);

  // ---- per span (warp kw of group 0): the block rows of an item (paged) and
  // its k and v scales, into the item's parity slot.  Scales go by cp.async,
  // zero past the span's keys; the warp waits for them before the item.
  auto block_rows = [&](const Item& it, int slot) {
    if constexpr (PG) {
      if (producer && it.b >= 0) {
        const Span s = span_of(it, kw, M);
        if (lane < s.nb) sm.brow[kw][slot][lane] = it.row + paged_row(p, it.b, s.s0 + lane * kBlockBk);
        __syncwarp();
      }
    }
  };
  auto fetch_scales = [&](const Item& it, int slot) {
    if (!producer) return;
    const Span s = span_of(it, kw, M);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = s.s0 + lane + 32 * e;
      const bool in = it.b >= 0 && key < s.s1;
      int row = 0;
      if (in) row = PG ? sm.brow[kw][slot][(key - s.s0) >> 5] + (key & 31) : it.row + key;
      cp_async4(&sm.scale[slot][kw][0][lane + 32 * e], p.k_scale + row, in ? 4 : 0);
      cp_async4(&sm.scale[slot][kw][1][lane + 32 * e], p.v_scale + row, in ? 4 : 0);
    }
    cp_async_commit();
  };
  block_rows(it0, 0);
  fetch_scales(it0, 0);
  block_rows(sm.item[1], 1);
  fetch_scales(sm.item[1], 1);

  // ---- producer of span kw (lane 0 issues, every lane keeps the counters).
  // The K cursor runs up to kWStages blocks ahead and the V cursor one block
  // ahead, each over this item's blocks, then the next item's.
  struct Cursor {
    int row, nb, item, blk, st, inflight;
    uint32_t used, eph;                           // stages filled before; their empty parities
  };
  Cursor kc{0, 0, 0, 0, 0, 0, 0u, 0u};
  {
    const Span s0 = span_of(it0, kw, M);
    kc.row = s0.row;
    kc.nb = it0.b >= 0 ? s0.nb : 0;
  }
  Cursor vc = kc;
  // Issue the copies the ring has room for; false if a stage was never released.
  auto produce = [&](Cursor& cu, int stages, uint64_t* full, uint64_t* empty, bool is_k) -> bool {
    if (!producer) return true;
    while (cu.inflight < stages) {
      if (cu.blk < cu.nb) {
        if ((cu.used >> cu.st) & 1u) {            // every group has read the stage
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[cu.st], (cu.eph >> cu.st) & 1u)))
            return false;
          cu.eph ^= 1u << cu.st;
        }
        cu.used |= 1u << cu.st;
        if (lane == 0) {
          const int row = PG ? sm.brow[kw][par ^ cu.item][cu.blk] : cu.row + cu.blk * kBlockBk;
          asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
          mbar_expect_tx(&full[cu.st], kBlockBytes);
          if (is_k) tma_load_block(sm.kring[kw][cu.st], &maps.k, row, &full[cu.st], kv_policy);
          else tma_load_block(sm.vring[kw], &maps.v, row, &full[cu.st], kv_policy);
        }
        ++cu.blk;
        ++cu.inflight;
        cu.st = cu.st + 1 == stages ? 0 : cu.st + 1;
      } else if (cu.item == 0) {
        const Item nx = sm.item[par ^ 1];
        if (nx.b < 0) break;
        const Span s1 = span_of(nx, kw, M);
        cu.item = 1;
        cu.blk = 0;
        cu.row = s1.row;
        cu.nb = s1.nb;
      } else {
        break;
      }
    }
    return true;
  };
  auto produce_k = [&]() { return produce(kc, kWStages, sm.kfull[kw], sm.kempty[kw], true); };
  auto produce_v = [&]() { return produce(vc, 1, &sm.vfull[kw], &sm.vempty[kw], false); };
  bool ok = produce_k() && produce_v();

  int kcst = 0, vph = 0;                          // consumer: K stage; V parity
  uint32_t kcph = 0, qph = 0;
  int commits = 0, waited = 0;                    // MMA groups committed / waited for
  bool failed = false;

  while (it0.b >= 0 && !failed) {
    const int ctx = it0.ctx;
    const Span sp = span_of(it0, kw, M);
    // every span's accumulator starts at +0: warps q and q + 4 split the spans
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      float z[32];
#pragma unroll
      for (int x = 0; x < 32; ++x) z[x] = 0.0f;
      tc_st32(tmem + tlane + 32 * (2 * grp + s2), z);
    }
    if (producer) cp_async_wait<1>();             // this item's scales (the next item's may fly)
    const bool q_ok = __all_sync(0xffffffffu, mbar_wait_bounded(&sm.qbar, qph));
    if (tid == 0 && q_ok) q_pending = false;
    if (__syncthreads_or(!q_ok || !ok)) {         // also: the scales are visible to all
      failed = true;
      break;
    }
    const float* ksc = sm.scale[par][kw][0];
    const float* vsc = sm.scale[par][kw][1];
    uint32_t qw8[NR][8];
    float qs_row[NR][2];
    {
      const float* qsb = reinterpret_cast<const float*>(&sm.qbuf[kWRows * kD]);
#pragma unroll
      for (int nr = 0; nr < NR; ++nr) {
        const uint4* src = reinterpret_cast<const uint4*>(&sm.qbuf[(row0 + 8 * nr + g) * kD + 32 * c]);
        const uint4 lo = src[0], hi = src[1];
        qw8[nr][0] = lo.x; qw8[nr][1] = lo.y; qw8[nr][2] = lo.z; qw8[nr][3] = lo.w;
        qw8[nr][4] = hi.x; qw8[nr][5] = hi.y; qw8[nr][6] = hi.z; qw8[nr][7] = hi.w;
        qs_row[nr][0] = qsb[row0 + 8 * nr + 2 * c];
        qs_row[nr][1] = qsb[row0 + 8 * nr + 2 * c + 1];
      }
    }
    // 2^E per row from the largest v_scale among the span's keys the row sees
    // (key k of the span at index k - s0 of the scale slot)
    float up_row[NR][2], down_row[NR][2];
    {
      const int kc2 = min(sp.s1, ctx);
      float vm = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (sp.s0 + lane + 32 * e < kc2) vm = fmaxf(vm, vsc[lane + 32 * e]);
      vm = warp_max(vm);
#pragma unroll
      for (int nr = 0; nr < NR; ++nr)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float vmax = vm;                        // the draft keys ctx + q, q < j, in the span
          for (int q = 0; q < jrow[nr][e]; ++q) {
            const int rel = ctx + q - sp.s0;
            if (rel >= 0 && ctx + q < sp.s1) vmax = fmaxf(vmax, vsc[rel]);
          }
          const int bexp = min(max(268 - (int)((__float_as_uint(vmax) >> 23) & 0xffu), 1), 253);
          up_row[nr][e] = __uint_as_float((uint32_t)bexp << 23);
          down_row[nr][e] = __uint_as_float((uint32_t)(254 - bexp) << 23);
        }
    }
    float m_run[NR][2], l_run[NR][2];
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        m_run[nr][e] = -INFINITY;
        l_run[nr][e] = 0.0f;
      }

    const int nsteps = span_of(it0, 0, M).nb;     // span 0 has the most blocks
    for (int i = 0; i < nsteps; ++i) {
      const bool act = i < sp.nb;                 // this warp's span has block i
      bool rescale = false;
      bool wok = true;
      float alpha[NR][2];
      uint32_t ph[2][NR][2], pl[2][NR][2];        // P operand words [half][n-tile][k pair]
      if (act) {
        const int t0 = sp.s0 + i * kBlockBk;
        // ---- QK of the warp's rows on the int8 MMA (scores as in the M = 1 kernel)
        wok = __all_sync(0xffffffffu, mbar_wait_bounded(&sm.kfull[kw][kcst], kcph));
        float sc[2][NR][4];
        {
          const uint8_t* Kt = sm.kring[kw][kcst];
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int ra = 16 * hf + g, rb = ra + 8;
            const uint4 a_lo = lds128(Kt + swz(ra, 2 * c)), a_hi = lds128(Kt + swz(ra, 2 * c + 1));
            const uint4 b_lo = lds128(Kt + swz(rb, 2 * c)), b_hi = lds128(Kt + swz(rb, 2 * c + 1));
            const uint32_t wa[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
            const uint32_t wb[8] = {b_lo.x, b_lo.y, b_lo.z, b_lo.w, b_hi.x, b_hi.y, b_hi.z, b_hi.w};
#pragma unroll
            for (int nr = 0; nr < NR; ++nr) {
              int iacc[4] = {0, 0, 0, 0}, iacc2[4] = {0, 0, 0, 0};
#pragma unroll
              for (int s4 = 0; s4 < 4; ++s4)
                mma_i8((s4 & 1) ? iacc2 : iacc, wa[2 * s4], wb[2 * s4], wa[2 * s4 + 1],
                       wb[2 * s4 + 1], qw8[nr][2 * s4], qw8[nr][2 * s4 + 1]);
#pragma unroll
              for (int u = 0; u < 4; ++u) sc[hf][nr][u] = __int2float_rn(iacc[u] + iacc2[u]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.kempty[kw][kcst]);   // this group is done with the stage
        if (++kcst == kWStages) {
          kcst = 0;
          kcph ^= 1u;
        }
        if (producer) --kc.inflight;
        wok = produce_k() && wok;
        // scales of keys 32i + g + 8q (q = 0..3)
        float ks4[4], vs4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          ks4[q] = ksc[32 * i + g + 8 * q];
          vs4[q] = vsc[32 * i + g + 8 * q];
        }
        // ---- scores ((S * (qs * ks)) * sm_scale), masked past each row's L
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int nr = 0; nr < NR; ++nr)
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
              const float ksv = ks4[2 * hf + k2];
              const float2 qk = f2_mul(make_float2(qs_row[nr][0], qs_row[nr][1]), make_float2(ksv, ksv));
              float2 s2 = f2_mul(make_float2(sc[hf][nr][2 * k2], sc[hf][nr][2 * k2 + 1]), qk);
              s2 = f2_mul(s2, make_float2(p.sm_scale, p.sm_scale));
              sc[hf][nr][2 * k2] = s2.x;
              sc[hf][nr][2 * k2 + 1] = s2.y;
            }
        if (t0 + kBlockBk > ctx) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int nr = 0; nr < NR; ++nr)
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int key = t0 + 16 * hf + g + 8 * (u >> 1);
                if (key >= ctx + jrow[nr][u & 1]) sc[hf][nr][u] = -INFINITY;
              }
        }
        // ---- online softmax of rows row0 + 8nr + 2c + e over the block
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
            if (mnew != -INFINITY) {
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
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              sc[hf][nr][e] = __fmul_rn(__fmul_rn(round_p_t<PM>(pk[hf][0]), vs4[2 * hf]), up_row[nr][e]);
              sc[hf][nr][2 + e] =
                  __fmul_rn(__fmul_rn(round_p_t<PM>(pk[hf][1]), vs4[2 * hf + 1]), up_row[nr][e]);
            }
          }
        // ---- P operand words: {a[key 2c][row g], a[key 2c+1][row g]} and keys
        // 2c+8, 2c+9 of each half, split into f16 hi + lo (the M = 1 kernel's
        // B fragments)
        {
          const int srcA = 8 * c + (g >> 1), srcB = srcA + 4;
          const bool odd = g & 1;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int nr = 0; nr < NR; ++nr) {
              float fA[4], fB[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                fA[u] = __shfl_sync(0xffffffffu, sc[hf][nr][u], srcA);
                fB[u] = __shfl_sync(0xffffffffu, sc[hf][nr][u], srcB);
              }
              split_f16x2(odd ? fA[1] : fA[0], odd ? fB[1] : fB[0], ph[hf][nr][0], pl[hf][nr][0]);
              split_f16x2(odd ? fA[3] : fA[2], odd ? fB[3] : fB[2], ph[hf][nr][1], pl[hf][nr][1]);
            }
        }
      }
      // ---- the previous step's MMAs read vt and pb: wait for them
      if (commits > waited) {
        const bool ok_m = __all_sync(0xffffffffu, mbar_wait_bounded(&sm.mbar, (uint32_t)(commits - 1) & 1u));
        if (ok_m) waited = commits;               // else the exit waits again
        wok = ok_m && wok;
        tc_fence_after();
      }
      if (act) {
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) {
          const int r = row0 + 8 * nr + g;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            *reinterpret_cast<uint32_t*>(sm.pb[kw][hf][0] + op_off(r, 2 * c)) = ph[hf][nr][0];
            *reinterpret_cast<uint32_t*>(sm.pb[kw][hf][0] + op_off(r, 2 * c + 8)) = ph[hf][nr][1];
            if constexpr (PM != KATTN_P_E4M3_DIRECT) {   // that mode has no low part
              *reinterpret_cast<uint32_t*>(sm.pb[kw][hf][1] + op_off(r, 2 * c)) = pl[hf][nr][0];
              *reinterpret_cast<uint32_t*>(sm.pb[kw][hf][1] + op_off(r, 2 * c + 8)) = pl[hf][nr][1];
            }
          }
          if (g == 0) {
            sm.alpha[kw][row0 + 8 * nr + 2 * c] = alpha[nr][0];
            sm.alpha[kw][row0 + 8 * nr + 2 * c + 1] = alpha[nr][1];
          }
        }
        // ---- V operand: group grp converts keys 16 grp .. 16 grp + 15 of the
        // block (its half) for all 128 channels.  Lane l takes channels 4l ..
        // 4l + 3: one 4-byte load per key row, byte permutes into key pairs, and
        // 16-byte stores into the transposed K-major operand, channel 4l +
        // ((t + l / 2) mod 4) for store t (spread over the bank groups).
        wok = __all_sync(0xffffffffu, mbar_wait_bounded(&sm.vfull[kw], (uint32_t)vph)) && wok;
        {
          const uint8_t* Vt = sm.vring[kw];
          uint8_t* vdst = sm.vt[kw][grp];
          const uint32_t x0 = (uint32_t)(lane >> 1) & 3u, x1 = (x0 + 1u) & 3u;
          const uint32_t selA = x0 | ((4u + x0) << 4) | (((x0 + 2u) & 3u) << 8) | ((4u + ((x0 + 2u) & 3u)) << 12);
          const uint32_t selB = x1 | ((4u + x1) << 4) | (((x1 + 2u) & 3u) << 8) | ((4u + ((x1 + 2u) & 3u)) << 12);
#pragma unroll
          for (int k8 = 0; k8 < 2; ++k8) {        // keys 16 grp + 8 k8 .. + 7
            uint32_t W[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              W[j] = *reinterpret_cast<const uint32_t*>(
                  Vt + swz(16 * grp + 8 * k8 + j, lane >> 2) + 4 * (lane & 3));
            uint32_t h[4][4];                       // [store t][word m]
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const uint32_t uA = __byte_perm(W[2 * m], W[2 * m + 1], selA) ^ 0x80808080u;
              const uint32_t uB = __byte_perm(W[2 * m], W[2 * m + 1], selB) ^ 0x80808080u;
              h[0][m] = i8pair_to_h2(uA, 0x4140u);
              h[2][m] = i8pair_to_h2(uA, 0x4342u);
              h[1][m] = i8pair_to_h2(uB, 0x4140u);
              h[3][m] = i8pair_to_h2(uB, 0x4342u);
            }
#pragma unroll
            for (int t4 = 0; t4 < 4; ++t4) {
              const int d = 4 * lane + ((t4 + (lane >> 1)) & 3);
              *reinterpret_cast<uint4*>(vdst + op_off(d, 8 * k8)) =
                  make_uint4(h[t4][0], h[t4][1], h[t4][2], h[t4][3]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.vempty[kw]);   // this group is done with the V block
        vph ^= 1;
        if (producer) --vc.inflight;
        wok = produce_v() && wok;
      }
      const bool mv = __any_sync(0xffffffffu, act && rescale);
      if (lane == 0) {
        sm.moved[i & 1][kw][grp] = mv ? 1 : 0;
        if (!wok) sm.fail[warp] = 1;
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      tc_fence_before();
      __syncthreads();
      {
        int any_fail = 0;                         // uniform: read after the barrier
#pragma unroll
        for (int w = 0; w < kWWarps; ++w) any_fail |= sm.fail[w];
        if (any_fail) {
          failed = true;
          break;
        }
      }
      // ---- rows whose max moved: D_s *= alpha (not at a span's first block,
      // where D_s is still +0).  Warp q + 4 grp rescales spans 2 grp, 2 grp + 1
      // on its lane quarter.
      int nb_s[kSpansPerCta];
#pragma unroll
      for (int s = 0; s < kSpansPerCta; ++s) nb_s[s] = span_of(it0, s, M).nb;
      bool need2 = false;                         // uniform: any span rescaled this step
#pragma unroll
      for (int s = 0; s < kSpansPerCta; ++s)
        need2 |= i > 0 && i < nb_s[s] && (sm.moved[i & 1][s][0] | sm.moved[i & 1][s][1]);
      if (need2) {
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const int s = 2 * grp + s2;
          if (i > 0 && i < nb_s[s] && (sm.moved[i & 1][s][0] | sm.moved[i & 1][s][1])) {
#pragma unroll
            for (int h16 = 0; h16 < 2; ++h16) {
              float v[16];
              tc_ld16(tmem + tlane + 32 * s + 16 * h16, v);
#pragma unroll
              for (int j4 = 0; j4 < 4; ++j4) {
                const float4 a4 = reinterpret_cast<const float4*>(sm.alpha[s])[4 * h16 + j4];
                v[4 * j4] = __fmul_rn(v[4 * j4], a4.x);
                v[4 * j4 + 1] = __fmul_rn(v[4 * j4 + 1], a4.y);
                v[4 * j4 + 2] = __fmul_rn(v[4 * j4 + 2], a4.z);
                v[4 * j4 + 3] = __fmul_rn(v[4 * j4 + 3], a4.w);
              }
              tc_st16(tmem + tlane + 32 * s + 16 * h16, v);
            }
          }
        }
        tc_wait_st();
        tc_fence_before();
        __syncthreads();
      }
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < kSpansPerCta; ++s) {
          if (i >= nb_s[s]) continue;
          const uint32_t dcol = tmem + 32 * s;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            tc_mma(dcol, smem_desc(sm.vt[s][hf]), smem_desc(sm.pb[s][hf][0]));
            if constexpr (PM != KATTN_P_E4M3_DIRECT)
              tc_mma(dcol, smem_desc(sm.vt[s][hf]), smem_desc(sm.pb[s][hf][1]));
          }
        }
        tc_commit(&sm.mbar);
        if (i == 0) {                             // every warp has read this item's queries
          const Item nx = sm.item[par ^ 1];
          if (nx.b >= 0) fetch_queries(nx);
        }
      }
      ++commits;
    }
    if (failed) break;

    // ---- the span's row sums and maxima (the M = 1 reduction order)
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = l_run[nr][e];
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 16));
        if (g == 0) {
          const int r = row0 + 8 * nr + 2 * c + e;
          sm.wl[kw][r] = v;
          sm.wm[kw][r] = m_run[nr][e];
          sm.wd[kw][r] = down_row[nr][e];
        }
      }
    // The current item's slot is free: the item after the next one goes there.
    if (tid == 0) sm.item[par] = load_item(p, t + 2 * G, total);
    // ---- window end: the last MMAs land, then the spans are merged per row
    //   o = (w0 o0 + w1 o1) + (w2 o2 + w3 o3),  w_s = e^(m_s - max m) * 2^-E_s
    // in the M = 1 kernel's order; l in span order.
    bool ok_e = true;
    if (commits > waited) {
      ok_e = __all_sync(0xffffffffu, mbar_wait_bounded(&sm.mbar, (uint32_t)(commits - 1) & 1u));
      if (ok_e) waited = commits;
      tc_fence_after();
    }
    if (__syncthreads_or(!ok_e)) {
      failed = true;
      break;
    }
    float wt[kSpansPerCta], mwin, lwin = 0.0f;    // lane r: the weights of row r
    {
      const int r = lane;
      mwin = sm.wm[0][r];
#pragma unroll
      for (int s = 1; s < kSpansPerCta; ++s) mwin = fmaxf(mwin, sm.wm[s][r]);
#pragma unroll
      for (int s = 0; s < kSpansPerCta; ++s) {
        wt[s] = __fmul_rn(merge_weight(sm.wm[s][r], mwin), sm.wd[s][r]);
        lwin = __fmaf_rn(sm.wl[s][r], merge_weight(sm.wm[s][r], mwin), lwin);
      }
    }
    {
      const int b = it0.b, kh = it0.kh;
      const bool whole = !p.shard_mode && nsplit_for(ctx + M - 1) == 1;
      float* part = p.partials + (((size_t)b * p.part_ws + (it0.w - p.win_begin)) * p.Hkv + kh) *
                                     partial_stride(R);
      const int d = 32 * kw + lane;               // this thread's channel
      if (!whole && warp == 0 && lane < R) {
        part[(size_t)R * kD + lane] = mwin;
        part[(size_t)R * kD + R + lane] = lwin;
      }
#pragma unroll 1
      for (int r8 = 2 * grp; r8 < 2 * grp + 2 && 8 * r8 < R; ++r8) {
        float o[kSpansPerCta][8];
#pragma unroll
        for (int s = 0; s < kSpansPerCta; ++s) tc_ld8(tmem + tlane + 32 * s + 8 * r8, o[s]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = 8 * r8 + j;
          float w[kSpansPerCta];
#pragma unroll
          for (int s = 0; s < kSpansPerCta; ++s) w[s] = __shfl_sync(0xffffffffu, wt[s], r);
          const float l = __shfl_sync(0xffffffffu, lwin, r);
          if (r >= R) continue;
          const float y0 = __fmaf_rn(o[0][j], w[0], __fmul_rn(o[1][j], w[1]));
          const float y2 = __fmaf_rn(o[2][j], w[2], __fmul_rn(o[3][j], w[3]));
          const float y = __fadd_rn(y0, y2);
          if (whole)
            p.out[((int64_t)b * M * p.Hq + kh * gq + (r / gq) * p.Hq + r % gq) * kD + d] = __fdiv_rn(y, l);
          else
            part[(size_t)r * kD + d] = y;
        }
      }
    }
    // every warp is done with the accumulators, (m, l) and the scale slot of
    // this item; the item after the next is in its slot
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- next item
    t += G;
    par ^= 1;
    it0 = sm.item[par];
    if (it0.b < 0) break;
    {
      const Item nx = sm.item[par ^ 1];           // the next item: rows and scales ahead
      block_rows(nx, par ^ 1);
      fetch_scales(nx, par ^ 1);
    }
    // the producers are already on this item, or had nothing left to read ahead
    auto next_item = [&](Cursor& cu) {
      if (cu.item == 1) {
        cu.item = 0;
      } else {
        const Span s0 = span_of(it0, kw, M);
        cu.row = s0.row;
        cu.nb = s0.nb;
        cu.blk = 0;
      }
    };
    next_item(kc);
    next_item(vc);
    qph ^= 1u;
    ok = produce_k() && produce_v();
  }

  // ---- leave: every copy and MMA in flight lands (bounded) before the
  // tensor memory is released
  if (producer) {
    if (lane == 0) {
      int s = kcst;
      uint32_t ph2 = kcph;
      for (int k = 0; k < kc.inflight; ++k) {
        mbar_wait_bounded(&sm.kfull[kw][s], ph2);
        if (++s == kWStages) {
          s = 0;
          ph2 ^= 1u;
        }
      }
      if (vc.inflight > 0) mbar_wait_bounded(&sm.vfull[kw], (uint32_t)vph);
    }
    cp_async_wait<0>();
  }
  if (tid == 0) {
    if (q_pending) mbar_wait_bounded(&sm.qbar, qph);
    if (failed) atomicOr(p.err_word, KATTN_DEVERR_TIMEOUT);
  }
  if (commits > waited) mbar_wait_bounded(&sm.mbar, (uint32_t)(commits - 1) & 1u);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kWCols));
}

template <int PM, bool PG>
cudaError_t launch_tcw_mode(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  const int smem = (int)sizeof(TcwSmem) + 1024;  // + alignment slack
  const auto kern = decode_tcw_kernel<PM, PG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  static std::atomic<int> slots_cache[kMaxDevices];
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  int slots = (dev >= 0 && dev < kMaxDevices) ? slots_cache[dev].load() : 0;
  if (slots <= 0) {
    // CTAs per SM from the SM's shared memory, capped by the launch bounds
    // (registers) -- the occupancy query is not used for tcgen05 kernels.
    int sms = 0, smem_sm = 0, reserved = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
            cudaSuccess)
      return e;
    int per_sm = smem_sm / (smem + reserved);
    per_sm = per_sm < 1 ? 1 : (per_sm > kWCtasPerSm ? kWCtasPerSm : per_sm);
    slots = sms * per_sm;
    if (dev >= 0 && dev < kMaxDevices) slots_cache[dev].store(slots);
  }
  const int64_t items = (int64_t)p.B * p.nsplit_max * p.Hkv;   // an upper bound
  const int grid = (int)(items < slots ? items : slots);
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kWThreads), (size_t)smem, stream, p, maps);
}

template <bool PG>
cudaError_t launch_tcw_layout(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  switch (p.p_mode) {
    case KATTN_P_BF16: return launch_tcw_mode<KATTN_P_BF16, PG>(p, maps, stream);
    case KATTN_P_E4M3: return launch_tcw_mode<KATTN_P_E4M3, PG>(p, maps, stream);
    case KATTN_P_E4M3_X448: return launch_tcw_mode<KATTN_P_E4M3_X448, PG>(p, maps, stream);
    case KATTN_P_E4M3_X256: return launch_tcw_mode<KATTN_P_E4M3_X256, PG>(p, maps, stream);
    case KATTN_P_E4M3_DIRECT: return launch_tcw_mode<KATTN_P_E4M3_DIRECT, PG>(p, maps, stream);
    default: return launch_tcw_mode<KATTN_P_F32, PG>(p, maps, stream);
  }
}

}  // namespace

// The split-KV pass for 17..32 query rows per (sequence, kv head) with warps
// owning spans and P.V on tcgen05, contiguous or paged cache.
cudaError_t launch_split_tcw(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  return p.block_table != nullptr ? launch_tcw_layout<true>(p, maps, stream)
                                  : launch_tcw_layout<false>(p, maps, stream);
}

}  // namespace kattn
