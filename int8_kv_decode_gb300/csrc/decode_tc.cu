// The split-KV pass for 17..32 query rows per (sequence, kv head) with P.V on
// the fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Each row gets the arithmetic of the M = 1 kernel (decode_split.cuh) in the
// same order: the int8 QK on mma.sync for one 8-row tile per warp, the same
// online softmax per 32-key block with the maximum reset at every 128-key
// span, the same P.V operands (V exact in f16, a = round_p(p) * v_scale * 2^E
// split into f16 hi + lo) and the same order of 16-key MMA steps: hi then lo
// of the first half of a block, then of the second.  tcgen05 kind::f16 with an
// f32 accumulator adds such a step to the accumulator exactly as mma.sync
// m16n8k16 does (measured on this GPU: identical bits), so every row equals
// the M = 1 kernel's bytes and batch invariance holds.
//
// Layout: one CTA of 4 warps per work item (sequence, 512-key window, kv
// head), persistent over the work list, 4 CTAs per SM (tensor memory: 128
// columns each).  The window's 16 blocks of 32 keys go through in order, span
// after span; for each block warp w computes the scores and P of rows
// 8w..8w+7 and converts keys 8w..8w+7 of V to f16 for all 128 channels.  One
// thread issues the block's four MMAs (two with p_mode e4m3-direct, which has
// no low part):
//   D_s[d][row] += Vt[d][key] * P[row][key]   (M = 128 channels, N = 32
// rows, K = 16 keys), D_s = span s's accumulator in tensor memory (lanes =
// channels, columns 32s .. 32s + 31 = rows).  When a row's running max moves,
// the four warps rescale their 32 lanes of D_s by alpha before the MMAs.  At
// the window's end each warp merges the four spans for its 32 channels in the
// same order as the M = 1 kernel.  PG: the paged cache, block rows from the
// block table.
#include "tcgen05_common.cuh"

namespace kattn {
namespace {

constexpr int kTcRows = 32;                      // rows per CTA (R in 17..32)
constexpr int kTcWarps = 4;
constexpr int kTcStages = 4;                     // TMA stages of 32 keys (K and V)
constexpr int kTcCols = kSpansPerCta * kTcRows;  // tensor-memory columns: 128
constexpr int kTcCtasPerSm = 512 / kTcCols;       // resident CTAs: all of tensor memory
static_assert(kTcRows == kTcN, "the instruction descriptor's N");

struct __align__(1024) TcSmem {
  uint8_t ring[kTcStages][2][kBlockBytes];       // K and V blocks of 32 keys (128-byte swizzle)
  // MMA operands of the block in flight (no swizzle, K-major, 16 keys per
  // half): element (row, key) at (row / 8) * 256 + (key / 8) * 128 +
  // (row % 8) * 16 + (key % 8) * 2.
  uint8_t vt[2][128 * 16 * 2];                   // [half] V transposed: rows = channels
  uint8_t pb[2][2][kTcRows * 16 * 2];            // [half][hi | lo] P: rows = query rows
  uint8_t qbuf[kTcRows * (kD + 4)];              // the item's int8 rows, then scales
  uint64_t full[kTcStages];                      // the stage's K and V landed
  uint64_t qbar, mbar;                           // queries landed / MMAs done
  __align__(16) float alpha[kTcRows];            // this block's alpha per row
  float wm[kSpansPerCta][kTcRows], wl[kSpansPerCta][kTcRows], wd[kSpansPerCta][kTcRows];
  int brow[2][kSplitC / kBlockBk];               // paged: cache rows of an item's blocks, by parity
  uint32_t tmem;
  // A copy or an MMA group never completed, by block parity: a warp may flag
  // block n + 1 before a slower one has read the flag of block n.
  int fail[2];
};

template <int PM, bool PG>
__global__ void __launch_bounds__(kTcWarps * 32, kTcCtasPerSm)
decode_tc_kernel(const DecodeParams p, const __grid_constant__ TmaMaps maps) {
  extern __shared__ unsigned char smem_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t kQBytes = kTcRows * (kD + 4);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int gq = p.g, M = p.M, R = p.R;
  const int row0 = 8 * warp;                      // this warp's 8 query rows
  int jrow[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) jrow[e] = min((row0 + 2 * c + e) / gq, M - 1);

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) mbar_init(&sm.full[s], 1);
    mbar_init(&sm.qbar, 1);
    mbar_init(&sm.mbar, 1);
    sm.fail[0] = sm.fail[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                 ::"r"(smem_u32(&sm.tmem)), "r"(kTcCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const uint32_t tlane = (uint32_t)(32 * warp) << 16;   // this warp's lanes
  griddep_wait();                                 // the work list and the packed queries
  griddep_launch_dependents();

  const int total = (int)__ldcg(p.item_count);
  const int G = gridDim.x;
  const uint64_t kv_policy = l2_evict_first();
  int gbase = 0;                                  // blocks of the items before this one
  int issued = 0;                                 // thread 0: blocks whose copies are issued
  int cons = 0;                                   // blocks every warp is done with
  int commits = 0, waited = 0;                    // MMA groups committed / waited for
  uint32_t qph = 0;
  bool failed = false, q_pending = false;
  Item it = load_item(p, blockIdx.x, total), nxt = load_item(p, blockIdx.x + G, total);
  RawUnit raw = fetch_unit(p, blockIdx.x + 2 * G, total, 1);   // decoded one item later
  int nbs[kSpansPerCta], nbs_n[kSpansPerCta], nbt = 0, nbt_n = 0;
  auto blocks_of = [&](const Item& x, int (&n)[kSpansPerCta]) {
    int tot = 0;
#pragma unroll
    for (int s = 0; s < kSpansPerCta; ++s) {
      n[s] = x.b >= 0 ? span_of(x, s, M).nb : 0;
      tot += n[s];
    }
    return tot;
  };
  auto fetch_queries = [&](const Item& x) {      // thread 0
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    mbar_expect_tx(&sm.qbar, kQBytes);
    bulk_load(sm.qbuf, p.qpack + ((size_t)x.b * p.Hkv + x.kh) * kQBytes, kQBytes, &sm.qbar);
    q_pending = true;
  };
  // Block k of an item holds keys w * kSplitC + 32k .. + 31 (every span but
  // the last non-empty one is full).  Paged: the rows come from brow, filled
  // by warp 0 -- the current item's (par) before the item starts, the next
  // item's (par ^ 1) after the current item's first block (nrows).
  int par = 0;
  bool nrows = !PG;                               // thread 0: brow[par ^ 1] is filled
  // Thread 0: issue the copies of blocks [issued, limit) -- this item's, then
  // the next item's.  A block's stage was last read by the block kTcStages
  // earlier, which every warp has passed (a CTA barrier follows each block).
  auto produce = [&](int limit) {
    while (issued < limit) {
      const int k = issued - gbase;
      int row;
      if (k < nbt) {
        row = PG ? sm.brow[par][k] : it.row + it.w * kSplitC + k * kBlockBk;
      } else if (k - nbt < nbt_n && nrows) {
        row = PG ? sm.brow[par ^ 1][k - nbt] : nxt.row + nxt.w * kSplitC + (k - nbt) * kBlockBk;
      } else {
        break;
      }
      const int st = issued % kTcStages;
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      mbar_expect_tx(&sm.full[st], 2 * kBlockBytes);
      tma_load_block(sm.ring[st][0], &maps.k, row, &sm.full[st], kv_policy);
      tma_load_block(sm.ring[st][1], &maps.v, row, &sm.full[st], kv_policy);
      ++issued;
    }
  };
  if (tid == 0 && it.b >= 0) fetch_queries(it);
  float ksn[4], vsn[4];                           // the next span's k and v scales
  load_span_scales<PG>(p, it, span_of(it, 0, M), lane, ksn, vsn);

  for (int t = blockIdx.x; t < total && !failed; t += G) {
    const int ctx = it.ctx, b = it.b, kh = it.kh;
    nbt = blocks_of(it, nbs);
    nbt_n = blocks_of(nxt, nbs_n);
    int pentry = 0;                               // paged, warp 0 lane k: the next item's block k
    if constexpr (PG) {
      if (warp == 0) {
        if (t == (int)blockIdx.x) {               // the first item: its rows now
          if (lane < nbt) {
            const int key = it.w * kSplitC + lane * kBlockBk;
            sm.brow[par][lane] = it.row + tc_page_row(p, tc_page_entry(p, it.b, key), key);
          }
          __syncwarp();
        }
        if (lane < nbt_n) pentry = tc_page_entry(p, nxt.b, nxt.w * kSplitC + lane * kBlockBk);
      }
      nrows = false;
    }
    if (tid == 0) produce(gbase + kTcStages);
    // every span's accumulator starts at +0 (each warp its own lanes)
    {
      float z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0.0f;
#pragma unroll
      for (int s = 0; s < kSpansPerCta; ++s) tc_st32(tmem + tlane + 32 * s, z);
    }
    const bool q_ok = mbar_wait_bounded(&sm.qbar, qph);
    if (__syncthreads_or(!q_ok)) {
      failed = true;
      break;
    }
    qph ^= 1u;
    if (tid == 0) q_pending = false;
    uint32_t qw8[8];
    {
      const uint4* src = reinterpret_cast<const uint4*>(&sm.qbuf[(row0 + g) * kD + 32 * c]);
      const uint4 lo = src[0], hi = src[1];
      qw8[0] = lo.x; qw8[1] = lo.y; qw8[2] = lo.z; qw8[3] = lo.w;
      qw8[4] = hi.x; qw8[5] = hi.y; qw8[6] = hi.z; qw8[7] = hi.w;
    }
    float qs_row[2];
    {
      const float* qsb = reinterpret_cast<const float*>(&sm.qbuf[kTcRows * kD]);
      qs_row[0] = qsb[row0 + 2 * c];
      qs_row[1] = qsb[row0 + 2 * c + 1];
    }
    int Lrow[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) Lrow[e] = ctx + jrow[e];

    int kb = 0;                                   // item block index
    for (int s = 0; s < kSpansPerCta && !failed; ++s) {
      const Span sp = span_of(it, s, M);
      float ksp[4], vsp[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ksp[e] = ksn[e];
        vsp[e] = vsn[e];
      }
      // the next span's scales, one span ahead (this item's, else the next item's first)
      if (s + 1 < kSpansPerCta) load_span_scales<PG>(p, it, span_of(it, s + 1, M), lane, ksn, vsn);
      else load_span_scales<PG>(p, nxt, span_of(nxt, 0, M), lane, ksn, vsn);
      // 2^E per row from the largest v_scale among the keys the row sees
      float up_row[2], down_row[2];
      {
        const int kc = min(sp.s1, ctx);
        float vm = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (sp.s0 + lane + 32 * e < kc) vm = fmaxf(vm, vsp[e]);
        vm = warp_max(vm);
        float vtl[kMaxM - 1];
#pragma unroll
        for (int q = 0; q < kMaxM - 1; ++q) vtl[q] = 0.0f;
        if (sp.s1 > ctx) {
#pragma unroll
          for (int q = 0; q < kMaxM - 1; ++q) {
            const int rel = ctx + q - sp.s0;
            if (q < M - 1 && rel >= 0 && ctx + q < sp.s1) {
              const int e = rel >> 5;
              const float mine = e == 0 ? vsp[0] : e == 1 ? vsp[1] : e == 2 ? vsp[2] : vsp[3];
              vtl[q] = __shfl_sync(0xffffffffu, mine, rel & 31);
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float vmax = vm;
#pragma unroll
          for (int q = 0; q < kMaxM - 1; ++q)
            if (q < jrow[e]) vmax = fmaxf(vmax, vtl[q]);
          const int bexp = min(max(268 - (int)((__float_as_uint(vmax) >> 23) & 0xffu), 1), 253);
          up_row[e] = __uint_as_float((uint32_t)bexp << 23);
          down_row[e] = __uint_as_float((uint32_t)(254 - bexp) << 23);
        }
      }
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
      for (int i = 0; i < sp.nb; ++i, ++kb) {
        const int gb = gbase + kb, st = gb % kTcStages;
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
        bool ok_b = mbar_wait_bounded(&sm.full[st], (uint32_t)(gb / kTcStages) & 1u);
        const uint8_t* Kt = sm.ring[st][0];
        const uint8_t* Vt = sm.ring[st][1];
        // ---- QK of rows row0 .. row0 + 7 on the int8 MMA (sc as in the M = 1 kernel)
        float sc[2][4];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int ra = 16 * hf + g, rb = ra + 8;
          const uint4 a_lo = lds128(Kt + swz(ra, 2 * c)), a_hi = lds128(Kt + swz(ra, 2 * c + 1));
          const uint4 b_lo = lds128(Kt + swz(rb, 2 * c)), b_hi = lds128(Kt + swz(rb, 2 * c + 1));
          const uint32_t wa[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
          const uint32_t wb[8] = {b_lo.x, b_lo.y, b_lo.z, b_lo.w, b_hi.x, b_hi.y, b_hi.z, b_hi.w};
          int iacc[4] = {0, 0, 0, 0}, iacc2[4] = {0, 0, 0, 0};
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4)
            mma_i8((s4 & 1) ? iacc2 : iacc, wa[2 * s4], wb[2 * s4], wa[2 * s4 + 1], wb[2 * s4 + 1],
                   qw8[2 * s4], qw8[2 * s4 + 1]);
#pragma unroll
          for (int u = 0; u < 4; ++u) sc[hf][u] = __int2float_rn(iacc[u] + iacc2[u]);
        }
        // ---- scores ((S * (qs * ks)) * sm_scale), masked past each row's L
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const float ksv = ks4[2 * hf + k2];
            const float2 qk = f2_mul(make_float2(qs_row[0], qs_row[1]), make_float2(ksv, ksv));
            float2 s2 = f2_mul(make_float2(sc[hf][2 * k2], sc[hf][2 * k2 + 1]), qk);
            s2 = f2_mul(s2, make_float2(p.sm_scale, p.sm_scale));
            sc[hf][2 * k2] = s2.x;
            sc[hf][2 * k2 + 1] = s2.y;
          }
        if (t0 + kBlockBk > ctx) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int key = t0 + 16 * hf + g + 8 * (u >> 1);
              if (key >= Lrow[u & 1]) sc[hf][u] = -INFINITY;
            }
        }
        // ---- online softmax of rows row0 + 2c + e over the block (a in sc)
        float alpha[2];
        bool rescale = false;
        softmax_tile<PM>(sc[0], sc[1], m_run, l_run, up_row, vs4, alpha, rescale);
        // ---- P operand words: {a[key 2c][row g], a[key 2c+1][row g]} and keys
        // 2c+8, 2c+9 of each half, split into f16 hi + lo (as the M = 1 kernel's
        // B fragments)
        uint32_t ph[2][2], pl[2][2];
        {
          const int srcA = 8 * c + (g >> 1), srcB = srcA + 4;
          const bool odd = g & 1;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            float fA[4], fB[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              fA[u] = __shfl_sync(0xffffffffu, sc[hf][u], srcA);
              fB[u] = __shfl_sync(0xffffffffu, sc[hf][u], srcB);
            }
            split_f16x2(odd ? fA[1] : fA[0], odd ? fB[1] : fB[0], ph[hf][0], pl[hf][0]);
            split_f16x2(odd ? fA[3] : fA[2], odd ? fB[3] : fB[2], ph[hf][1], pl[hf][1]);
          }
        }
        // ---- V operand: warp w takes keys 8w .. 8w + 7 of the block (half
        // w / 2), lane l channels 4l .. 4l + 3.  Word m of a channel's 16-byte
        // row holds keys 2m, 2m + 1.  Store t writes channel 4l + ((t + l / 2)
        // mod 4), which spreads the 32 lanes over all eight 16-byte bank groups.
        uint4 vo[4];
        {
          uint32_t W[8];
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8)
            W[k8] = *reinterpret_cast<const uint32_t*>(Vt + swz(8 * warp + k8, lane >> 2) + 4 * (lane & 3));
          const uint32_t x0 = (uint32_t)(lane >> 1) & 3u, x1 = (x0 + 1u) & 3u;
          const uint32_t selA = x0 | ((4u + x0) << 4) | (((x0 + 2u) & 3u) << 8) | ((4u + ((x0 + 2u) & 3u)) << 12);
          const uint32_t selB = x1 | ((4u + x1) << 4) | (((x1 + 2u) & 3u) << 8) | ((4u + ((x1 + 2u) & 3u)) << 12);
          uint32_t h[4][4];                                // [store t][word m]
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
          for (int t4 = 0; t4 < 4; ++t4) vo[t4] = make_uint4(h[t4][0], h[t4][1], h[t4][2], h[t4][3]);
        }
        // the stage is read: it may be refilled after the barrier below
        // ---- wait for the previous block's MMAs (they read vt and pb)
        if (commits > waited) {
          const bool ok_m = mbar_wait_bounded(&sm.mbar, (uint32_t)(commits - 1) & 1u);
          if (ok_m) waited = commits;             // else the exit waits again
          ok_b = ok_m && ok_b;
          tc_fence_after();
        }
        {
          const int r = row0 + g;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            *reinterpret_cast<uint32_t*>(sm.pb[hf][0] + op_off(r, 2 * c)) = ph[hf][0];
            *reinterpret_cast<uint32_t*>(sm.pb[hf][0] + op_off(r, 2 * c + 8)) = ph[hf][1];
            if constexpr (PM != KATTN_P_E4M3_DIRECT) {   // that mode has no low part
              *reinterpret_cast<uint32_t*>(sm.pb[hf][1] + op_off(r, 2 * c)) = pl[hf][0];
              *reinterpret_cast<uint32_t*>(sm.pb[hf][1] + op_off(r, 2 * c + 8)) = pl[hf][1];
            }
          }
          uint8_t* vdst = sm.vt[warp >> 1];
#pragma unroll
          for (int t4 = 0; t4 < 4; ++t4) {
            const int d = 4 * lane + ((t4 + (lane >> 1)) & 3);
            *reinterpret_cast<uint4*>(vdst + op_off(d, 8 * (warp & 1))) = vo[t4];
          }
          if (g == 0) {
            sm.alpha[row0 + 2 * c] = alpha[0];
            sm.alpha[row0 + 2 * c + 1] = alpha[1];
          }
        }
        if (!ok_b) sm.fail[gb & 1] = 1;
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        tc_fence_before();
        const bool resc = __syncthreads_or(rescale) != 0;
        if (sm.fail[gb & 1]) {
          failed = true;
          break;
        }
        cons = gb + 1;
        if (resc && i > 0) {                      // rows whose max moved: D_s *= alpha
#pragma unroll
          for (int h16 = 0; h16 < 2; ++h16) {
            float v[16];
            tc_ld16(tmem + tlane + 32 * s + 16 * h16, v);
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 a4 = reinterpret_cast<const float4*>(sm.alpha)[4 * h16 + j4];
              v[4 * j4] = __fmul_rn(v[4 * j4], a4.x);
              v[4 * j4 + 1] = __fmul_rn(v[4 * j4 + 1], a4.y);
              v[4 * j4 + 2] = __fmul_rn(v[4 * j4 + 2], a4.z);
              v[4 * j4 + 3] = __fmul_rn(v[4 * j4 + 3], a4.w);
            }
            tc_st16(tmem + tlane + 32 * s + 16 * h16, v);
          }
          tc_wait_st();
          tc_fence_before();
          __syncthreads();
        }
        if (PG && kb == 0 && warp == 0) {        // the next item's block rows
          if (lane < nbt_n) {
            const int key = nxt.w * kSplitC + lane * kBlockBk;
            sm.brow[par ^ 1][lane] = nxt.row + tc_page_row(p, pentry, key);
          }
          __syncwarp();
          nrows = true;
        }
        if (tid == 0) {
          tc_fence_after();
          const uint32_t dcol = tmem + 32 * s;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            tc_mma(dcol, smem_desc(sm.vt[hf]), smem_desc(sm.pb[hf][0]));
            if constexpr (PM != KATTN_P_E4M3_DIRECT)
              tc_mma(dcol, smem_desc(sm.vt[hf]), smem_desc(sm.pb[hf][1]));
          }
          tc_commit(&sm.mbar);
          if (kb == 0 && nxt.b >= 0) fetch_queries(nxt);   // every warp has read this item's
          produce(gb + 1 + kTcStages);
        }
        ++commits;
      }
      if (failed) break;
      // ---- the span's row sums and maxima (the M = 1 reduction order)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = l_run[e];
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 16));
        if (g == 0) {
          const int r = row0 + 2 * c + e;
          sm.wl[s][r] = v;
          sm.wm[s][r] = m_run[e];
          sm.wd[s][r] = down_row[e];
        }
      }
    }
    if (failed) break;

    // ---- window end: the last MMAs land, then the spans are merged per row
    //   o = (w0 o0 + w1 o1) + (w2 o2 + w3 o3),  w_s = e^(m_s - max m) * 2^-E_s
    // in the M = 1 kernel's order; l in span order.
    bool ok_e = true;
    if (commits > waited) {
      ok_e = mbar_wait_bounded(&sm.mbar, (uint32_t)(commits - 1) & 1u);
      if (ok_e) waited = commits;
      tc_fence_after();
    }
    if (__syncthreads_or(!ok_e)) {
      failed = true;
      break;
    }
    // lane r: the weights of row r
    float wt[kSpansPerCta], mwin, lwin = 0.0f;
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
    const bool whole = !p.shard_mode && nsplit_for(ctx + M - 1) == 1;
    float* part = p.partials + (((size_t)b * p.part_ws + (it.w - p.win_begin)) * p.Hkv + kh) *
                                   partial_stride(R);
    const int d = 32 * warp + lane;               // this thread's channel
    if (!whole && warp == 0 && lane < R) {
      part[(size_t)R * kD + lane] = mwin;
      part[(size_t)R * kD + R + lane] = lwin;
    }
#pragma unroll 1
    for (int r8 = 0; r8 < kTcRows / 8 && 8 * r8 < R; ++r8) {
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
    gbase += nbt;
    it = nxt;
    nxt = decode_unit(raw);
    raw = fetch_unit(p, t + 3 * G, total, 1);
    par ^= 1;
  }

  // ---- leave: every copy and MMA in flight lands (bounded) before the
  // tensor memory is released
  if (tid == 0) {
    for (int k = cons; k < issued; ++k)
      mbar_wait_bounded(&sm.full[k % kTcStages], (uint32_t)(k / kTcStages) & 1u);
    if (q_pending) mbar_wait_bounded(&sm.qbar, qph);
    if (failed) atomicOr(p.err_word, KATTN_DEVERR_TIMEOUT);
  }
  if (commits > waited) mbar_wait_bounded(&sm.mbar, (uint32_t)(commits - 1) & 1u);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTcCols));
}

template <int PM, bool PG>
cudaError_t launch_tc_mode(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  const int smem = (int)sizeof(TcSmem) + 1024;   // + alignment slack
  constexpr int kThreads = kTcWarps * 32;
  const auto kern = decode_tc_kernel<PM, PG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  static std::atomic<int> slots_cache[kMaxDevices];
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  int slots = (dev >= 0 && dev < kMaxDevices) ? slots_cache[dev].load() : 0;
  if (slots <= 0) {
    // CTAs per SM from the SM's shared memory (the occupancy query reports
    // one for this kernel), capped by the 512 tensor-memory columns (kTcCols
    // per CTA) and by the register file (launch bounds: 4 CTAs of 128 threads).
    int sms = 0, smem_sm = 0, reserved = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
            cudaSuccess)
      return e;
    int per_sm = smem_sm / (smem + reserved);
    per_sm = per_sm < 1 ? 1 : (per_sm > kTcCtasPerSm ? kTcCtasPerSm : per_sm);
    slots = sms * per_sm;
    if (dev >= 0 && dev < kMaxDevices) slots_cache[dev].store(slots);
  }
  const int64_t items = (int64_t)p.B * p.nsplit_max * p.Hkv;   // an upper bound
  const int grid = (int)(items < slots ? items : slots);
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), (size_t)smem, stream, p, maps);
}

template <bool PG>
cudaError_t launch_tc_layout(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  switch (p.p_mode) {
    case KATTN_P_BF16: return launch_tc_mode<KATTN_P_BF16, PG>(p, maps, stream);
    case KATTN_P_E4M3: return launch_tc_mode<KATTN_P_E4M3, PG>(p, maps, stream);
    case KATTN_P_E4M3_X448: return launch_tc_mode<KATTN_P_E4M3_X448, PG>(p, maps, stream);
    case KATTN_P_E4M3_X256: return launch_tc_mode<KATTN_P_E4M3_X256, PG>(p, maps, stream);
    case KATTN_P_E4M3_DIRECT: return launch_tc_mode<KATTN_P_E4M3_DIRECT, PG>(p, maps, stream);
    default: return launch_tc_mode<KATTN_P_F32, PG>(p, maps, stream);
  }
}

}  // namespace

// The split-KV pass on the fifth-generation tensor cores for 17..32 query rows
// per (sequence, kv head), contiguous or paged cache.
cudaError_t launch_split_tc(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  return p.block_table != nullptr ? launch_tc_layout<true>(p, maps, stream)
                                  : launch_tc_layout<false>(p, maps, stream);
}

}  // namespace kattn
