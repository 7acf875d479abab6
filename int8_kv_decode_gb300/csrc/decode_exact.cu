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
// in parallel per chunk of 128 keys; then thread i walks channel i's chain
// through the chunk.  One CTA of 128 threads per query row.
#include "device_common.cuh"

namespace kattn {
namespace {

constexpr int kChunk = 128;

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

__global__ void __launch_bounds__(kChunk)
decode_exact_kernel(DecodeParams p, ExpfConsts consts) {
  __shared__ ExpfConsts c;
  __shared__ __align__(16) uint32_t q8[kD / 4];
  __shared__ float red[kChunk / 32];
  __shared__ float s_alpha[kChunk], s_p[kChunk], s_pr[kChunk], s_vs[kChunk];
  __shared__ float s_carry;
  __shared__ int s_row[kChunk];                   // plane rows of the chunk's keys

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x % p.Hq;
  const int j = (blockIdx.x / p.Hq) % p.M;
  const int b = blockIdx.x / (p.Hq * p.M);
  const int kh = h / p.g;
  const int64_t qrow = ((int64_t)b * p.M + j) * p.Hq + h;
  float* orow = p.out + qrow * kD;

  if (!sequence_valid(p, b)) {
    orow[tid] = __int_as_float(0x7fc00000);
    return;
  }
  const int L = p.ctx_len[b] + j;
  const int rs = sequence_row0(p, b);

  for (int i = tid; i < (int)(sizeof(ExpfConsts) / sizeof(double)); i += kChunk)
    reinterpret_cast<double*>(&c)[i] = reinterpret_cast<const double*>(&consts)[i];

  // int8 query: absmax over the 128 channels, then one IEEE division each.
  const float x = p.q[qrow * kD + tid];
  float amax = warp_max(fabsf(x));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const float qs = quant_scale(amax);
  reinterpret_cast<int8_t*>(q8)[tid] = (int8_t)quant_one(x, qs);
  if (tid == 0) s_carry = -INFINITY;
  __syncthreads();

  // Key t is row `row` of head kh's plane: rs + t, or from the block table.
  const int64_t plane = (int64_t)kh * p.cap_rows;
  const int8_t* kbase = p.k + plane * kD;
  const int8_t* vbase = p.v + plane * kD;
  const float* ksb = p.k_scale + plane;
  const float* vsb = p.v_scale + plane;

  float o = 0.0f, l = 0.0f;
  for (int t0 = 0; t0 < L; t0 += kChunk) {
    const int t = t0 + tid;
    const bool live = t < L;
    float s = -INFINITY;
    const int row = !live ? 0 : p.block_table == nullptr ? rs + t : paged_row(p, b, t);
    s_row[tid] = row;
    if (live) {
      const int4* krow = reinterpret_cast<const int4*>(kbase + (int64_t)row * kD);
      int acc = 0;
#pragma unroll
      for (int cc = 0; cc < kD / 16; ++cc) {
        const int4 kv = krow[cc];
        acc = __dp4a((int)kv.x, (int)q8[4 * cc + 0], acc);
        acc = __dp4a((int)kv.y, (int)q8[4 * cc + 1], acc);
        acc = __dp4a((int)kv.z, (int)q8[4 * cc + 2], acc);
        acc = __dp4a((int)kv.w, (int)q8[4 * cc + 3], acc);
      }
      s = __fmul_rn(__fmul_rn((float)acc, __fmul_rn(qs, ksb[row])), p.sm_scale);
    }
    // Inclusive prefix max over the chunk, seeded with the running max.
    float pm = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o2 = __shfl_up_sync(0xffffffffu, pm, off);
      if (lane >= off) pm = fmaxf(pm, o2);
    }
    if (lane == 31) red[warp] = pm;
    const float carry = s_carry;
    __syncthreads();
    for (int w = 0; w < warp; ++w) pm = fmaxf(pm, red[w]);
    pm = fmaxf(pm, carry);
    // Running max before this key: the previous lane's inclusive max, or for
    // a warp's first lane the max of the carry and all earlier warps.
    float prev = __shfl_up_sync(0xffffffffu, pm, 1);
    if (lane == 0) {
      float pw = carry;
      for (int w = 0; w < warp; ++w) pw = fmaxf(pw, red[w]);
      prev = pw;
    }
    if (live) {
      const float a = expf_tang(__fsub_rn(prev, pm), c);
      const float pp = expf_tang(__fsub_rn(s, pm), c);
      s_alpha[tid] = a;
      s_p[tid] = pp;
      s_pr[tid] = round_p_exact(pp, p.p_mode);
      s_vs[tid] = vsb[row];
    }
    __syncthreads();
    if (tid == min(kChunk, L - t0) - 1) s_carry = pm;
    const int n = min(kChunk, L - t0);
    for (int u = 0; u < n; ++u) {
      const float a = s_alpha[u];
      const float vdeq = __fmul_rn((float)vbase[(int64_t)s_row[u] * kD + tid], s_vs[u]);
      o = __fadd_rn(__fmul_rn(o, a), __fmul_rn(s_pr[u], vdeq));
      l = __fadd_rn(__fmul_rn(l, a), s_p[u]);
    }
    __syncthreads();
  }
  orow[tid] = __fdiv_rn(o, l);
}

}  // namespace

cudaError_t launch_decode_exact(const DecodeParams& p, const ExpfConsts& c,
                                cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.M * p.Hq;
  decode_exact_kernel<<<(unsigned)rows, kChunk, 0, stream>>>(p, c);
  return cudaGetLastError();
}

}  // namespace kattn
