// Allocation-free form of the fast decode.
//
// Some callers of this library cannot hand it a workspace: an engine whose
// device memory is owned by its own arena (a cudaMalloc from inside it would
// bypass that budget), a serving loop that must not pay cudaMalloc's latency
// and implicit synchronisation between steps, or a plugin interface that
// passes only input and output buffers.  For them kattn_decode_noalloc keeps
// the fast decode's scratch (merge counters and per-window partial results)
// in a fixed device array that lives in this file for the life of the
// process, so the call itself never allocates.
#include <cmath>
#include <mutex>

#include "kattn_internal.cuh"

namespace {

constexpr size_t kScratchBytes = KATTN_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  Every GPU that loads this library holds one copy of
// it until the process exits.  In host code `g_scratch` is only a handle for
// the symbol, never a device address: the address is looked up per device.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// The array's address on each device, looked up on the first call that
// succeeds in doing so: a failed lookup stores nothing, so a later call
// tries again (for instance once memory is no longer short).
struct DeviceScratch {
  std::mutex lock;
  void* ptr = nullptr;
};
DeviceScratch g_device_scratch[kMaxDevices];

// The scratch address on the current device `dev`, or nullptr if the
// lookup failed (the caller reports KATTN_ERR_CUDA).
void* scratch_on(int dev) {
  DeviceScratch& ds = g_device_scratch[dev];
  std::lock_guard<std::mutex> guard(ds.lock);
  if (ds.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return nullptr;
    ds.ptr = p;
  }
  return ds.ptr;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// The same argument rules as kattn_decode (fast mode), checked here first so
// that an invalid call enqueues nothing at all.
int check_args(const float* q, const int8_t* k, const float* k_scale, const int8_t* v,
               const float* v_scale, const int64_t* row_start, const int32_t* ctx_len, int B,
               int M, int Hq, int Hkv, int d, int cap_rows, int max_ctx, float sm_scale,
               int p_mode, float* out) {
  if (B < 0 || M < 1 || Hq < 1 || Hkv < 1 || cap_rows < 1 || max_ctx < 1)
    return KATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || B > 65535 || Hkv > 65535) return KATTN_ERR_INVALID_ARG;
  if (d != KATTN_HEAD_DIM) return KATTN_ERR_UNSUPPORTED;
  if (M > KATTN_MAX_M || (Hq / Hkv) * M > KATTN_MAX_ROWS) return KATTN_ERR_UNSUPPORTED;
  if ((int64_t)max_ctx + M - 1 > (int64_t)INT32_MAX / 2) return KATTN_ERR_INVALID_ARG;
  if ((int64_t)Hkv * cap_rows > (int64_t)INT32_MAX - 4096) return KATTN_ERR_UNSUPPORTED;
  if (p_mode < KATTN_P_F32 || p_mode > KATTN_P_E4M3_DIRECT) return KATTN_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return KATTN_ERR_INVALID_ARG;
  if (B == 0) return KATTN_OK;
  if (kattn::workspace_layout(B, M, Hq, max_ctx).total > kScratchBytes)
    return KATTN_ERR_WORKSPACE;
  if (!q || !k || !k_scale || !v || !v_scale || !row_start || !ctx_len || !out)
    return KATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(k_scale, 4) || !aligned(v, 16) ||
      !aligned(v_scale, 4) || !aligned(row_start, 8) || !aligned(ctx_len, 4) ||
      !aligned(out, 16))
    return KATTN_ERR_MISALIGNED;
  return KATTN_OK;
}

}  // namespace

extern "C" int kattn_decode_noalloc(const float* q, const int8_t* k, const float* k_scale,
                                    const int8_t* v, const float* v_scale,
                                    const int64_t* row_start, const int32_t* ctx_len, int B,
                                    int M, int Hq, int Hkv, int d, int cap_rows, int max_ctx,
                                    float sm_scale, int p_mode, float* out, void* stream) {
  const int st = check_args(q, k, k_scale, v, v_scale, row_start, ctx_len, B, M, Hq, Hkv, d,
                            cap_rows, max_ctx, sm_scale, p_mode, out);
  if (st != KATTN_OK || B == 0) return st;

  // Set-up, once per device and with that device current: find where the
  // scratch array lives on it (retried by the next call if it failed).
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KATTN_ERR_UNSUPPORTED;
  void* scratch = scratch_on(dev);
  if (scratch == nullptr) return KATTN_ERR_CUDA;

  // The array keeps whatever the previous call left in it.  The header (the
  // error word) must start at zero; the work list, the quantized queries and
  // the partials are always written before they are read.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 256, s) != cudaSuccess) return KATTN_ERR_CUDA;
  return kattn_decode(q, k, k_scale, v, v_scale, row_start, ctx_len, B, M, Hq, Hkv, d, cap_rows,
                      max_ctx, sm_scale, p_mode, 0, out, scratch, kScratchBytes, stream);
}
