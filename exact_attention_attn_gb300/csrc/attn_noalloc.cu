// attn_fwd_splitkv_noalloc: the split-KV path with its partial results in a
// fixed, file-scope device array instead of a per-call allocation, for
// callers that may not allocate device memory (see include/attn.h).
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "attn.h"
#include "attn_internal.h"

namespace attn {
namespace {

constexpr size_t kScratchFloats = ATTN_NOALLOC_SCRATCH_BYTES / sizeof(float);

// The scratch.  Device code could name it directly; host code must not use
// the symbol as an address (on the host it is only a stand-in): the device
// address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
float *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch on `device` (which is current); looked up on
// the first call for that device.
int scratch_address(int device, float **out) {
  if (device < 0 || device >= kMaxDevices) return ATTN_ERR_ARCH;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[device]) {
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) return record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    g_scratch_ptr[device] = static_cast<float *>(ptr);
  }
  *out = g_scratch_ptr[device];
  return ATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace attn

extern "C" int attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                                        int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                                        float scale, int causal, int kv_splits, attn_stream_t stream) {
  using namespace attn;
  // the size and flag checks of attn_fwd, then this entry point's own
  int rc = check_problem(B, Hq, Hkv, Nq, Nkv, D, causal);
  if (rc != ATTN_OK) return rc;
  if (!isfinite(scale) || kv_splits < 2 || kv_splits > kMaxSplits) return ATTN_ERR_ARG;
  if (B == 0 || Nq == 0) return ATTN_OK;
  if (!q || !o || !lse) return ATTN_ERR_ARG;
  if (Nkv > 0 && (!k || !v)) return ATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_ALIGN;
  if (Nkv > 0 && (!aligned16(k) || !aligned16(v))) return ATTN_ERR_ALIGN;
  const int64_t rows = (int64_t)B * Hq * Nq;
  const int64_t need = (int64_t)kv_splits * rows * (D + 1);  // floats
  if (Nkv > 0 && need > (int64_t)kScratchFloats) return ATTN_ERR_SCRATCH;

  int device = 0, sm_count = 0;
  int *status = nullptr;
  rc = current_device(&device, &sm_count, &status);
  if (rc != ATTN_OK) return rc;

  Problem p{};
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.k = static_cast<const __nv_bfloat16 *>(k);
  p.v = static_cast<const __nv_bfloat16 *>(v);
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = Nq; p.Nkv = Nkv; p.D = D;
  p.scale = scale;
  p.causal = causal;
  p.status = status;
  p.kv_splits = 1;
  p.debug_flags = debug_flags();
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  cudaError_t e;
  if (Nkv == 0) {
    e = launch_nokeys(p, sm_count, st);
    return e == cudaSuccess ? ATTN_OK : record_cuda_error(e);
  }
  float *scratch = nullptr;
  rc = scratch_address(device, &scratch);
  if (rc != ATTN_OK) return rc;
  p.kv_splits = kv_splits;
  p.ws_o = scratch;
  p.ws_lse = scratch + (int64_t)kv_splits * rows * D;  // 16-byte aligned: D is a multiple of 64
  // the kernel choice, wait bound and debug flags of attn_fwd_splitkv
  e = launch_tensor(p, device, st);
  if (e == cudaSuccess) e = launch_combine(p, st);
  return e == cudaSuccess ? ATTN_OK : record_cuda_error(e);
}
