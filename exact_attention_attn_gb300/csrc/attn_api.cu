// Host side of the C ABI declared in include/attn.h: argument checks, the
// per-device status word, and the choice of kernel.
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"

namespace attn {
namespace {

// Device status word: the first kernel error on a device wins; attn_fwd_status
// reads and clears it.
__device__ int g_status;

constexpr int kMaxDevices = 64;
// bounded device-side waits give up after this long (a healthy wait lasts
// microseconds)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
std::atomic<long long> g_wait_limit_ns{(long long)kWaitLimitNs};
std::atomic<int> g_debug_flags{0};
struct DeviceInfo {
  bool ready = false;
  bool arch_ok = false;
  int sm_count = 0;
  int *status = nullptr;
  int device = 0;
  // the split-KV workspace's memory pool: it keeps its memory between calls
  // (the default pool hands memory back to the driver at every synchronise,
  // and a fresh block from the driver costs more than the split saves)
  cudaMemPool_t ws_pool = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

thread_local char t_last_error[256] = "";

int record(cudaError_t e) {
  snprintf(t_last_error, sizeof(t_last_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return ATTN_ERR_LAUNCH;
}

// Reads the compute capability and the status word's device address once
// per device (with that device current).
int device_info(DeviceInfo **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_ARCH;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return record(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return record(e);
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return record(e);
    d.arch_ok = (major == 10 && minor == 3);
    d.device = dev;
    d.sm_count = sms;
    if (d.arch_ok) {
      void *ptr = nullptr;
      if ((e = cudaGetSymbolAddress(&ptr, g_status)) != cudaSuccess) return record(e);
      d.status = static_cast<int *>(ptr);
    }
    d.ready = true;
  }
  if (!d.arch_ok) return ATTN_ERR_ARCH;
  *out = &d;
  return ATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_sizes(int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal) {
  if (B < 0 || Nq < 0 || Nkv < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_ARG;
  if (D < 64 || D > ATTN_MAX_HEAD_DIM || D % 64 != 0) return ATTN_ERR_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  // element counts must fit the kernels' 64-bit index math with room to spare
  if ((int64_t)B * Hq * Nq * (int64_t)D > (int64_t)1 << 46) return ATTN_ERR_ARG;
  if ((int64_t)B * Hkv * Nkv * (int64_t)D > (int64_t)1 << 46) return ATTN_ERR_ARG;
  return ATTN_OK;
}

// CTAs of the tensor-core launch for one key range per query tile.
// D-slices per 128-row tile: the cluster kernel's CTAs per cluster where it
// runs, else the per-slice kernel's output slices.
int d_slices(int D) {
  const int nx = (debug_flags() & ATTN_DEBUG_NO_CLUSTER) ? 0 : tcx_slices(D);
  return nx > 0 ? nx : tc_config(D).nslices;
}

int64_t base_ctas(const Problem &p) {
  const int64_t tiles = (p.Nq + 127) / 128;
  if (tc2_supports(p.D)) return ((tiles + 1) / 2) * p.B * p.Hq;
  return tiles * p.B * p.Hq * d_slices(p.D);
}

// Key-range splits when one CTA per query tile leaves SMs idle: the split
// count s (<= 16, at least two key blocks per range, at most two waves of
// CTAs so that the fp32 partials stay small next to the work) that minimises
// the number of CTA waves per unit of work, ceil(ctas*s / SMs) / s; kept at 1
// unless that saves at least 10 %.
int auto_splits(const Problem &p, int sm_count) {
  const int64_t ctas = base_ctas(p);
  const int64_t kblocks = (p.Nkv + 127) / 128;
  if (ctas >= sm_count || kblocks < 4) return 1;
  const int64_t smax = (2 * (int64_t)sm_count) / ctas;
  int best = 1;
  double best_cost = 1.0;
  for (int s = 2; s <= 16 && s <= smax && kblocks / s >= 2; ++s) {
    const double cost = (double)((ctas * s + sm_count - 1) / sm_count) / s;
    if (cost < best_cost * 0.9 - 1e-12 || (cost < best_cost - 1e-12 && best > 1)) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// splits: 0 = choose automatically, otherwise the caller's count.
void make_plan(const Problem &p, const DeviceInfo &dev, int splits, attn_plan *plan) {
  memset(plan, 0, sizeof(*plan));
  plan->kv_splits = 1;
  plan->d_slices = 1;
  if (p.B == 0 || p.Nq == 0) {
    plan->path = ATTN_PATH_NONE;
    return;
  }
  if (p.Nkv == 0) {  // no keys: every row is O = 0, LSE = -inf
    plan->path = ATTN_PATH_NOKEYS;
    plan->launches = 1;
    const int64_t blocks = ((int64_t)p.B * p.Hq * p.Nq * (p.D / 8) + 255) / 256;
    plan->grid = (int)(blocks < (int64_t)dev.sm_count * 8 ? (blocks < 1 ? 1 : blocks) : (int64_t)dev.sm_count * 8);
    return;
  }
  const int s = splits > 0 ? splits : auto_splits(p, dev.sm_count);
  plan->kv_splits = s;
  plan->d_slices = tc2_supports(p.D) ? 1 : d_slices(p.D);
  plan->grid = (int)(base_ctas(p) * s);
  if (s == 1) {
    plan->path = ATTN_PATH_TC;
    plan->launches = 1;
  } else {
    plan->path = ATTN_PATH_TC_SPLITKV;
    plan->launches = 2;
    plan->workspace_bytes = (long long)s * p.B * p.Hq * (long long)p.Nq * (p.D + 1) * 4;
  }
}

// Split-KV workspace on `st`: from the device's library pool (created on
// first use, outside stream capture), or with cudaMallocAsync while `st` is
// being captured into a graph (a graph memory node).
cudaError_t workspace_alloc(const DeviceInfo &dev_c, void **ptr, size_t bytes, cudaStream_t st) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) return e;
  if (cap != cudaStreamCaptureStatusNone) return cudaMallocAsync(ptr, bytes, st);
  DeviceInfo &dev = const_cast<DeviceInfo &>(dev_c);
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!dev.ws_pool) {
      cudaMemPoolProps props;
      memset(&props, 0, sizeof(props));
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev.device;
      cudaMemPool_t pool = nullptr;
      if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return e;
      uint64_t keep = ~0ull;
      if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
        cudaMemPoolDestroy(pool);
        return e;
      }
      dev.ws_pool = pool;
    }
  }
  return cudaMallocFromPoolAsync(ptr, bytes, dev.ws_pool, st);
}

int launch_plan(Problem &p, const DeviceInfo &dev, const attn_plan &plan, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  switch (plan.path) {
    case ATTN_PATH_NONE:
      return ATTN_OK;
    case ATTN_PATH_NOKEYS:
      p.kv_splits = 1;
      e = launch_nokeys(p, dev.sm_count, st);
      break;
    case ATTN_PATH_TC:
      p.kv_splits = 1;
      e = launch_tensor(p, dev.device, st);
      break;
    case ATTN_PATH_TC_SPLITKV: {
      // stream-ordered workspace: allocated and freed on the caller's stream
      void *ws = nullptr;
      if (workspace_alloc(dev, &ws, (size_t)plan.workspace_bytes, st) != cudaSuccess || !ws) {
        cudaGetLastError();
        return ATTN_ERR_NOMEM;
      }
      const int64_t rows = (int64_t)p.B * p.Hq * p.Nq;
      p.kv_splits = plan.kv_splits;
      p.ws_o = static_cast<float *>(ws);
      p.ws_lse = p.ws_o + (int64_t)plan.kv_splits * rows * p.D;
      e = launch_tensor(p, dev.device, st);
      if (e == cudaSuccess) e = launch_combine(p, st);
      cudaError_t f = cudaFreeAsync(ws, st);
      if (e == cudaSuccess) e = f;
      break;
    }
    default:
      return ATTN_ERR_ARG;
  }
  if (e != cudaSuccess) return record(e);
  return ATTN_OK;
}

}  // namespace

// For other translation units of the library: the current device's facts
// (same per-device cache and checks as attn_fwd) and the last-error record.
int current_device(int *device, int *sm_count, int **status) {
  DeviceInfo *d = nullptr;
  const int rc = device_info(&d);
  if (rc != ATTN_OK) return rc;
  *device = d->device;
  *sm_count = d->sm_count;
  *status = d->status;
  return ATTN_OK;
}

int record_cuda_error(cudaError_t e) { return record(e); }

cudaError_t scratch_alloc(void **ptr, size_t bytes, cudaStream_t st) {
  DeviceInfo *d = nullptr;
  if (device_info(&d) != ATTN_OK) return cudaErrorInvalidDevice;
  return workspace_alloc(*d, ptr, bytes, st);
}

// The tensor-core kernel for the head dim: two-tile (D 64, 128), cluster
// Split-D (D 384 ... 1024), else the Split-D kernel with per-slice scores.
cudaError_t launch_tensor(const Problem &p, int device, cudaStream_t st) {
  if (tc2_supports(p.D)) return launch_tc2(p, device, wait_limit_ns(), st);
  if (tcx_supports(p.D) && !(debug_flags() & ATTN_DEBUG_NO_CLUSTER)) {
    const cudaError_t e = launch_tcx(p, device, wait_limit_ns(), st);
    if (e != cudaErrorNotSupported) return e;  // else no room for the cluster: per-slice kernel
  }
  return launch_tc(p, device, wait_limit_ns(), st);
}

int check_problem(int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal) {
  return check_sizes(B, Hq, Hkv, Nq, Nkv, D, causal);
}

uint64_t wait_limit_ns() { return (uint64_t)g_wait_limit_ns.load(std::memory_order_relaxed); }
int debug_flags() { return g_debug_flags.load(std::memory_order_relaxed); }

}  // namespace attn

extern "C" {

int attn_version(void) { return 100; /* 0.1.0 */ }

int attn_shutdown(void) {
  int cur = 0;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return attn::record(e);
  cudaError_t first = cudaSuccess;
  for (int dev = 0; dev < attn::kMaxDevices; ++dev) {
    cudaMemPool_t pool = nullptr;
    {
      std::lock_guard<std::mutex> lock(attn::g_dev_mu);
      pool = attn::g_dev[dev].ws_pool;
    }
    if (!pool) continue;
    // every stream-ordered free has completed once the device is idle
    if ((e = cudaSetDevice(dev)) == cudaSuccess && (e = cudaDeviceSynchronize()) == cudaSuccess)
      e = cudaMemPoolTrimTo(pool, 0);
    if (first == cudaSuccess) first = e;
  }
  e = attn::release_host_copy_memory();
  if (first == cudaSuccess) first = e;
  e = cudaSetDevice(cur);
  if (first == cudaSuccess) first = e;
  return first == cudaSuccess ? ATTN_OK : attn::record(first);
}

const char *attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_ARG: return "invalid argument (null pointer, bad size, Hq % Hkv != 0, unsupported D or non-finite scale)";
    case ATTN_ERR_ALIGN: return "tensor base address not 16-byte aligned";
    case ATTN_ERR_ARCH: return "current device is not an sm_103 (compute capability 10.3) GPU";
    case ATTN_ERR_LAUNCH: return "CUDA error (see attn_last_cuda_error)";
    case ATTN_ERR_TIMEOUT: return "a bounded device-side wait ran out; outputs undefined";
    case ATTN_ERR_NOMEM: return "could not allocate the split-KV workspace";
    case ATTN_ERR_DEVICE: return "a kernel consistency check failed; outputs undefined";
    case ATTN_ERR_SCRATCH: return "split-KV partials larger than the fixed scratch of attn_fwd_splitkv_noalloc";
    default: return "unknown attn error code";
  }
}

const char *attn_last_cuda_error(void) { return attn::t_last_error; }

int attn_set_debug(int flags, long long wait_limit_ns) {
  if (flags & ~(ATTN_DEBUG_DROP_V_COPY | ATTN_DEBUG_NO_CLUSTER | ATTN_DEBUG_HOST_CHUNKS)) return ATTN_ERR_ARG;
  if (wait_limit_ns < 0) return ATTN_ERR_ARG;
  attn::g_debug_flags.store(flags);
  attn::g_wait_limit_ns.store(wait_limit_ns == 0 ? (long long)attn::kWaitLimitNs : wait_limit_ns);
  return ATTN_OK;
}

}  // extern "C"

namespace attn {
namespace {

// attn_fwd_splitkv and attn_fwd_masked: checks, problem description, plan,
// launch.  mask == nullptr: no additive mask.
int fwd_common(const void *q, const void *k, const void *v, const void *mask, long long msb, long long msh,
               long long msq, void *o, float *lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D, float scale,
               int causal, int kv_splits, attn_stream_t stream) {
  int rc = check_sizes(B, Hq, Hkv, Nq, Nkv, D, causal);
  if (rc != ATTN_OK) return rc;
  if (!isfinite(scale) || kv_splits < 0 || kv_splits > kMaxSplits) return ATTN_ERR_ARG;
  if (B == 0 || Nq == 0) return ATTN_OK;
  if (!q || !o || !lse) return ATTN_ERR_ARG;
  if (Nkv > 0 && (!k || !v)) return ATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_ALIGN;
  if (Nkv > 0 && (!aligned16(k) || !aligned16(v))) return ATTN_ERR_ALIGN;
  if (mask && Nkv > 0 && !aligned16(mask)) return ATTN_ERR_ALIGN;

  DeviceInfo *dev = nullptr;
  rc = device_info(&dev);
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
  p.status = dev->status;
  p.kv_splits = 1;
  p.debug_flags = debug_flags();
  if (mask && Nkv > 0) {  // without keys the mask has nothing to act on
    p.mask = static_cast<const __nv_bfloat16 *>(mask);
    p.mask_sb = msb;
    p.mask_sh = msh;
    p.mask_sq = msq;
  }

  attn_plan plan;
  make_plan(p, *dev, kv_splits, &plan);
  return launch_plan(p, *dev, plan, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace attn

extern "C" {

int attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                     float scale, int causal, int kv_splits, attn_stream_t stream) {
  return attn::fwd_common(q, k, v, nullptr, 0, 0, 0, o, lse, B, Hq, Hkv, Nq, Nkv, D, scale, causal, kv_splits,
                          stream);
}

int attn_fwd_masked(const void *q, const void *k, const void *v, const void *mask, long long mask_stride_b,
                    long long mask_stride_h, long long mask_stride_q, void *o, float *lse, int B, int Hq, int Hkv,
                    int Nq, int Nkv, int D, float scale, int causal, attn_stream_t stream) {
  if (!mask) return ATTN_ERR_ARG;
  if (mask_stride_b < 0 || mask_stride_h < 0 || mask_stride_q < 0) return ATTN_ERR_ARG;
  if (mask_stride_b % 8 || mask_stride_h % 8 || mask_stride_q % 8) return ATTN_ERR_ALIGN;
  return attn::fwd_common(q, k, v, mask, mask_stride_b, mask_stride_h, mask_stride_q, o, lse, B, Hq, Hkv, Nq, Nkv,
                          D, scale, causal, 0, stream);
}

int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int Hq, int Hkv, int Nq, int Nkv, int D,
             float scale, int causal, attn_stream_t stream) {
  return attn_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, D, scale, causal, 0, stream);
}

int attn_fwd_plan(int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, attn_plan *plan) {
  using namespace attn;
  if (!plan) return ATTN_ERR_ARG;
  int rc = check_sizes(B, Hq, Hkv, Nq, Nkv, D, causal);
  if (rc != ATTN_OK) return rc;
  DeviceInfo *dev = nullptr;
  rc = device_info(&dev);
  if (rc != ATTN_OK) return rc;
  Problem p{};
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = Nq; p.Nkv = Nkv; p.D = D; p.causal = causal;
  make_plan(p, *dev, 0, plan);
  return ATTN_OK;
}

int attn_fwd_status(attn_stream_t stream) {
  using namespace attn;
  DeviceInfo *dev = nullptr;
  int rc = device_info(&dev);
  if (rc != ATTN_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record(e);
  int h = 0;
  if ((e = cudaMemcpy(&h, dev->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return record(e);
  if (h != 0) {
    const int zero = 0;
    if ((e = cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess) return record(e);
  }
  return h;
}

}  // extern "C"
