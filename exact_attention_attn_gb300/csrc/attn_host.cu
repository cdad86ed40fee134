// attn_fwd_host: the attention forward of attn_fwd on host buffers, with the
// host<->device copies overlapped with the kernels.
//
// The (b, kv-head) groups of a problem are independent attention problems, and
// each group's rows are contiguous in the [B, H, N, D] layouts: Q, O and LSE
// planes g*G .. g*G + G - 1 (G = Hq / Hkv query heads per kv head), K and V
// plane g.  The groups are cut into chunks of about kChunkBytes of inputs (at
// most kMaxChunks, at most one per group); chunk c's inputs go up on one
// copy stream, its kernels run on a compute stream of its own once they have
// landed, and its outputs come back on a second copy stream, so that the
// copies of one chunk overlap the kernels and copies of the others, and the
// kernels of chunks too small to fill the GPU run side by side.  Every chunk
// uses the key split count of the whole problem, and each (b, h) row tile is
// computed by the same kernel code as in attn_fwd: the results are
// bit-identical to attn_fwd.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "attn.h"
#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kMaxDev = 64;
// About 25 MiB of inputs per chunk, at most 8 chunks: measured on GB300 with
// pinned buffers, causal B4 H16 N2048 D128 (100 MB of inputs) ran fastest in
// 4 chunks (0.69 ms; 8 chunks 0.72, 16 chunks 0.81) and GQA causal B2 Hq32
// Hkv8 N8192 D128 (201 MB) in 8 (1.45 ms; 4 chunks 1.55, 16 chunks 1.59):
// past that the uploads of later chunks and the downloads of earlier ones
// share the host link, and the last chunk's inputs land no sooner.
constexpr int kMaxChunks = 8;
constexpr size_t kChunkBytes = (size_t)25 << 20;

struct CopyStreams {
  cudaStream_t in = nullptr, out = nullptr;
  cudaStream_t k[kMaxChunks] = {};  // chunk c's kernels
  // the call's events, created once: a call waits for all of them before it
  // returns, so the next call may record them again
  cudaEvent_t ev_start = nullptr, ev_out = nullptr, ev_indone = nullptr, ev_in[kMaxChunks] = {}, ev_k[kMaxChunks] = {};
  // the library's own pool for the device copies: it keeps its memory between
  // calls (the default pool hands it back to the driver at every synchronise,
  // and a 100 MB block from the driver costs more than the copies it serves)
  cudaMemPool_t pool = nullptr;
};
CopyStreams g_copy[kMaxDev];
std::mutex g_copy_mu[kMaxDev];

}  // namespace

cudaError_t release_host_copy_memory() {
  cudaError_t first = cudaSuccess;
  for (int dev = 0; dev < kMaxDev; ++dev) {
    std::lock_guard<std::mutex> lock(g_copy_mu[dev]);
    if (!g_copy[dev].pool) continue;
    cudaError_t e = cudaSetDevice(dev);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemPoolTrimTo(g_copy[dev].pool, 0);
    if (first == cudaSuccess) first = e;
  }
  return first;
}

}  // namespace attn

extern "C" int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                             int Hkv, int Nq, int Nkv, int D, float scale, int causal, attn_stream_t stream) {
  using namespace attn;
  // the argument checks of attn_fwd, all on the host before any device work
  int rc = check_problem(B, Hq, Hkv, Nq, Nkv, D, causal);
  if (rc != ATTN_OK) return rc;
  if (!isfinite(scale)) return ATTN_ERR_ARG;
  if (B == 0 || Nq == 0) return ATTN_OK;
  if (!q || !o || !lse || (Nkv > 0 && (!k || !v))) return ATTN_ERR_ARG;
  attn_plan plan;  // the key split count of the whole problem
  if ((rc = attn_fwd_plan(B, Hq, Hkv, Nq, Nkv, D, causal, &plan)) != ATTN_OK) return rc;
  int device = 0, sms = 0, *status = nullptr;
  if ((rc = current_device(&device, &sms, &status)) != ATTN_OK) return rc;
  if (device < 0 || device >= kMaxDev) return ATTN_ERR_ARCH;

  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int grp = Hq / Hkv, groups = B * Hkv;
  const size_t qplane = (size_t)Nq * D * 2, kvplane = (size_t)Nkv * D * 2, lplane = (size_t)Nq * 4;
  const size_t qbytes = (size_t)B * Hq * qplane, kvbytes = (size_t)B * Hkv * kvplane;
  int chunks = (debug_flags() & ATTN_DEBUG_HOST_CHUNKS) ? kMaxChunks
                                                         : (int)((qbytes + 2 * kvbytes + kChunkBytes - 1) / kChunkBytes);
  if (chunks > kMaxChunks) chunks = kMaxChunks;
  if (chunks > groups) chunks = groups;
  if (chunks < 1) chunks = 1;

  std::lock_guard<std::mutex> lock(g_copy_mu[device]);
  CopyStreams &cs = g_copy[device];
  cudaError_t e = cudaSuccess;
  if (!cs.in && (e = cudaStreamCreateWithFlags(&cs.in, cudaStreamNonBlocking)) != cudaSuccess)
    return record_cuda_error(e);
  if (!cs.out && (e = cudaStreamCreateWithFlags(&cs.out, cudaStreamNonBlocking)) != cudaSuccess)
    return record_cuda_error(e);
  for (int c = 0; c < chunks; ++c)
    if (!cs.k[c] && (e = cudaStreamCreateWithFlags(&cs.k[c], cudaStreamNonBlocking)) != cudaSuccess)
      return record_cuda_error(e);
  if (!cs.pool) {
    cudaMemPoolProps props;
    memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = device;
    if ((e = cudaMemPoolCreate(&cs.pool, &props)) != cudaSuccess) {
      cs.pool = nullptr;
      return record_cuda_error(e);
    }
    uint64_t keep = ~0ull;
    if ((e = cudaMemPoolSetAttribute(cs.pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess)
      return record_cuda_error(e);
  }

  // device buffers, stream-ordered on the caller's stream (one block, 256-byte
  // aligned pieces; each chunk's LSE rows in a piece of their own, so that
  // every chunk's LSE starts aligned whatever Nq is)
  auto up = [](size_t n) { return (n + 255) & ~(size_t)255; };
  auto g0 = [&](int c) { return (int)((int64_t)groups * c / chunks); };
  const size_t off_k = up(qbytes), off_v = off_k + up(kvbytes), off_o = off_v + up(kvbytes);
  size_t off_l[kMaxChunks + 1];
  off_l[0] = off_o + up(qbytes);
  for (int c = 0; c < chunks; ++c) off_l[c + 1] = off_l[c] + up((size_t)(g0(c + 1) - g0(c)) * grp * lplane);
  const size_t total = off_l[chunks];
  char *buf = nullptr;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void **>(&buf), total, cs.pool, st) != cudaSuccess || !buf) {
    cudaGetLastError();
    return ATTN_ERR_NOMEM;
  }
  auto make_event = [&](cudaEvent_t *ev) {
    if (e == cudaSuccess && !*ev) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  };
  make_event(&cs.ev_start);
  make_event(&cs.ev_out);
  make_event(&cs.ev_indone);
  for (int c = 0; c < chunks; ++c) {
    make_event(&cs.ev_in[c]);
    make_event(&cs.ev_k[c]);
  }
  cudaEvent_t ev_start = cs.ev_start, ev_out = cs.ev_out, ev_indone = cs.ev_indone;
  cudaEvent_t *ev_in = cs.ev_in, *ev_k = cs.ev_k;
  // the copy streams start after the allocation on the caller's stream
  if (e == cudaSuccess) e = cudaEventRecord(ev_start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.in, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, ev_start, 0);

  // inputs, chunk by chunk
  for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
    const int a = g0(c), n = g0(c + 1) - a;
    const size_t qo = (size_t)a * grp * qplane, qn = (size_t)n * grp * qplane;
    const size_t ko = (size_t)a * kvplane, kn = (size_t)n * kvplane;
    e = cudaMemcpyAsync(buf + qo, static_cast<const char *>(q) + qo, qn, cudaMemcpyHostToDevice, cs.in);
    if (e == cudaSuccess && kn)
      e = cudaMemcpyAsync(buf + off_k + ko, static_cast<const char *>(k) + ko, kn, cudaMemcpyHostToDevice, cs.in);
    if (e == cudaSuccess && kn)
      e = cudaMemcpyAsync(buf + off_v + ko, static_cast<const char *>(v) + ko, kn, cudaMemcpyHostToDevice, cs.in);
    if (e == cudaSuccess) e = cudaEventRecord(ev_in[c], cs.in);
  }
  // kernels and outputs, chunk by chunk (chunk c's kernels, and the split-KV
  // workspace they may take, on compute stream c)
  int launched = 0;
  for (int c = 0; c < chunks && e == cudaSuccess && rc == ATTN_OK; ++c) {
    const int a = g0(c), n = g0(c + 1) - a;
    const size_t qo = (size_t)a * grp * qplane, qn = (size_t)n * grp * qplane;
    const size_t ko = (size_t)a * kvplane, lo = (size_t)a * grp * lplane, ln = (size_t)n * grp * lplane;
    float *dl = reinterpret_cast<float *>(buf + off_l[c]);
    e = cudaStreamWaitEvent(cs.k[c], ev_in[c], 0);
    if (e != cudaSuccess) break;
    launched = c + 1;
    rc = attn_fwd_splitkv(buf + qo, buf + off_k + ko, buf + off_v + ko, buf + off_o + qo, dl, 1, n * grp, n, Nq,
                          Nkv, D, scale, causal, plan.kv_splits, reinterpret_cast<attn_stream_t>(cs.k[c]));
    if (rc != ATTN_OK) break;
    e = cudaEventRecord(ev_k[c], cs.k[c]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, ev_k[c], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(static_cast<char *>(o) + qo, buf + off_o + qo, qn, cudaMemcpyDeviceToHost, cs.out);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(reinterpret_cast<char *>(lse) + lo, dl, ln, cudaMemcpyDeviceToHost, cs.out);
  }
  // the buffers are freed after every copy and kernel on the library's streams
  // (also when a step above failed: then, if the streams cannot be ordered by
  // events, by waiting for them); the call returns when the outputs are in
  // host memory
  bool ordered = ev_indone && ev_out && cudaEventRecord(ev_indone, cs.in) == cudaSuccess &&
                 cudaEventRecord(ev_out, cs.out) == cudaSuccess &&
                 cudaStreamWaitEvent(st, ev_indone, 0) == cudaSuccess &&
                 cudaStreamWaitEvent(st, ev_out, 0) == cudaSuccess;
  for (int c = 0; c < launched && ordered; ++c)
    ordered = ev_k[c] && cudaEventRecord(ev_k[c], cs.k[c]) == cudaSuccess &&
              cudaStreamWaitEvent(st, ev_k[c], 0) == cudaSuccess;
  if (!ordered) {
    cudaStreamSynchronize(cs.in);
    cudaStreamSynchronize(cs.out);
    for (int c = 0; c < launched; ++c) cudaStreamSynchronize(cs.k[c]);
  }
  cudaError_t f = cudaFreeAsync(buf, st);
  const cudaError_t fs = cudaStreamSynchronize(st);
  if (f == cudaSuccess) f = fs;
  if (e == cudaSuccess) e = f;
  if (rc != ATTN_OK) return rc;
  if (e != cudaSuccess) return record_cuda_error(e);
  return ATTN_OK;
}
