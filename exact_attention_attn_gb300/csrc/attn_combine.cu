// Split-KV combine: merges the partial results that several CTAs computed over
// disjoint key ranges of the same query rows.
//
// The merge is the one the ZYFA page relies on for chunked prefill ("The
// details that make it production-grade": log-sum-exp values let results over
// different key ranges merge consistently): with partial outputs O_s
// (normalised within their range) and natural-log partial LSE_s,
//     LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) * O_s.
// Ranges in which a row saw no key carry LSE_s = -inf and weigh nothing; a row
// that saw no key anywhere gets O = 0, LSE = -inf.
//
// Memory-bound: each thread owns 8 consecutive output columns of one row, so
// a warp reads 32 contiguous 32-byte segments per split and writes 16-byte
// bf16 vectors.
#include <math.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) attn_combine_kernel(Problem p) {
  const int D = p.D;
  const int chunks = D / 8;
  const int64_t rows = (int64_t)p.B * p.Hq * p.Nq;
  const int64_t gid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t row = gid / chunks;
  const int c8 = (int)(gid % chunks);
  if (row >= rows) return;
  const int S = p.kv_splits;

  float m = -INFINITY;
  for (int s = 0; s < S; ++s) m = fmaxf(m, p.ws_lse[(int64_t)s * rows + row]);

  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  float tot = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float ls = p.ws_lse[(int64_t)s * rows + row];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - m);
      tot += w;
      const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + ((int64_t)s * rows + row) * D + c8 * 8);
      const float4 a = src[0], b = src[1];
      acc[0] = fmaf(w, a.x, acc[0]);
      acc[1] = fmaf(w, a.y, acc[1]);
      acc[2] = fmaf(w, a.z, acc[2]);
      acc[3] = fmaf(w, a.w, acc[3]);
      acc[4] = fmaf(w, b.x, acc[4]);
      acc[5] = fmaf(w, b.y, acc[5]);
      acc[6] = fmaf(w, b.z, acc[6]);
      acc[7] = fmaf(w, b.w, acc[7]);
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  __nv_bfloat162 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
  *reinterpret_cast<uint4 *>(p.o + row * D + c8 * 8) = *reinterpret_cast<const uint4 *>(h);
  if (c8 == 0) p.lse[row] = (tot > 0.f) ? m + logf(tot) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const Problem &p, cudaStream_t stream) {
  const int64_t threads = (int64_t)p.B * p.Hq * p.Nq * (p.D / 8);
  const int64_t blocks = (threads + kThreads - 1) / kThreads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  attn_combine_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
