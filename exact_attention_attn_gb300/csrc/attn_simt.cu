// Exact attention forward on CUDA cores (fp32 FMA), one online-softmax pass.
//
// The algorithm is the tiled online softmax of "FlashAttention v1/v2/v3/v4"
// (lo0.es), section "El truco que hizo posible todo: online softmax": keys are
// visited in tiles, each row keeps a running max m and a running sum l, the
// partial output is rescaled by 2^(m_old - m_new) when the max grows, and the
// output is divided by l at the end.  Scores never leave the chip.
//
// Work split: a CTA of 256 threads owns 64 query rows of one (b, hq) head and
// one slice of at most 256 output columns (large head dims use several
// slices, each recomputing the scores: the D-slicing of the FFPA page's
// "Split-D and TiledMMA" section applied to the output).  Each warp owns 8
// rows; lane l holds the score of key j0+l for its 8 rows, and output columns
// lane + 32*c.
#include <math.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kRows = 64;      // query rows per CTA
constexpr int kKeys = 32;      // keys per tile
constexpr int kChunk = 32;     // head-dim chunk for the score contraction
constexpr int kSlice = 256;    // output columns per CTA
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(kThreads) attn_simt_kernel(Problem p) {
  __shared__ float sq[kRows][kChunk];
  __shared__ float sk[kKeys][kChunk + 1];
  __shared__ float sv[kKeys][kSlice];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // 1-D grid: slice fastest, then query tile, then (b, hq)
  const int nslices = (p.D + kSlice - 1) / kSlice;
  const int ntiles = (p.Nq + kRows - 1) / kRows;
  const int64_t bid = blockIdx.x;
  const int slice = (int)(bid % nslices);
  const int tile = (int)((bid / nslices) % ntiles);
  const int bh = (int)(bid / ((int64_t)nslices * ntiles));
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int kvh = hq / (p.Hq / p.Hkv);
  const int q0 = tile * kRows;
  const int c0 = slice * kSlice;
  const int D = p.D;
  const int ncols = min(kSlice, D - c0);

  const __nv_bfloat16 *qb = p.q + ((int64_t)b * p.Hq + hq) * (int64_t)p.Nq * D;
  const __nv_bfloat16 *kb = p.k + ((int64_t)b * p.Hkv + kvh) * (int64_t)p.Nkv * D;
  const __nv_bfloat16 *vb = p.v + ((int64_t)b * p.Hkv + kvh) * (int64_t)p.Nkv * D;

  const int shift = p.Nkv - p.Nq;  // bottom-right causal alignment
  int kv_end = p.Nkv;
  if (p.causal) kv_end = max(0, min(p.Nkv, q0 + kRows - 1 + shift + 1));

  const float sl2 = p.scale * kLog2e;
  float m[8], l[8], acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[i][c] = 0.f;
  }

  for (int j0 = 0; j0 < kv_end; j0 += kKeys) {
    float s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = 0.f;
    for (int d0 = 0; d0 < D; d0 += kChunk) {
      __syncthreads();
      for (int e = tid; e < kRows * kChunk; e += kThreads) {
        const int r = e / kChunk, c = e % kChunk, qi = q0 + r;
        sq[r][c] = qi < p.Nq ? __bfloat162float(qb[(int64_t)qi * D + d0 + c]) : 0.f;
      }
      for (int e = tid; e < kKeys * kChunk; e += kThreads) {
        const int r = e / kChunk, c = e % kChunk, kj = j0 + r;
        sk[r][c] = kj < p.Nkv ? __bfloat162float(kb[(int64_t)kj * D + d0 + c]) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int c = 0; c < kChunk; ++c) {
        const float kk = sk[lane][c];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i] = fmaf(sq[warp * 8 + i][c], kk, s[i]);
      }
    }
    // mask, running max, rescale
    const int kj = j0 + lane;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int qi = q0 + warp * 8 + i;
      const bool vis = kj < p.Nkv && (!p.causal || kj <= qi + shift);
      const float x = vis ? s[i] * sl2 : -INFINITY;
      const float mnew = fmaxf(m[i], warp_max(x));
      const float muse = (mnew == -INFINITY) ? 0.f : mnew;
      const float alpha = exp2f(m[i] - muse);
      const float pe = exp2f(x - muse);
      l[i] = l[i] * alpha + pe;
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[i][c] *= alpha;
      m[i] = mnew;
      s[i] = pe;
    }
    __syncthreads();
    for (int e = tid; e < kKeys * kSlice; e += kThreads) {
      const int r = e / kSlice, c = e % kSlice, kj2 = j0 + r;
      sv[r][c] = (kj2 < p.Nkv && c < ncols) ? __bfloat162float(vb[(int64_t)kj2 * D + c0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < kKeys; ++j) {
      float pj[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) pj[i] = __shfl_sync(0xffffffffu, s[i], j);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float vv = sv[j][lane + 32 * c];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i][c] = fmaf(pj[i], vv, acc[i][c]);
      }
    }
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int qi = q0 + warp * 8 + i;
    const float L = warp_sum(l[i]);
    if (qi >= p.Nq) continue;
    const bool live = m[i] != -INFINITY;
    const float inv = live ? 1.f / L : 0.f;
    __nv_bfloat16 *orow = p.o + (((int64_t)b * p.Hq + hq) * p.Nq + qi) * D + c0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int col = lane + 32 * c;
      if (col < ncols) orow[col] = __float2bfloat16_rn(acc[i][c] * inv);
    }
    if (slice == 0 && lane == 0)
      p.lse[((int64_t)b * p.Hq + hq) * p.Nq + qi] = live ? (m[i] + log2f(L)) * kLn2 : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_simt(const Problem &p, cudaStream_t stream) {
  const int64_t blocks = (int64_t)((p.Nq + kRows - 1) / kRows) * p.B * p.Hq * ((p.D + kSlice - 1) / kSlice);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  attn_simt_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
