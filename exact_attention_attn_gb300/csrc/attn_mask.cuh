// Additive attention mask (the "Causal/Mask" feature of the FFPA README's
// feature table, read as SDPA's float mask): a bf16 value per (b, hq, query
// row, key) is added to the scaled score before the row maximum; -inf hides
// the key.  In the kernels' base-2 units the score of key j becomes
//     y_j = s_j * (scale * log2 e) + mask_j * log2 e.
//
// Ways to bring a row's values of one key block on chip:
//   - mask_load<NV>: NV values straight into NV / 2 registers (bf16 pairs),
//     issued before the thread waits for its scores so that the load latency
//     hides behind that wait;
//   - mask_stage128: cp.async into shared memory, 16 chunks of 8 values laid
//     out chunk-major ([16][nrows][16 bytes]) so that a warp's 16-byte reads
//     of one chunk are contiguous; for kernels whose registers are taken.
// Values at keys >= Nkv, and every value of a row >= Nq, are zero and never
// read from memory (those keys and rows are masked or discarded anyway).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "attn_internal.h"
#include "sm100_ptx.cuh"

namespace attn {

// Start of the mask row of (b, hq, query row qi), or null when the problem
// has no mask or the row lies past Nq.
__device__ __forceinline__ const __nv_bfloat16 *mask_row(const Problem &p, int b, int hq, int qi) {
  if (p.mask == nullptr || qi >= p.Nq) return nullptr;
  return p.mask + (int64_t)b * p.mask_sb + (int64_t)hq * p.mask_sh + (int64_t)qi * p.mask_sq;
}

// Low and high bf16 of a packed pair, as floats (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// mk[i] = values of keys kbase + 2i, kbase + 2i + 1, i < NV / 2 (zero where
// the key is >= nkv or row is null).  Whole 16-byte vectors are loaded where
// they lie below nkv, the one ragged vector value by value.
template <int NV>
__device__ __forceinline__ void mask_load(uint32_t (&mk)[NV / 2], const __nv_bfloat16 *row, int kbase, int nkv) {
  const int n = row ? nkv - kbase : 0;  // valid values from kbase on
  if (n >= NV) {  // every value below nkv: plain vector loads
    const uint4 *src = reinterpret_cast<const uint4 *>(row + kbase);
#pragma unroll
    for (int v = 0; v < NV / 8; ++v) {
      const uint4 w = __ldg(src + v);
      mk[4 * v + 0] = w.x;
      mk[4 * v + 1] = w.y;
      mk[4 * v + 2] = w.z;
      mk[4 * v + 3] = w.w;
    }
    return;
  }
#pragma unroll
  for (int v = 0; v < NV / 8; ++v) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (8 * v + 8 <= n) {
      w = __ldg(reinterpret_cast<const uint4 *>(row + kbase + 8 * v));
    } else if (8 * v < n) {
      uint32_t e[4] = {0u, 0u, 0u, 0u};
      const unsigned short *src = reinterpret_cast<const unsigned short *>(row + kbase + 8 * v);
      for (int t = 0; t < n - 8 * v; ++t) e[t >> 1] |= (uint32_t)__ldg(src + t) << (16 * (t & 1));
      w = make_uint4(e[0], e[1], e[2], e[3]);
    }
    mk[4 * v + 0] = w.x;
    mk[4 * v + 1] = w.y;
    mk[4 * v + 2] = w.z;
    mk[4 * v + 3] = w.w;
  }
}

// cp.async of the same 128 values into shared memory at dst (byte address),
// chunk c of row r at dst + (c * nrows + r) * 16; commits one group.  A null
// row zero-fills its chunks without reading memory (src_bytes 0, with the
// source pointing at `fallback`, any valid global address).
__device__ __forceinline__ void mask_stage128(uint32_t dst, int nrows, int r, const __nv_bfloat16 *row, int kbase,
                                              int nkv, const void *fallback) {
  const int n = row ? nkv - kbase : 0;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const int have = n - 8 * c;  // values of this chunk below nkv
    const uint32_t bytes = have >= 8 ? 16u : (have > 0 ? (uint32_t)have * 2u : 0u);
    const void *src = bytes ? static_cast<const void *>(row + kbase + 8 * c) : fallback;
    ptx::cp_async16(dst + (uint32_t)((c * nrows + r) * 16), src, bytes);
  }
  ptx::cp_async_commit();
}

}  // namespace attn
