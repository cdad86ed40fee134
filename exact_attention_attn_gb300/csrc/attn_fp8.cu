// FP8 (e4m3) attention forward for head dim 128 on the sm_103a tensor cores
// (tcgen05.mma kind::f8f6f4), and the quantisation that feeds it.
//
// The FP8 scheme follows two pages: "FlashAttention v1/v2/v3/v4" (lo0.es),
// "FA3 -- el momento Hopper": Q and K quantised with one scale per tile of
// rows, after a Hadamard-based orthogonal rotation that spreads outliers;
// and "ZYFA: FP8 FlashAttention Kernels for AMD MI355X": a Hadamard rotation
// of Q and K before quantisation, power-of-two descales, and probabilities
// multiplied by a power of two before they are rounded to FP8 ("The three
// techniques", per-block scaling).  Concretely:
//
//   quantisation (attn_fp8_quantize):
//     Q, K: each row rotated by H / sqrt(128) (H the Sylvester Hadamard
//       matrix; the fast transform in registers and warp shuffles, float32,
//       butterflies of stride 1, 2, ..., 64), then per 128-row block of one
//       head the scale s = 2^k, k the smallest integer with max|x| <= 448 2^k,
//       and the codes e4m3(x / s);
//     V: one such scale per (b, kv head) over all its values, codes stored
//       transposed ([128 head-dim rows x keys], keys contiguous, rows padded
//       to a multiple of 128 keys with code 0) so that V enters the P V
//       product K-major.
//   attention (attn_fwd_fp8): the two-tile ping-pong of the bf16 kernel
//     (two 128-row query tiles per CTA sharing every K and V block), with
//     S = Q8 K8^T on kind::f8f6f4; the softmax works on s * (scale * sq *
//     sk * log2 e) (sq, sk the tile's and the block's scales); P is written
//     as 2^(y - m + 2) rounded to e4m3 (the factor 2^2 and the lazy rescale
//     threshold of 6.5 in log2 units keep it below 2^8.5 < 448; e4m3 rounds
//     relative to each value, so the factor moves only the few p below
//     2^-8 into subnormals, and the large threshold spares the O rescales
//     that a threshold of 0.5 with a factor 2^8 cost: 1450 -> 1719 TFLOP/s
//     on GQA causal N8192); O = sv * (P8 V8) / l with l the fp32 sum of the
//     same 2^(y - m + 2).
//
// Since (Q H)(K H)^T = Q K^T, the result approximates exact attention on
// the original inputs; it equals exact attention on the dequantised inputs
// up to the rounding of P to e4m3 and fp32 accumulation.
#include <limits.h>
#include <math.h>
#include <string.h>

#include <atomic>

#include "attn.h"
#include "attn_internal.h"
#include "sm100_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int HD = 128;                 // head dim of the FP8 path
constexpr int BM = 128, BN = 128;
constexpr int TILE = 128 * 128;         // one 128-row x 128-byte e4m3 tile
constexpr float kInvSqrtD = 0.08838834764831845f;  // 1/sqrt(128), rounded to float32
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float TAU = 6.5f;             // lazy rescale threshold, log2 units
constexpr float P_SHIFT = 2.f;          // P is stored as 2^2 p
constexpr int THREADS = 352;
constexpr int WARP_LOAD_K = 8, WARP_LOAD_V = 10, WARP_MMA = 9;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_KST = 8, MAX_VST = 4;
constexpr int kSmemMax = 232448;

// ---------------------------------------------------------------- quantisation

// k for the smallest integer k with amax <= 448 2^k; 0 when amax == 0.
// With amax = m 2^e, m in [0.5, 1), and 448 = 0.875 2^9: k = e - 9, plus one
// when m > 0.875.
__device__ __forceinline__ int pow2_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  int e;
  const float m = frexpf(amax, &e);
  return e - 9 + (m > 0.875f ? 1 : 0);
}
__device__ __forceinline__ float pow2_scale(float amax) { return ldexpf(1.f, pow2_exp(amax)); }

// x / 2^k exactly: a multiply by 2^-k where that is a normal float, else a
// division (inputs that small do not occur in practice).
struct InvPow2 {
  float s, inv;
  bool mul;
  __device__ __forceinline__ explicit InvPow2(int k) : s(ldexpf(1.f, k)), inv(ldexpf(1.f, -k)), mul(k > -126 && k < 126) {}
  __device__ __forceinline__ float operator()(float x) const { return mul ? x * inv : x / s; }
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Rotation and block quantisation of a [planes, N, 128] bf16 tensor: rotate
// every row, take the scale of each 128-row block, write the e4m3 codes
// [planes, N, 128] and the scales [planes, nblk].  The units (plane, block)
// are dealt to the CTAs round-robin; a CTA of 128 threads copies its next
// unit into the second of two shared-memory buffers while it works on the
// current one.  Thread t owns row t of a unit: the unit is copied with
// coalesced 16-byte copies (rows past N read as zeros), chunk c of row r at
//     r * 256 + (c / 8) * 128 + ((c % 8) ^ (r % 8)) * 16,
// so that 8 consecutive threads reading chunk c of their own rows touch all
// 32 banks once; every butterfly then runs in the thread's registers on
// packed fp32 pairs, and the codes leave through the same kind of layout with
// coalesced 16-byte stores.
// zero_bits (may be null): the CTA that takes block 0 of a plane also zeroes
// zero_bits[plane].
constexpr int ROW_THREADS = BM;
constexpr int ROW_CTAS_PER_SM = 3;
constexpr int ROW_BUF = BM * HD * 2;  // one unit of bf16 rows
constexpr int ROW_SMEM = 2 * ROW_BUF;

// Wait until at most the most recent cp.async group of this thread is pending.
__device__ __forceinline__ void cp_async_wait_all_but_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ void rows_copy(uint32_t buf, const uint8_t *src, int rows, int tid) {
#pragma unroll
  for (int j = 0; j < ROW_BUF / 16 / ROW_THREADS; ++j) {
    const int i = j * ROW_THREADS + tid, r = i >> 4, c = i & 15;  // chunk i = 16 r + c of the unit
    const bool in = r < rows;
    cp_async16(buf + r * 256 + (c >> 3) * 128 + (((c & 7) ^ (r & 7)) << 4), src + (in ? (int64_t)i * 16 : 0),
               in ? 16u : 0u);
  }
  cp_async_commit();
}

__global__ void __launch_bounds__(ROW_THREADS, ROW_CTAS_PER_SM)
    attn_fp8_rows_kernel(const __nv_bfloat16 *x, uint8_t *codes, float *scales, int N, int nblk, int nunits,
                         unsigned *zero_bits) {
  extern __shared__ __align__(128) uint8_t rows_smem[];
  __shared__ float wmax[ROW_THREADS / 32];
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t smem_s = smem_u32(rows_smem);
  const uint64_t kM1 = f2_pack(-1.f, -1.f), kNZ = f2_pack(-0.f, -0.f), kC = f2_pack(kInvSqrtD, kInvSqrtD);
  auto unit_rows = [&](int u) { return min(BM, N - (u % nblk) * BM); };  // >= 1: block < nblk
  auto unit_src = [&](int u) {
    return reinterpret_cast<const uint8_t *>(x + ((int64_t)(u / nblk) * N + (int64_t)(u % nblk) * BM) * HD);
  };
  int unit = blockIdx.x, buf = 0;
  if (unit < nunits) rows_copy(smem_s, unit_src(unit), unit_rows(unit), tid);
  for (; unit < nunits; unit += gridDim.x, buf ^= 1) {
    const int plane = unit / nblk, blk = unit % nblk, rows = unit_rows(unit);
    if (zero_bits && blk == 0 && tid == 0) zero_bits[plane] = 0u;
    const int next = unit + gridDim.x;
    if (next < nunits) {
      rows_copy(smem_s + (buf ^ 1) * ROW_BUF, unit_src(next), unit_rows(next), tid);
      cp_async_wait_all_but_1();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
    uint8_t *tb = rows_smem + buf * ROW_BUF;
    uint64_t p[HD / 2];  // p[j] = elements (2j, 2j + 1) of this thread's row
    const uint8_t *mine = tb + tid * 256;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 w = *reinterpret_cast<const uint4 *>(mine + (c >> 3) * 128 + (((c & 7) ^ (tid & 7)) << 4));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) p[4 * c + e] = f2_pack(__uint_as_float(ws[e] << 16), __uint_as_float(ws[e] & 0xffff0000u));
    }
    // butterflies of stride 1, 2, ..., 64 in that order: the lower element
    // keeps lo + hi, the upper lo - hi, each rounded once (stride 1 inside a
    // pair; from stride 2 on, two butterflies per packed add and fma(-1, hi, lo))
#pragma unroll
    for (int j = 0; j < HD / 2; ++j) {
      float lo, hi;
      f2_unpack(p[j], lo, hi);
      p[j] = f2_pack(__fadd_rn(lo, hi), __fsub_rn(lo, hi));
    }
#pragma unroll
    for (int h = 1; h < HD / 2; h <<= 1) {
#pragma unroll
      for (int j = 0; j < HD / 2; ++j) {
        if ((j & h) == 0) {
          const uint64_t lo = p[j], hi = p[j + h];
          p[j] = f2_add(lo, hi);
          p[j + h] = f2_fma(kM1, hi, lo);
        }
      }
    }
    // times 1/sqrt(D), rounded once (adding -0 keeps the sign of a zero product)
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < HD / 2; ++j) {
      p[j] = f2_fma(p[j], kC, kNZ);
      float lo, hi;
      f2_unpack(p[j], lo, hi);
      amax = max3f(amax, fabsf(lo), fabsf(hi));
    }
    amax = warp_max(amax);
    if ((tid & 31) == 0) wmax[warp] = amax;
    __syncthreads();  // also: every thread has read its row out of the buffer
    float a = wmax[0];
#pragma unroll
    for (int w = 1; w < ROW_THREADS / 32; ++w) a = fmaxf(a, wmax[w]);
    const InvPow2 d(pow2_exp(a));
    if (tid == 0) scales[(int64_t)plane * nblk + blk] = d.s;
    if (d.mul) {
      const uint64_t inv = f2_pack(d.inv, d.inv);
#pragma unroll
      for (int j = 0; j < HD / 2; ++j) p[j] = f2_fma(p[j], inv, kNZ);  // exact: a power of two, normal result
    } else {
#pragma unroll
      for (int j = 0; j < HD / 2; ++j) {
        float lo, hi;
        f2_unpack(p[j], lo, hi);
        p[j] = f2_pack(lo / d.s, hi / d.s);
      }
    }
    // codes of this row: 8 chunks of 16 elements, chunk c at tid * 128 + ((c ^ (tid % 8)) * 16)
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v0, v1, v2, v3;
        f2_unpack(p[8 * c + 2 * e], v0, v1);
        f2_unpack(p[8 * c + 2 * e + 1], v2, v3);
        w[e] = pack_e4m3x2(v0, v1) | (pack_e4m3x2(v2, v3) << 16);
      }
      *reinterpret_cast<uint4 *>(tb + tid * 128 + ((c ^ (tid & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
    uint8_t *dst = codes + ((int64_t)plane * N + (int64_t)blk * BM) * HD;
#pragma unroll
    for (int j = 0; j < BM * HD / 16 / ROW_THREADS; ++j) {
      const int i = j * ROW_THREADS + tid, r = i >> 3, c = i & 7;  // chunk i = 8 r + c of the codes
      if (r < rows)
        *reinterpret_cast<uint4 *>(dst + (int64_t)i * 16) =
            *reinterpret_cast<const uint4 *>(tb + r * 128 + ((c ^ (r & 7)) << 4));
    }
    __syncthreads();  // the buffer's codes are out before the next copy into it
  }
}

// One CTA per (plane, 128-key block) of V: the block's max |v|, folded into
// the head's maximum by an atomic max on its bits (non-negative floats order
// like their bit patterns); the K rows kernel, earlier on the stream, zeroed
// them.
__global__ void __launch_bounds__(256) attn_fp8_vmax_kernel(const __nv_bfloat16 *v, unsigned *vmax_bits, int N,
                                                            int nblk) {
  __shared__ float wmax[8];
  const int plane = blockIdx.x / nblk, blk = blockIdx.x % nblk;
  const int rows = min(BN, N - blk * BN);
  const uint4 *src = reinterpret_cast<const uint4 *>(v + ((int64_t)plane * N + (int64_t)blk * BN) * HD);
  float amax = 0.f;
  for (int i = threadIdx.x; i < rows * (HD / 8); i += 256) {
    const uint4 w = src[i];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(ws[c] << 16)), fabsf(__uint_as_float(ws[c] & 0xffff0000u))));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = wmax[0];
    for (int w = 1; w < 8; ++w) a = fmaxf(a, wmax[w]);
    atomicMax(vmax_bits + plane, __float_as_uint(a));
  }
}

// sv[i] = the power-of-two scale of the head maximum whose bits sv holds.
__global__ void __launch_bounds__(256) attn_fp8_vscale_kernel(float *sv, int n) {
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i < n) sv[i] = pow2_scale(__uint_as_float(reinterpret_cast<unsigned *>(sv)[i]));
}

// One CTA per (plane, 128-key block): V codes e4m3(v / sv) written transposed,
// vt[plane][d][key] with rows of nkv_pad = 128 * nblk bytes (keys >= N hold
// code 0).  Thread t converts keys 4 (t % 32) .. + 3 at head dims
// 16 (t / 32) .. + 15 and packs each head dim's four codes into one word.
__global__ void __launch_bounds__(256) attn_fp8_vt_kernel(const __nv_bfloat16 *v, const float *scales, uint8_t *vt,
                                                          int N, int nkv_pad, int nblk) {
  __shared__ uint32_t tile[HD][BN / 4 + 1];  // [d][key / 4], rows padded against bank conflicts
  const int plane = blockIdx.x / nblk, blk = blockIdx.x % nblk;
  const int k0 = blk * BN;
  // the head's max |v| (bits, see attn_fp8_vmax_kernel) -> its scale
  const InvPow2 dv(pow2_exp(__uint_as_float(reinterpret_cast<const unsigned *>(scales)[plane])));
  {
    const int kg = threadIdx.x & 31, dg = threadIdx.x >> 5;
    uint32_t w[4][8];  // [key][bf16 pairs of the 16 head dims]
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = k0 + 4 * kg + e;
      uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
      if (key < N) {
        const uint4 *src = reinterpret_cast<const uint4 *>(v + ((int64_t)plane * N + key) * HD + 16 * dg);
        a = src[0];
        b = src[1];
      }
      w[e][0] = a.x; w[e][1] = a.y; w[e][2] = a.z; w[e][3] = a.w;
      w[e][4] = b.x; w[e][5] = b.y; w[e][6] = b.z; w[e][7] = b.w;
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        x[e] = dv(__uint_as_float((c & 1) ? (w[e][c >> 1] & 0xffff0000u) : (w[e][c >> 1] << 16)));
      tile[16 * dg + c][kg] = pack_e4m3x2(x[0], x[1]) | (pack_e4m3x2(x[2], x[3]) << 16);
    }
  }
  __syncthreads();
  // thread t writes head-dim row d = t / 2, keys (t % 2) * 64 .. + 64, in 16-byte pieces
  {
    const int d = threadIdx.x >> 1, h = threadIdx.x & 1;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int wi = h * 16 + 4 * c;
      *reinterpret_cast<uint4 *>(vt + ((int64_t)plane * HD + d) * nkv_pad + k0 + 4 * wi) =
          make_uint4(tile[d][wi], tile[d][wi + 1], tile[d][wi + 2], tile[d][wi + 3]);
    }
  }
}

// ---------------------------------------------------------------- attention

struct Fp8Params {
  __nv_bfloat16 *o;
  float *lse;
  const float *sq, *sk, *sv;  // scales: [B*Hq, nqb], [B*Hkv, nkb], [B*Hkv]
  int B, Hq, Hkv, Nq, Nkv, nqb, nkb;
  float scale;
  int causal;
  int *status;
  int npairs;
  int kst, vst;
  uint32_t off_k, off_v, off_bar;
  uint64_t wait_limit_ns;
};

struct Fp8Bars {
  uint64_t q_full;
  uint64_t k_full[MAX_KST];
  uint64_t k_empty[MAX_KST];
  uint64_t v_full[MAX_VST];
  uint64_t v_empty[MAX_VST];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t done;
  uint32_t tmem_slot;
  int abort;
};

__device__ __forceinline__ void raise_abort(Fp8Bars *bars, int *status) {
  atomicCAS(status, 0, kStatusTimeout);
  *reinterpret_cast<volatile int *>(&bars->abort) = 1;
}

// CTA = 11 warps: 0-3 softmax + epilogue of tile 0, 4-7 of tile 1, 8 TMA
// producer of Q and K, 9 TMEM allocator and MMA issuer, 10 TMA producer of V.
// TMEM: S_t [128t, 128t+128) fp32 with P_t (e4m3, four keys per column) over
// its first 32 columns; O_t [256 + 128t, 256 + 128t + 128).  The MMA issue
// order and its reliance on in-order execution are those of the bf16
// two-tile kernel: per block j, PV0_j, S0_{j+1}, PV1_j, S1_{j+1}.
__global__ void __launch_bounds__(THREADS, 1)
    attn_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_vt, const Fp8Params prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t *sq = smem;  // tile t at t * TILE
  uint8_t *sk = smem + prm.off_k;
  uint8_t *sv = smem + prm.off_v;
  Fp8Bars *bars = reinterpret_cast<Fp8Bars *>(smem + prm.off_bar);
  volatile int *abortf = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t limit = prm.wait_limit_ns;

  // ---- work unit: (b, hq) fastest, then tile pair (heaviest causal pairs first)
  const int BH = prm.B * prm.Hq;
  const int bh = blockIdx.x % BH;
  const int t_idx = blockIdx.x / BH;
  const int pair = prm.causal ? (prm.npairs - 1 - t_idx) : t_idx;
  const int b = bh / prm.Hq, hq = bh % prm.Hq;
  const int bkv = b * prm.Hkv + hq / (prm.Hq / prm.Hkv);
  const int shift = prm.Nkv - prm.Nq;
  int nblk_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int q0 = pair * 2 * BM + t * BM;
    int kv_end = prm.Nkv;
    if (prm.causal) kv_end = max(0, min(prm.Nkv, q0 + BM - 1 + shift + 1));
    nblk_t[t] = (q0 < prm.Nq) ? (kv_end + BN - 1) / BN : 0;
  }
  const int nblk = max(nblk_t[0], nblk_t[1]);

  if (tid == 0) {
    mbar_init(&bars->q_full, 2);
    for (int i = 0; i < prm.kst; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < prm.vst; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->o_done[t], 1);
    }
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(&bars->tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  if (warp == WARP_LOAD_K || warp == WARP_LOAD_V) {
    // ------------------------------------------------------------ producers
    if (lane == 0 && nblk > 0) {
      const bool is_k = warp == WARP_LOAD_K;
      uint32_t ctr = 0;
      int slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int qt = is_k ? 0 : 1;
      mbar_arrive_expect_tx(&bars->q_full, TILE);
      tma_load_3d(sq + qt * TILE, &tm_q, &bars->q_full, 0, pair * 2 * BM + qt * BM, bh);
      const int nst = is_k ? prm.kst : prm.vst;
      for (int j = 0; j < nblk; ++j) {
        uint64_t *empty = is_k ? &bars->k_empty[slot] : &bars->v_empty[slot];
        uint64_t *full = is_k ? &bars->k_full[slot] : &bars->v_full[slot];
        if (!mbar_wait(empty, phase ^ 1u, abortf, limit)) { ok = false; break; }
        mbar_arrive_expect_tx(full, TILE);
        if (is_k)
          tma_load_3d(sk + slot * TILE, &tm_k, full, 0, j * BN, bkv);
        else
          tma_load_3d(sv + slot * TILE, &tm_vt, full, j * BN, 0, bkv);
        ++ctr;
        if (++slot == nst) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) raise_abort(bars, prm.status);
      mbar_wait_drain(&bars->q_full, 0, limit);
      const uint32_t n = ctr < (uint32_t)nst ? ctr : (uint32_t)nst;
      for (uint32_t i = ctr - n; i < ctr; ++i)
        mbar_wait_drain(is_k ? &bars->k_full[i % nst] : &bars->v_full[i % nst], (i / nst) & 1, limit);
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nblk > 0) {
      const uint32_t idesc = idesc_e4m3(BM, BN);  // S (N = 128 keys) and P V (N = 128 head dims)
      bool ok = mbar_wait(&bars->q_full, 0, abortf, limit);
      // K-major 128B-swizzled tiles; a K = 32 step is 32 bytes (2 in the >>4 field)
      constexpr uint64_t kTileD = TILE >> 4;
      const uint64_t qd_base = smem_desc(smem_u32(sq), 16, 1024);
      const uint64_t kd_base = smem_desc(smem_u32(sk), 16, 1024);
      const uint64_t vd_base = smem_desc(smem_u32(sv), 16, 1024);
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      auto issue_s = [&](int t, bool wait_full, bool release) -> bool {
        if (wait_full && !mbar_wait(&bars->k_full[ks], kph, abortf, limit)) return false;
        tc_fence_after();
        const uint64_t qd0 = qd_base + (uint64_t)t * kTileD, kd0 = kd_base + (uint64_t)ks * kTileD;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f8_ss(tmem + 128 * t, qd0 + kk * 2, kd0 + kk * 2, idesc, kk != 0);
        if (release) mma_commit(&bars->k_empty[ks]);
        mma_commit(&bars->s_full[t]);
        return true;
      };
      auto next_k = [&]() {
        if (++ks == prm.kst) {
          ks = 0;
          kph ^= 1u;
        }
      };
      auto act = [&](int t, int j) { return j < nblk_t[t]; };
      if (ok && act(0, 0)) ok = issue_s(0, true, !act(1, 0));
      if (ok && act(1, 0)) ok = issue_s(1, !act(0, 0), true);
      next_k();
      for (int j = 0; j < nblk && ok; ++j) {
        const uint64_t vd0 = vd_base + (uint64_t)vs * kTileD;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!act(t, j)) continue;
          if (!mbar_wait(&bars->p_full[t], j & 1, abortf, limit)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8_ts(tmem + 256 + 128 * t, tmem + 128 * t + kk * 8, vd0 + kk * 2, idesc, (j > 0 || kk > 0) ? 1u : 0u);
          if (j == nblk_t[t] - 1) mma_commit(&bars->o_done[t]);
          if (act(t, j + 1)) {
            const bool last = (t == 1) || !act(1, j + 1);
            if (!issue_s(t, false, last)) { ok = false; break; }
          }
        }
        if (!ok) break;
        mma_commit(&bars->v_empty[vs]);
        next_k();
        if (++vs == prm.vst) {
          vs = 0;
          vph ^= 1u;
        }
      }
      if (!ok) raise_abort(bars, prm.status);
      mma_commit(&bars->done);
      if (!mbar_wait_drain(&bars->done, 0, limit)) raise_abort(bars, prm.status);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue
    const int t = warp >> 2;
    const int row = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + 128 * t;
    const uint32_t tO = tmem + lane_base + 256 + 128 * t;
    const int tile = pair * 2 + t;
    const int qi = tile * BM + row;
    const int nb = nblk_t[t];
    const int vis_end = prm.causal ? min(prm.Nkv, qi + shift + 1) : prm.Nkv;
    // log2-unit multiplier of the raw code products: scale * sq * sk_j * log2 e
    const float cq = (nb > 0) ? prm.scale * kLog2e * prm.sq[(int64_t)bh * prm.nqb + tile] : 0.f;
    const float *skp = prm.sk + (int64_t)bkv * prm.nkb;
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    uint32_t ring = 1u << 8;  // V slot bits 0-7, K slot 8-15, V phase bit 16, K phase bit 24
    for (int j = 0; j < nb; ++j) {
      const float c = cq * __ldg(skp + j);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[t], j & 1, abortf, limit))) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sr[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) reg_fence32(sr[cc]);
      const int kbase = j * BN;
      // warp-uniform: both paths end in the warp-collective tcgen05.st
      const bool full = __all_sync(0xffffffffu, kbase + BN <= vis_end);
      float mblk;
      if (full) {
        // block max of the raw scores, four chains of 3-input maxima
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int q = 0; q < BN; q += 8) {
          mx0 = max3f(mx0, __uint_as_float(sr[q >> 5][(q & 31) + 0]), __uint_as_float(sr[q >> 5][(q & 31) + 1]));
          mx1 = max3f(mx1, __uint_as_float(sr[q >> 5][(q & 31) + 2]), __uint_as_float(sr[q >> 5][(q & 31) + 3]));
          mx2 = max3f(mx2, __uint_as_float(sr[q >> 5][(q & 31) + 4]), __uint_as_float(sr[q >> 5][(q & 31) + 5]));
          mx3 = max3f(mx3, __uint_as_float(sr[q >> 5][(q & 31) + 6]), __uint_as_float(sr[q >> 5][(q & 31) + 7]));
        }
        mblk = max3f(mx0, mx1, fmaxf(mx2, mx3)) * c;
      } else {
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < BN; ++q) {
          const float x = __uint_as_float(sr[q >> 5][q & 31]);
          mx[q & 3] = fmaxf(mx[q & 3], (kbase + q < vis_end) ? x : -INFINITY);
        }
        const float ext = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        mblk = (ext == -INFINITY) ? -INFINITY : ext * c;
      }
      const float m_new = fmaxf(m_use, mblk);
      if (__any_sync(0xffffffffu, m_new > m_use + TAU)) {
        const float alpha = (m_use == -INFINITY) ? 0.f : ex2_approx(m_use - m_new);
        if (j > 0) {
#pragma unroll 1
          for (int cc = 0; cc < HD / 16; ++cc) {
            uint32_t r[16];
            tmem_ld16(tO + cc * 16, r);
            tmem_wait_ld();
            reg_fence16(r);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st16(tO + cc * 16, r);
          }
        }
        l *= alpha;
        m_use = m_new;
      }
      // 2^2 p = 2^(s c - m + 2); quarter h of the keys lands as e4m3 in
      // columns [8h, 8h + 8), all inside the first quarter, already read
      const float bias = P_SHIFT - ((m_use == -INFINITY) ? 0.f : m_use);
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      if (full) {
        // every key visible: y on f32x2 pairs, exp2 on the MUFU
        const uint64_t c2 = f2_pack(c, c), b2 = f2_pack(bias, bias);
        uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t pk[8];
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            const uint64_t y01 = f2_fma(f2_pack(__uint_as_float(sr[h][4 * w]), __uint_as_float(sr[h][4 * w + 1])), c2, b2);
            const uint64_t y23 =
                f2_fma(f2_pack(__uint_as_float(sr[h][4 * w + 2]), __uint_as_float(sr[h][4 * w + 3])), c2, b2);
            float y0, y1, y2, y3;
            f2_unpack(y01, y0, y1);
            f2_unpack(y23, y2, y3);
            const float p0 = ex2_approx(y0), p1 = ex2_approx(y1), p2 = ex2_approx(y2), p3 = ex2_approx(y3);
            acc0 = f2_add(acc0, f2_pack(p0, p1));
            acc1 = f2_add(acc1, f2_pack(p2, p3));
            pk[w] = pack_e4m3x2(p0, p1) | (pack_e4m3x2(p2, p3) << 16);
          }
          tmem_st8(tS + 8 * h, pk);
        }
        float a0, a1, b0, b1;
        f2_unpack(acc0, a0, a1);
        f2_unpack(acc1, b0, b1);
        ls[0] = a0 + a1;
        ls[1] = b0 + b1;
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t pk[8];
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int q = 32 * h + 4 * w + e;
              p[e] = (kbase + q < vis_end) ? ex2_approx(fmaf(__uint_as_float(sr[h][4 * w + e]), c, bias)) : 0.f;
            }
            ls[w & 3] += (p[0] + p[1]) + (p[2] + p[3]);
            pk[w] = pack_e4m3x2(p[0], p[1]) | (pack_e4m3x2(p[2], p[3]) << 16);
          }
          tmem_st8(tS + 8 * h, pk);
        }
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      tmem_wait_st();
      tc_fence_before();
      // tile 0 (or tile 1 where tile 0 has no keys in this block) vouches for
      // V_j and K_{j+1}, so that the MMA thread waits for P alone
      if (row == 0 && (t == 0 || j >= nblk_t[0])) {
        bool got = mbar_wait(&bars->v_full[ring & 0xffu], (ring >> 16) & 1u, abortf, limit);
        if (got && j + 1 < nblk) got = mbar_wait(&bars->k_full[(ring >> 8) & 0xffu], ring >> 24, abortf, limit);
        if (!got) raise_abort(bars, prm.status);
      }
      if (row == 0) {
        ring += 1u;
        if ((ring & 0xffu) == (uint32_t)prm.vst) ring = (ring & ~0xffu) ^ (1u << 16);
        ring += 1u << 8;
        if (((ring >> 8) & 0xffu) == (uint32_t)prm.kst) ring = (ring & ~0xff00u) ^ (1u << 24);
      }
      mbar_arrive(&bars->p_full[t]);
    }
    if (!ok) raise_abort(bars, prm.status);

    // ---- epilogue: O = sv * acc / l (l holds 2^2 times the sum of p)
    if (ok && nb > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_done[t], 0, abortf, limit))) {
        raise_abort(bars, prm.status);
        ok = false;
      }
    }
    if (ok) {
      tc_fence_after();
      const float inv = (l > 0.f) ? prm.sv[bkv] / l : 0.f;
      const float lse_val =
          (m_use == -INFINITY || !(l > 0.f)) ? -INFINITY : (m_use + log2f(l) - P_SHIFT) * kLn2;
      const int64_t row_idx = (int64_t)bh * prm.Nq + qi;
      __nv_bfloat16 *orow = prm.o + row_idx * HD;
#pragma unroll
      for (int cc = 0; cc < HD / 32; ++cc) {
        uint32_t r[32];
        if (nb > 0) {
          tmem_ld32(tO + cc * 32, r);
          tmem_wait_ld();
          reg_fence32(r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (qi < prm.Nq) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[v4 * 8 + 0]) * inv, __uint_as_float(r[v4 * 8 + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(r[v4 * 8 + 2]) * inv, __uint_as_float(r[v4 * 8 + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(r[v4 * 8 + 4]) * inv, __uint_as_float(r[v4 * 8 + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(r[v4 * 8 + 6]) * inv, __uint_as_float(r[v4 * 8 + 7]) * inv);
            dst[v4] = w;
          }
        }
      }
      if (qi < prm.Nq) prm.lse[row_idx] = lse_val;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// CTAs of a rows launch: at most ROW_CTAS_PER_SM per SM, one per unit below that.
unsigned rows_grid(int64_t units, int sms) {
  const int64_t g = (int64_t)ROW_CTAS_PER_SM * sms;
  return (unsigned)(units < g ? units : g);
}

// The rows kernel's 64 KB of dynamic shared memory, allowed once per device.
cudaError_t rows_ready(int device) {
  static std::atomic<int> done[64];
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  if (done[device].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(attn_fp8_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ROW_SMEM);
  if (e == cudaSuccess) done[device].store(1, std::memory_order_release);
  return e;
}

int fp8_sizes_ok(int B, int Hq, int Hkv, int Nq, int Nkv, int D) {
  const int rc = check_problem(B, Hq, Hkv, Nq, Nkv, D, 0);
  if (rc != ATTN_OK) return rc;
  return D == HD ? ATTN_OK : ATTN_ERR_ARG;
}

}  // namespace
}  // namespace attn

extern "C" int attn_fp8_quantize(const void *q, const void *k, const void *v, void *q8, void *k8, void *vt8,
                                 float *sq, float *sk, float *sv, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                                 attn_stream_t stream) {
  using namespace attn;
  int rc = fp8_sizes_ok(B, Hq, Hkv, Nq, Nkv, D);
  if (rc != ATTN_OK) return rc;
  if (B == 0) return ATTN_OK;
  const bool has_q = Nq > 0, has_k = Nkv > 0;
  if (has_q && (!q || !q8 || !sq)) return ATTN_ERR_ARG;
  if (has_k && (!k || !v || !k8 || !vt8 || !sk || !sv)) return ATTN_ERR_ARG;
  if (has_q && (!aligned16(q) || !aligned16(q8) || !aligned16(sq))) return ATTN_ERR_ALIGN;
  if (has_k && (!aligned16(k) || !aligned16(v) || !aligned16(k8) || !aligned16(vt8) || !aligned16(sk) ||
                !aligned16(sv)))
    return ATTN_ERR_ALIGN;
  int device = 0, sms = 0, *status = nullptr;
  if ((rc = current_device(&device, &sms, &status)) != ATTN_OK) return rc;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int nqb = (Nq + BM - 1) / BM, nkb = (Nkv + BN - 1) / BN, nkv_pad = nkb * BN;
  // one rows unit per (plane, 128-row block); the V kernels take one CTA per unit
  if ((int64_t)B * Hq * nqb > INT_MAX || (int64_t)B * Hkv * nkb > INT_MAX) return ATTN_ERR_ARG;
  if (const cudaError_t e = rows_ready(device); e != cudaSuccess) return record_cuda_error(e);
  const auto *qb = static_cast<const __nv_bfloat16 *>(q);
  const auto *kb = static_cast<const __nv_bfloat16 *>(k);
  const auto *vb = static_cast<const __nv_bfloat16 *>(v);
  if (has_q) {
    const int64_t units = (int64_t)B * Hq * nqb;
    attn_fp8_rows_kernel<<<rows_grid(units, sms), ROW_THREADS, ROW_SMEM, st>>>(
        qb, static_cast<uint8_t *>(q8), sq, Nq, nqb, (int)units, nullptr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda_error(e);
  }
  if (has_k) {
    // sv carries the bits of each head's max |v| until the last kernel turns
    // them into the scales: K rows (zeroing them), V block maxima (atomic
    // max), V codes (each block derives the scale from the maximum), scales
    unsigned *vbits = reinterpret_cast<unsigned *>(sv);
    const unsigned g = (unsigned)((int64_t)B * Hkv * nkb);
    attn_fp8_rows_kernel<<<rows_grid(g, sms), ROW_THREADS, ROW_SMEM, st>>>(kb, static_cast<uint8_t *>(k8), sk, Nkv,
                                                                          nkb, (int)g, vbits);
    attn_fp8_vmax_kernel<<<g, 256, 0, st>>>(vb, vbits, Nkv, nkb);
    attn_fp8_vt_kernel<<<g, 256, 0, st>>>(vb, sv, static_cast<uint8_t *>(vt8), Nkv, nkv_pad, nkb);
    attn_fp8_vscale_kernel<<<(unsigned)((B * Hkv + 255) / 256), 256, 0, st>>>(sv, B * Hkv);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda_error(e);
  }
  return ATTN_OK;
}

extern "C" int attn_fwd_fp8(const void *q8, const void *k8, const void *vt8, const float *sq, const float *sk,
                            const float *sv, void *o, float *lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                            float scale, int causal, attn_stream_t stream) {
  using namespace attn;
  int rc = fp8_sizes_ok(B, Hq, Hkv, Nq, Nkv, D);
  if (rc != ATTN_OK) return rc;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  if (!isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_ARG;
  if (B == 0 || Nq == 0) return ATTN_OK;
  if (!q8 || !sq || !o || !lse) return ATTN_ERR_ARG;
  if (Nkv > 0 && (!k8 || !vt8 || !sk || !sv)) return ATTN_ERR_ARG;
  if (!aligned16(q8) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_ALIGN;
  if (Nkv > 0 && (!aligned16(k8) || !aligned16(vt8))) return ATTN_ERR_ALIGN;
  int device = 0, sms = 0, *status = nullptr;
  if ((rc = current_device(&device, &sms, &status)) != ATTN_OK) return rc;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (Nkv == 0) {  // no keys: O = 0, LSE = -inf
    Problem p{};
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = Nq; p.Nkv = 0; p.D = D;
    const cudaError_t e = launch_nokeys(p, sms, st);
    return e == cudaSuccess ? ATTN_OK : record_cuda_error(e);
  }
  const int nkv_pad = (Nkv + BN - 1) / BN * BN;  // V^T row length
  Fp8Params prm;
  memset(&prm, 0, sizeof(prm));
  prm.o = static_cast<__nv_bfloat16 *>(o);
  prm.lse = lse;
  prm.sq = sq;
  prm.sk = sk;
  prm.sv = sv;
  prm.B = B; prm.Hq = Hq; prm.Hkv = Hkv; prm.Nq = Nq; prm.Nkv = Nkv;
  prm.nqb = (Nq + BM - 1) / BM;
  prm.nkb = (Nkv + BN - 1) / BN;
  prm.scale = scale;
  prm.causal = causal;
  prm.status = status;
  prm.npairs = (prm.nqb + 1) / 2;
  prm.wait_limit_ns = wait_limit_ns();
  // shared memory: the Q pair, then K and V rings of 16 KB slots
  const int avail = kSmemMax - 2048 - 2 * TILE;
  prm.vst = MAX_VST;
  prm.kst = (avail - prm.vst * TILE) / TILE;
  if (prm.kst > MAX_KST) prm.kst = MAX_KST;
  prm.off_k = 2 * TILE;
  prm.off_v = prm.off_k + prm.kst * TILE;
  prm.off_bar = prm.off_v + prm.vst * TILE;
  const int smem = (int)prm.off_bar + (int)sizeof(Fp8Bars) + 1024;
  if (prm.kst < 2 || smem > kSmemMax) return record_cuda_error(cudaErrorInvalidConfiguration);
  CUtensorMap tq, tk, tvt;
  if (!make_u8_map(&tq, q8, HD, Nq, B * Hq) || !make_u8_map(&tk, k8, HD, Nkv, B * Hkv) ||
      !make_u8_map(&tvt, vt8, nkv_pad, HD, B * Hkv))
    return record_cuda_error(cudaErrorInvalidValue);
  static std::atomic<int> attr_set[64];
  if (device < 0 || device >= 64) return ATTN_ERR_ARCH;
  cudaError_t e = cudaSuccess;
  if (!attr_set[device].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(attn_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return record_cuda_error(e);
    attr_set[device].store(1, std::memory_order_release);
  }
  const int64_t grid = (int64_t)prm.npairs * B * Hq;
  if (grid > 0x7fffffffLL) return record_cuda_error(cudaErrorInvalidConfiguration);
  attn_fp8_kernel<<<(unsigned)grid, THREADS, smem, st>>>(tq, tk, tvt, prm);
  e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : record_cuda_error(e);
}
