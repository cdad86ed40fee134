// Exact attention backward for head dims 64 and 128 on the sm_103a tensor
// cores: dQ, dK and dV from Q, K, V, O, dO and the forward's LSE.
//
// What is computed is the gradient of the forward definition (the chain rule
// through the row softmax): with P = exp(scale Q K^T - LSE) (masked entries 0),
//     dV = P^T dO,   dP = dO V^T,   Delta_i = sum_d dO_id O_id,
//     dS = P * (dP - Delta),   dQ = scale dS K,   dK = scale dS^T Q.
// As the "FlashAttention v1/v2/v3/v4" page says of FA1's backward ("FA1 --
// el cambio de orden de las operaciones", and the FlashAttention summary
// card), nothing N x N is stored: S is recomputed block by block from Q, K
// and the row statistics (here the LSE, so P needs no running max).
//
// Three kernels:
//   prep  Delta_i and LSE_i * log2 e for every query row, into padded
//         per-head vectors (+inf for rows that saw no key and for padding
//         rows, which makes their P exactly 0);
//   dkdv  one CTA per (b, kv head, 128-key tile), looping over the query
//         blocks of every query head of its GQA group, so that the group's
//         sum is formed in TMEM with no atomics: S^T = K Q^T and
//         dP^T = V dO^T on the tensor cores, P^T and dS^T by the math warps
//         (one key row per thread) written back to TMEM as bf16, then
//         dV += P^T dO and dK += dS^T Q with P^T / dS^T read from TMEM;
//   dq    one CTA per (b, q head, pair of 128-row query tiles), looping
//         over key blocks shared by both tiles: S = Q K^T, dP = dO V^T in
//         the same TMEM columns once S has been read, dS by the math warps
//         (one query row per thread), dQ += dS K, the two tiles interleaved.
// The split into a key-stationary and a query-stationary kernel recomputes
// S and dP once more (7 block products instead of 5) but needs no atomic
// accumulation of dQ and gives the same bits on every run.
//
// dkdv CTA = 6 warps: 0-3 math (TMEM lanes 32w..32w+31), 4 TMA producer (one
// thread), 5 TMEM allocator and MMA issuer (one thread); dq CTA = 10 warps:
// 0-7 math (tile w / 4), 8 the two producers, 9 the MMA issuer.
//
// TMEM columns, dkdv: S^T/P^T [0,128), dP^T/dS^T [128,256), dV [256,256+D),
// dK [256+D, 256+2D); dq: S_t/dP_t/dS_t [128t, 128t+128), dQ_t
// [256 + Dt, 256 + Dt + D).
// P (bf16 pairs) overwrites the first 64 columns of S a quarter at a time
// after the quarter it lands on has been read; the same for dS over dP.
//
// Every wait is bounded; a role that gives up records ATTN_ERR_TIMEOUT in the
// status word, raises the CTA's abort flag, drains its own copies and MMAs,
// and the CTA frees its TMEM.
#include <math.h>
#include <string.h>

#include <atomic>

#include "attn.h"
#include "attn_internal.h"
#include "sm100_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

constexpr int BT = 128;                  // rows of a query or key tile
constexpr int CHUNK_BYTES = 128 * 128;   // 128 rows x 64 bf16 columns
constexpr int THREADS = 192;
constexpr int WARP_LOAD = 4, WARP_MMA = 5;
constexpr int NST = 2;                   // ring stages
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_DP = 128, TM_ACC = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSmemMax = 232448;
constexpr int VEC_BYTES = 1024;          // lse2[128] and delta[128] of one query block

struct BwdParams {
  const __nv_bfloat16 *o, *dout;  // [B, Hq, Nq, D]
  const float *lse;               // [B, Hq, Nq]
  __nv_bfloat16 *dq;              // [B, Hq, Nq, D]
  __nv_bfloat16 *dk, *dv;         // [B, Hkv, Nkv, D]
  float *lse2;                    // [B*Hq, nq_pad]: LSE * log2 e; +inf where no key / padding
  float *delta;                   // [B*Hq, nq_pad]: sum_d dO * O; 0 on padding rows
  int B, Hq, Hkv, Nq, Nkv, D, nq_pad;
  float scale;
  int causal;
  int *status;
  uint64_t wait_limit_ns;
};

struct BwdBars {
  uint64_t fixed_full;  // the CTA's resident tiles (K and V, or Q and dO)
  uint64_t full[NST];
  uint64_t empty[NST];
  uint64_t s_full, dp_full;  // MMA -> math
  uint64_t p_full;           // math -> MMA (dkdv: P^T written)
  uint64_t s_free;           // math -> MMA (dq: S read)
  uint64_t ds_full;          // math -> MMA (dS written, dP read)
  uint64_t o_done;           // MMA -> math (accumulators final)
  uint64_t done;
  uint32_t tmem_slot;
  int abort;
};

__device__ __forceinline__ void raise_abort(BwdBars *bars, int *status) {
  atomicCAS(status, 0, kStatusTimeout);
  *reinterpret_cast<volatile int *>(&bars->abort) = 1;
}

__device__ __forceinline__ void init_bars(BwdBars *bars) {
  mbar_init(&bars->fixed_full, 1);
  for (int i = 0; i < NST; ++i) {
    mbar_init(&bars->full[i], 1);
    mbar_init(&bars->empty[i], 1);
  }
  mbar_init(&bars->s_full, 1);
  mbar_init(&bars->dp_full, 1);
  mbar_init(&bars->p_full, 128);
  mbar_init(&bars->s_free, 128);
  mbar_init(&bars->ds_full, 128);
  mbar_init(&bars->o_done, 1);
  mbar_init(&bars->done, 1);
  bars->abort = 0;
  fence_mbar_init();
}

// ---------------------------------------------------------------- prep

// Delta = sum_d dO O (fp32) and LSE in log2 units for every padded query
// row.  D / 8 threads per row, each with one 16-byte load of O and of dO,
// summed by shuffles within the row's lanes: 256 / (D / 8) rows per CTA.
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p) {
  const int tpr = p.D / 8;  // threads per row: 8 (D = 64) or 16 (D = 128)
  const int64_t row = (int64_t)blockIdx.x * (256 / tpr) + threadIdx.x / tpr;
  const int part = threadIdx.x % tpr;
  const bool in = row < (int64_t)p.B * p.Hq * p.nq_pad;
  const int64_t bh = in ? row / p.nq_pad : 0;
  const int i = in ? (int)(row % p.nq_pad) : p.nq_pad;
  float acc = 0.f;
  if (in && i < p.Nq) {
    const int64_t base = (bh * p.Nq + i) * p.D + part * 8;
    const uint4 a = *reinterpret_cast<const uint4 *>(p.o + base);
    const uint4 d = *reinterpret_cast<const uint4 *>(p.dout + base);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, dv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      acc = fmaf(__uint_as_float(av[c] << 16), __uint_as_float(dv[c] << 16), acc);
      acc = fmaf(__uint_as_float(av[c] & 0xffff0000u), __uint_as_float(dv[c] & 0xffff0000u), acc);
    }
  }
  for (int off = tpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (in && part == 0) {
    float l2 = INFINITY;
    if (i < p.Nq) {
      const float l = p.lse[bh * p.Nq + i];
      if (l != -INFINITY) l2 = l * kLog2e;
    }
    p.lse2[row] = l2;
    p.delta[row] = acc;
  }
}

// Zero fill of n bf16 values (n a multiple of 8), grid-stride.
__global__ void __launch_bounds__(256) attn_bwd_zero_kernel(__nv_bfloat16 *x, int64_t n) {
  uint4 *v = reinterpret_cast<uint4 *>(x);
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n / 8; i += (int64_t)gridDim.x * 256)
    v[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Store 32 fp32 values times mul as bf16 (four 16-byte stores).
__device__ __forceinline__ void store_row32(__nv_bfloat16 *dst, const uint32_t (&r)[32], float mul) {
  uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int v4 = 0; v4 < 4; ++v4) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(r[v4 * 8 + 0]) * mul, __uint_as_float(r[v4 * 8 + 1]) * mul);
    w.y = pack_bf16x2(__uint_as_float(r[v4 * 8 + 2]) * mul, __uint_as_float(r[v4 * 8 + 3]) * mul);
    w.z = pack_bf16x2(__uint_as_float(r[v4 * 8 + 4]) * mul, __uint_as_float(r[v4 * 8 + 5]) * mul);
    w.w = pack_bf16x2(__uint_as_float(r[v4 * 8 + 6]) * mul, __uint_as_float(r[v4 * 8 + 7]) * mul);
    d4[v4] = w;
  }
}

// ---------------------------------------------------------------- dK, dV

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const BwdParams p) {
  constexpr int NC = D / 64;
  constexpr int TILE = NC * CHUNK_BYTES;         // one [128 x D] bf16 tile
  constexpr int STAGE = 2 * TILE + VEC_BYTES;    // Q block, dO block, their vectors
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t *sk = smem, *sv = smem + TILE;
  uint8_t *ring = smem + 2 * TILE;
  BwdBars *bars = reinterpret_cast<BwdBars *>(ring + NST * STAGE);
  volatile int *abortf = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t limit = p.wait_limit_ns;

  // ---- work unit: (b, kv head) fastest, then key tile (for causal the
  //      first tiles see the most queries: heaviest first)
  const int BHkv = p.B * p.Hkv;
  const int bhk = blockIdx.x % BHkv, kt = blockIdx.x / BHkv;
  const int b = bhk / p.Hkv, hkv = bhk % p.Hkv;
  const int g = p.Hq / p.Hkv;
  const int kv0 = kt * BT;
  const int shift = p.Nkv - p.Nq;
  const int nqt = (p.Nq + BT - 1) / BT;
  int qb0 = 0;  // first query block that sees a key of this tile
  if (p.causal) {
    const int first = kv0 - shift;
    qb0 = first <= 0 ? 0 : first / BT;
  }
  const int nqb = nqt > qb0 ? nqt - qb0 : 0;
  const int nblk = g * nqb;

  if (tid == 0) init_bars(bars);
  if (warp == WARP_MMA) {
    tmem_alloc(&bars->tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  if (warp == WARP_LOAD) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nblk > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(&bars->fixed_full, 2 * TILE);
      tma_load_4d(sk, &tm_k, &bars->fixed_full, 0, kv0, 0, bhk);
      tma_load_4d(sv, &tm_v, &bars->fixed_full, 0, kv0, 0, bhk);
      bool ok = true;
      int issued = 0;
      for (int jj = 0; jj < nblk; ++jj) {
        const int s = jj % NST;
        if (!mbar_wait(&bars->empty[s], ((jj / NST) & 1) ^ 1, abortf, limit)) { ok = false; break; }
        const int hq = hkv * g + jj / nqb, q0 = (qb0 + jj % nqb) * BT;
        const int plane = b * p.Hq + hq;
        uint8_t *st = ring + s * STAGE;
        mbar_arrive_expect_tx(&bars->full[s], STAGE);
        tma_load_4d(st, &tm_q, &bars->full[s], 0, q0, 0, plane);
        tma_load_4d(st + TILE, &tm_do, &bars->full[s], 0, q0, 0, plane);
        const int64_t vo = (int64_t)plane * p.nq_pad + q0;
        bulk_load(st + 2 * TILE, p.lse2 + vo, 512, &bars->full[s]);
        bulk_load(st + 2 * TILE + 512, p.delta + vo, 512, &bars->full[s]);
        ++issued;
      }
      if (!ok) raise_abort(bars, p.status);
      mbar_wait_drain(&bars->fixed_full, 0, limit);
      for (int i = issued > NST ? issued - NST : 0; i < issued; ++i)
        mbar_wait_drain(&bars->full[i % NST], (i / NST) & 1, limit);
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nblk > 0) {
      const uint32_t idesc_s = idesc_bf16(BT, BT, 0, 0);
      const uint32_t idesc_o = idesc_bf16(BT, D, 0, 1);
      constexpr uint64_t kChunkD = CHUNK_BYTES >> 4, kStageD = (uint64_t)STAGE >> 4;
      const uint64_t kd = smem_desc(smem_u32(sk), 16, 1024), vd = smem_desc(smem_u32(sv), 16, 1024);
      // ring operands: K-major (B of S^T and dP^T) and MN-major (B of dV, dK)
      const uint64_t q_km = smem_desc(smem_u32(ring), 16, 1024);
      const uint64_t do_km = smem_desc(smem_u32(ring + TILE), 16, 1024);
      const uint64_t q_mn = smem_desc(smem_u32(ring), CHUNK_BYTES, 1024);
      const uint64_t do_mn = smem_desc(smem_u32(ring + TILE), CHUNK_BYTES, 1024);
      // A [128 x D] K-major tile times B K-major block of stage s, into TMEM col
      auto issue_nt = [&](uint32_t col, uint64_t ad, uint64_t bd) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + col, ad + (uint64_t)(c * kChunkD + kk * 2), bd + (uint64_t)(c * kChunkD + kk * 2), idesc_s,
                   (c | kk) != 0);
      };
      bool ok = mbar_wait(&bars->fixed_full, 0, abortf, limit);
      if (ok) ok = mbar_wait(&bars->full[0], 0, abortf, limit);
      if (ok) {
        tc_fence_after();
        issue_nt(TM_S, kd, q_km);
        mma_commit(&bars->s_full);
        issue_nt(TM_DP, vd, do_km);
        mma_commit(&bars->dp_full);
      }
      for (int jj = 0; jj < nblk && ok; ++jj) {
        const int s = jj % NST, s1 = (jj + 1) % NST;
        const uint64_t so = (uint64_t)s * kStageD, so1 = (uint64_t)s1 * kStageD;
        // dV += P^T dO (P^T from TMEM over S^T)
        if (!mbar_wait(&bars->p_full, jj & 1, abortf, limit)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          mma_ts(tmem + TM_ACC, tmem + TM_S + kk * 8, do_mn + so + (uint64_t)(kk * (2048 >> 4)), idesc_o,
                 (jj > 0 || kk > 0) ? 1u : 0u);
        // S^T of the next block (P^T has been read by the MMA above: in order)
        if (jj + 1 < nblk) {
          if (!mbar_wait(&bars->full[s1], ((jj + 1) / NST) & 1, abortf, limit)) { ok = false; break; }
          tc_fence_after();
          issue_nt(TM_S, kd, q_km + so1);
          mma_commit(&bars->s_full);
        }
        // dK += dS^T Q (dS^T from TMEM over dP^T)
        if (!mbar_wait(&bars->ds_full, jj & 1, abortf, limit)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          mma_ts(tmem + TM_ACC + D, tmem + TM_DP + kk * 8, q_mn + so + (uint64_t)(kk * (2048 >> 4)), idesc_o,
                 (jj > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->empty[s]);
        if (jj + 1 < nblk) {
          issue_nt(TM_DP, vd, do_km + so1);
          mma_commit(&bars->dp_full);
        }
      }
      if (!ok) raise_abort(bars, p.status);
      mma_commit(&bars->o_done);
      mma_commit(&bars->done);
      if (!mbar_wait_drain(&bars->done, 0, limit)) raise_abort(bars, p.status);
    }
  } else {
    // ------------------------------------------------------------ math: one key row per thread
    const int row = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane_base + TM_S, tDP = tmem + lane_base + TM_DP;
    const int kk_row = kv0 + row;  // this thread's key
    const float sl2 = p.scale * kLog2e;
    bool ok = true;
    for (int jj = 0; jj < nblk; ++jj) {
      const int s = jj % NST;
      const int q0 = (qb0 + jj % nqb) * BT;
      const float *vec = reinterpret_cast<const float *>(ring + s * STAGE + 2 * TILE);  // lse2[128], delta[128]
      // the block's vectors were copied with its tiles (stage s complete)
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->full[s], (jj / NST) & 1, abortf, limit))) { ok = false; break; }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full, jj & 1, abortf, limit))) { ok = false; break; }
      tc_fence_after();
      // key kk_row is visible to query q iff kk_row <= q + shift (causal)
      const int qmin = kk_row - shift;  // first visible query
      float pr[BT];
      uint32_t qb[2][32];
      tmem_ld32(tS, qb[0]);
      tmem_wait_ld();
      reg_fence32(qb[0]);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t(&cur)[32] = qb[h & 1];
        if (h < 3) tmem_ld32(tS + 32 * (h + 1), qb[(h + 1) & 1]);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int c = 32 * h + i;
          const float4 l4 = *reinterpret_cast<const float4 *>(vec + (c & ~3));
          const float la = (c & 2) ? l4.z : l4.x, lb = (c & 2) ? l4.w : l4.y;
          const bool va = !p.causal || q0 + c >= qmin, vb = !p.causal || q0 + c + 1 >= qmin;
          pr[c] = va ? ex2_approx(fmaf(__uint_as_float(cur[i]), sl2, -la)) : 0.f;
          pr[c + 1] = vb ? ex2_approx(fmaf(__uint_as_float(cur[i + 1]), sl2, -lb)) : 0.f;
          pk[i >> 1] = pack_bf16x2(pr[c], pr[c + 1]);
        }
        tmem_st16(tS + 16 * h, pk);
        if (h < 3) {
          tmem_wait_ld();
          reg_fence32(qb[(h + 1) & 1]);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->dp_full, jj & 1, abortf, limit))) { ok = false; break; }
      tc_fence_after();
      tmem_ld32(tDP, qb[0]);
      tmem_wait_ld();
      reg_fence32(qb[0]);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t(&cur)[32] = qb[h & 1];
        if (h < 3) tmem_ld32(tDP + 32 * (h + 1), qb[(h + 1) & 1]);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int c = 32 * h + i;
          const float4 d4 = *reinterpret_cast<const float4 *>(vec + BT + (c & ~3));
          const float da = (c & 2) ? d4.z : d4.x, db = (c & 2) ? d4.w : d4.y;
          const float ds0 = pr[c] * (__uint_as_float(cur[i]) - da);
          const float ds1 = pr[c + 1] * (__uint_as_float(cur[i + 1]) - db);
          pk[i >> 1] = pack_bf16x2(ds0, ds1);
        }
        tmem_st16(tDP + 16 * h, pk);
        if (h < 3) {
          tmem_wait_ld();
          reg_fence32(qb[(h + 1) & 1]);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);
    }
    if (!ok) raise_abort(bars, p.status);
    // ---- epilogue: dV and scale * dK of this key row
    if (ok && nblk > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->o_done, 0, abortf, limit))) {
      raise_abort(bars, p.status);
      ok = false;
    }
    if (ok) {
      tc_fence_after();
      const int64_t r = (int64_t)bhk * p.Nkv + kk_row;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16 *dst = (which ? p.dk : p.dv) + r * D;
        const float mul = which ? p.scale : 1.f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t rr[32];
          if (nblk > 0) {
            tmem_ld32(tmem + lane_base + TM_ACC + which * D + cc * 32, rr);
            tmem_wait_ld();
            reg_fence32(rr);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = 0u;
          }
          if (kk_row < p.Nkv) store_row32(dst + cc * 32, rr, mul);
        }
      }
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

// ---------------------------------------------------------------- dQ

constexpr int DQ_THREADS = 320;  // warps 0-7 math (tile = warp / 4), 8 producers, 9 MMA
constexpr int DQ_WARP_LOAD = 8, DQ_WARP_MMA = 9;
constexpr int DQ_MAX_KST = 4, DQ_MAX_VST = 4;

struct DqBars {
  uint64_t q_full;  // Q_t and dO_t of both tiles (one producer each)
  uint64_t k_full[DQ_MAX_KST], k_empty[DQ_MAX_KST];
  uint64_t v_full[DQ_MAX_VST], v_empty[DQ_MAX_VST];
  uint64_t s_full[2], dp_full[2];  // MMA -> math
  uint64_t s_free[2], ds_full[2];  // math -> MMA
  uint64_t o_done[2];
  uint64_t done;
  uint32_t tmem_slot;
  int abort;
};

struct DqLayout {
  int kst, vst;
  uint32_t off_k, off_v, off_bar;
  int smem;
};

// Two 128-row query tiles per CTA share every K and V block; tile t keeps
// S_t, then dP_t, then dS_t (bf16 over its first 64 columns) in TMEM columns
// [128t, 128t + 128) and accumulates dQ_t in [256 + D t, 256 + D t + D).  Per
// key block j the MMA thread issues dP0, dP1 (each once its tile's math warps
// have read S), then dQ0 and S0 of the next block, dQ1 and S1 of the next
// block (each dQ once its tile's dS is written), so that one tile's math
// overlaps the other tile's products.  P stays in the math warps' registers
// (bf16) between S and dP.
template <int D>
__global__ void __launch_bounds__(DQ_THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const BwdParams p, const DqLayout lay) {
  constexpr int NC = D / 64;
  constexpr int TILE = NC * CHUNK_BYTES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t *sq = smem, *sdo = smem + 2 * TILE;  // tile t at + t * TILE
  uint8_t *sk = smem + lay.off_k, *sv = smem + lay.off_v;
  DqBars *bars = reinterpret_cast<DqBars *>(smem + lay.off_bar);
  volatile int *abortf = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t limit = p.wait_limit_ns;

  // ---- work unit: (b, hq) fastest, then tile pair (causal: heaviest first)
  const int BH = p.B * p.Hq;
  const int nqt = (p.Nq + BT - 1) / BT;
  const int npairs = (nqt + 1) / 2;
  const int bh = blockIdx.x % BH, t_idx = blockIdx.x / BH;
  const int pair = p.causal ? npairs - 1 - t_idx : t_idx;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int bkv = b * p.Hkv + hq / (p.Hq / p.Hkv);
  const int shift = p.Nkv - p.Nq;
  int nblk_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int q0 = (2 * pair + t) * BT;
    int kv_end = p.Nkv;
    if (p.causal) kv_end = max(0, min(p.Nkv, q0 + BT - 1 + shift + 1));
    nblk_t[t] = (q0 < p.Nq) ? (kv_end + BT - 1) / BT : 0;
  }
  const int nblk = max(nblk_t[0], nblk_t[1]);

  if (tid == 0) {
    mbar_init(&bars->q_full, 2);
    for (int i = 0; i < lay.kst; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < lay.vst; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->dp_full[t], 1);
      mbar_init(&bars->s_free[t], 128);
      mbar_init(&bars->ds_full[t], 128);
      mbar_init(&bars->o_done[t], 1);
    }
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == DQ_WARP_MMA) {
    tmem_alloc(&bars->tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  if (warp == DQ_WARP_LOAD) {
    // ------------------------------------------------------------ producers
    // lane 0: Q_0, dO_0, then the K ring; lane 1: Q_1, dO_1, then the V ring
    if (lane < 2 && nblk > 0) {
      const bool is_k = lane == 0;
      const int t = lane;
      const int nst = is_k ? lay.kst : lay.vst;
      uint8_t *ring = is_k ? sk : sv;
      const CUtensorMap *tm = is_k ? &tm_k : &tm_v;
      tma_prefetch_desc(tm);
      mbar_arrive_expect_tx(&bars->q_full, 2 * TILE);
      tma_load_4d(sq + t * TILE, &tm_q, &bars->q_full, 0, (2 * pair + t) * BT, 0, bh);
      tma_load_4d(sdo + t * TILE, &tm_do, &bars->q_full, 0, (2 * pair + t) * BT, 0, bh);
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int s = j % nst;
        uint64_t *empty = is_k ? &bars->k_empty[s] : &bars->v_empty[s];
        uint64_t *full = is_k ? &bars->k_full[s] : &bars->v_full[s];
        if (!mbar_wait(empty, ((j / nst) & 1) ^ 1, abortf, limit)) { ok = false; break; }
        mbar_arrive_expect_tx(full, TILE);
        tma_load_4d(ring + s * TILE, tm, full, 0, j * BT, 0, bkv);
        ++issued;
      }
      if (!ok) {
        atomicCAS(p.status, 0, kStatusTimeout);
        *reinterpret_cast<volatile int *>(&bars->abort) = 1;
      }
      mbar_wait_drain(&bars->q_full, 0, limit);
      for (int i = issued > nst ? issued - nst : 0; i < issued; ++i)
        mbar_wait_drain(is_k ? &bars->k_full[i % nst] : &bars->v_full[i % nst], (i / nst) & 1, limit);
    }
  } else if (warp == DQ_WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nblk > 0) {
      const uint32_t idesc_s = idesc_bf16(BT, BT, 0, 0);
      const uint32_t idesc_o = idesc_bf16(BT, D, 0, 1);
      constexpr uint64_t kChunkD = CHUNK_BYTES >> 4, kTileD = (uint64_t)TILE >> 4;
      const uint64_t qd = smem_desc(smem_u32(sq), 16, 1024), dod = smem_desc(smem_u32(sdo), 16, 1024);
      const uint64_t k_km = smem_desc(smem_u32(sk), 16, 1024), k_mn = smem_desc(smem_u32(sk), CHUNK_BYTES, 1024);
      const uint64_t v_km = smem_desc(smem_u32(sv), 16, 1024);
      auto abort_all = [&]() {
        atomicCAS(p.status, 0, kStatusTimeout);
        *reinterpret_cast<volatile int *>(&bars->abort) = 1;
      };
      // A [128 x D] K-major tile times B [128 x D] K-major block into TMEM col
      auto issue_nt = [&](uint32_t col, uint64_t ad, uint64_t bd) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + col, ad + (uint64_t)(c * kChunkD + kk * 2), bd + (uint64_t)(c * kChunkD + kk * 2), idesc_s,
                   (c | kk) != 0);
      };
      auto act = [&](int t, int j) { return j < nblk_t[t]; };
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      bool ok = mbar_wait(&bars->q_full, 0, abortf, limit);
      if (ok) ok = mbar_wait(&bars->k_full[0], 0, abortf, limit);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (act(t, 0)) {
            issue_nt(BT * t, qd + (uint64_t)t * kTileD, k_km);
            mma_commit(&bars->s_full[t]);
          }
      }
      for (int j = 0; j < nblk && ok; ++j) {
        // dP_t = dO_t V_j^T once tile t's math warps have read S_t
        if (!mbar_wait(&bars->v_full[vs], vph, abortf, limit)) { ok = false; break; }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!act(t, j)) continue;
          if (!mbar_wait(&bars->s_free[t], j & 1, abortf, limit)) { ok = false; break; }
          tc_fence_after();
          issue_nt(BT * t, dod + (uint64_t)t * kTileD, v_km + (uint64_t)vs * kTileD);
          mma_commit(&bars->dp_full[t]);
        }
        if (!ok) break;
        mma_commit(&bars->v_empty[vs]);
        if (++vs == lay.vst) {
          vs = 0;
          vph ^= 1u;
        }
        // dQ_t += dS_t K_j once dS_t is written, then S_t of the next block
        int ks1 = ks + 1;
        uint32_t kph1 = kph;
        if (ks1 == lay.kst) {
          ks1 = 0;
          kph1 ^= 1u;
        }
        if (j + 1 < nblk && !mbar_wait(&bars->k_full[ks1], kph1, abortf, limit)) { ok = false; break; }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!act(t, j)) continue;
          if (!mbar_wait(&bars->ds_full[t], j & 1, abortf, limit)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)
            mma_ts(tmem + TM_ACC + D * t, tmem + BT * t + kk * 8, k_mn + (uint64_t)ks * kTileD + (uint64_t)(kk * (2048 >> 4)),
                   idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
          if (j == nblk_t[t] - 1) mma_commit(&bars->o_done[t]);
          if (act(t, j + 1)) {
            issue_nt(BT * t, qd + (uint64_t)t * kTileD, k_km + (uint64_t)ks1 * kTileD);
            mma_commit(&bars->s_full[t]);
          }
        }
        if (!ok) break;
        mma_commit(&bars->k_empty[ks]);
        ks = ks1;
        kph = kph1;
      }
      if (!ok) abort_all();
      mma_commit(&bars->done);
      if (!mbar_wait_drain(&bars->done, 0, limit)) abort_all();
    }
  } else {
    // ------------------------------------------------------------ math: one query row per thread
    const int t = warp >> 2;
    const int row = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tR = tmem + lane_base + BT * t;
    const int qi = (2 * pair + t) * BT + row;
    const int nb = nblk_t[t];
    const int64_t vrow = (int64_t)bh * p.nq_pad + qi;  // padded rows hold lse2 = +inf
    const bool in_pad = qi < p.nq_pad;
    const float lse2 = in_pad ? p.lse2[vrow] : INFINITY, delta = in_pad ? p.delta[vrow] : 0.f;
    const int vis_end = p.causal ? min(p.Nkv, qi + shift + 1) : p.Nkv;  // keys [0, vis_end) visible
    const float sl2 = p.scale * kLog2e;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[t], j & 1, abortf, limit))) { ok = false; break; }
      tc_fence_after();
      const int kbase = j * BT;
      // the scores a quarter (32 keys) at a time, the next quarter's load in
      // flight while this one is turned into P
      float pf[BT];  // P in fp32 (dS = P (dP - Delta) is rounded once, to bf16)
      uint32_t qb[2][32];
      tmem_ld32(tR, qb[0]);
      tmem_wait_ld();
      reg_fence32(qb[0]);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t(&cur)[32] = qb[h & 1];
        if (h < 3) tmem_ld32(tR + 32 * (h + 1), qb[(h + 1) & 1]);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int c = kbase + 32 * h + i;
          pf[32 * h + i] = (c < vis_end) ? ex2_approx(fmaf(__uint_as_float(cur[i]), sl2, -lse2)) : 0.f;
          pf[32 * h + i + 1] = (c + 1 < vis_end) ? ex2_approx(fmaf(__uint_as_float(cur[i + 1]), sl2, -lse2)) : 0.f;
        }
        if (h < 3) {
          tmem_wait_ld();
          reg_fence32(qb[(h + 1) & 1]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->s_free[t]);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->dp_full[t], j & 1, abortf, limit))) { ok = false; break; }
      tc_fence_after();
      // dS a quarter at a time the same way; quarter h lands in columns
      // [16h, 16h + 16), already read, while the load in flight reads further on
      tmem_ld32(tR, qb[0]);
      tmem_wait_ld();
      reg_fence32(qb[0]);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t(&cur)[32] = qb[h & 1];
        if (h < 3) tmem_ld32(tR + 32 * (h + 1), qb[(h + 1) & 1]);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          pk[i >> 1] = pack_bf16x2(pf[32 * h + i] * (__uint_as_float(cur[i]) - delta),
                                   pf[32 * h + i + 1] * (__uint_as_float(cur[i + 1]) - delta));
        }
        tmem_st16(tR + 16 * h, pk);
        if (h < 3) {
          tmem_wait_ld();
          reg_fence32(qb[(h + 1) & 1]);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->ds_full[t]);
    }
    if (!ok) {
      atomicCAS(p.status, 0, kStatusTimeout);
      *reinterpret_cast<volatile int *>(&bars->abort) = 1;
    }
    if (ok && nb > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->o_done[t], 0, abortf, limit))) {
      atomicCAS(p.status, 0, kStatusTimeout);
      *reinterpret_cast<volatile int *>(&bars->abort) = 1;
      ok = false;
    }
    if (ok) {
      tc_fence_after();
      __nv_bfloat16 *dst = p.dq + ((int64_t)bh * p.Nq + qi) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t rr[32];
        if (nb > 0) {
          tmem_ld32(tmem + lane_base + TM_ACC + D * t + cc * 32, rr);
          tmem_wait_ld();
          reg_fence32(rr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
        if (qi < p.Nq) store_row32(dst + cc * 32, rr, p.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == DQ_WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int D>
DqLayout dq_layout() {
  constexpr int TILE = (D / 64) * CHUNK_BYTES;
  DqLayout L;
  const int avail = kSmemMax - 2048 - 4 * TILE;  // Q and dO of both tiles resident
  int slots = avail / TILE;                       // K and V ring slots
  L.kst = slots >= 4 ? (slots / 2 > DQ_MAX_KST ? DQ_MAX_KST : slots / 2) : 2;
  L.vst = slots - L.kst > DQ_MAX_VST ? DQ_MAX_VST : slots - L.kst;
  L.off_k = 4 * TILE;
  L.off_v = L.off_k + L.kst * TILE;
  L.off_bar = L.off_v + L.vst * TILE;
  L.smem = (int)L.off_bar + (int)sizeof(DqBars) + 1024;
  return L;
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams &prm, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                         const __nv_bfloat16 *v, int device, cudaStream_t st) {
  constexpr int TILE = (D / 64) * CHUNK_BYTES;
  constexpr int SM_DKDV = 2 * TILE + NST * (2 * TILE + VEC_BYTES) + (int)sizeof(BwdBars) + 1024;
  static_assert(SM_DKDV <= kSmemMax, "shared memory plan too large");
  const DqLayout dql = dq_layout<D>();
  if (dql.kst < 2 || dql.vst < 1 || dql.smem > kSmemMax) return cudaErrorInvalidConfiguration;
  CUtensorMap tq, tdo, tk, tv;
  if (!make_block_map(&tq, q, D, prm.Nq, prm.B * prm.Hq, BT)) return cudaErrorInvalidValue;
  if (!make_block_map(&tdo, prm.dout, D, prm.Nq, prm.B * prm.Hq, BT)) return cudaErrorInvalidValue;
  if (!make_block_map(&tk, k, D, prm.Nkv, prm.B * prm.Hkv, BT)) return cudaErrorInvalidValue;
  if (!make_block_map(&tv, v, D, prm.Nkv, prm.B * prm.Hkv, BT)) return cudaErrorInvalidValue;
  static std::atomic<int> attr_set[64];
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    attr_set[device].store(1, std::memory_order_release);
  }
  const int64_t prep_rows_per_cta = 256 / (D / 8);
  const int64_t prep_blocks = ((int64_t)prm.B * prm.Hq * prm.nq_pad + prep_rows_per_cta - 1) / prep_rows_per_cta;
  const int64_t g_dkdv = (int64_t)prm.B * prm.Hkv * ((prm.Nkv + BT - 1) / BT);
  const int64_t g_dq = (int64_t)prm.B * prm.Hq * (((prm.Nq + BT - 1) / BT + 1) / 2);
  if (prep_blocks > 0x7fffffffLL || g_dkdv > 0x7fffffffLL || g_dq > 0x7fffffffLL)
    return cudaErrorInvalidConfiguration;
  attn_bwd_prep_kernel<<<(unsigned)prep_blocks, 256, 0, st>>>(prm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_dkdv_kernel<D><<<(unsigned)g_dkdv, THREADS, SM_DKDV, st>>>(tq, tdo, tk, tv, prm);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  attn_bwd_dq_kernel<D><<<(unsigned)g_dq, DQ_THREADS, dql.smem, st>>>(tq, tdo, tk, tv, prm, dql);
  return cudaGetLastError();
}

cudaError_t launch_zero(void *x, int64_t n, int sms, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n / 8 + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  attn_bwd_zero_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<__nv_bfloat16 *>(x), n);
  return cudaGetLastError();
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace attn

extern "C" int attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                        const float *lse, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Nq, int Nkv,
                        int D, float scale, int causal, attn_stream_t stream) {
  using namespace attn;
  int rc = check_problem(B, Hq, Hkv, Nq, Nkv, D, causal);
  if (rc != ATTN_OK) return rc;
  if (D != 64 && D != 128) return ATTN_ERR_ARG;
  if (!isfinite(scale)) return ATTN_ERR_ARG;
  if (B == 0 || (Nq == 0 && Nkv == 0)) return ATTN_OK;
  const bool has_q = Nq > 0, has_k = Nkv > 0;
  if (has_q && (!q || !o || !dout || !lse || !dq)) return ATTN_ERR_ARG;
  if (has_k && (!k || !v || !dk || !dv)) return ATTN_ERR_ARG;
  if (has_q && (!aligned16(q) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) || !aligned16(dq)))
    return ATTN_ERR_ALIGN;
  if (has_k && (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv))) return ATTN_ERR_ALIGN;
  int device = 0, sms = 0, *status = nullptr;
  if ((rc = current_device(&device, &sms, &status)) != ATTN_OK) return rc;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  // one side empty: the other side's gradients are zero
  if (!has_q || !has_k) {
    if (!has_q) {
      e = launch_zero(dk, (int64_t)B * Hkv * Nkv * D, sms, st);
      if (e == cudaSuccess) e = launch_zero(dv, (int64_t)B * Hkv * Nkv * D, sms, st);
    } else {
      e = launch_zero(dq, (int64_t)B * Hq * Nq * D, sms, st);
    }
    return e == cudaSuccess ? ATTN_OK : record_cuda_error(e);
  }
  BwdParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.o = static_cast<const __nv_bfloat16 *>(o);
  prm.dout = static_cast<const __nv_bfloat16 *>(dout);
  prm.lse = lse;
  prm.dq = static_cast<__nv_bfloat16 *>(dq);
  prm.dk = static_cast<__nv_bfloat16 *>(dk);
  prm.dv = static_cast<__nv_bfloat16 *>(dv);
  prm.B = B; prm.Hq = Hq; prm.Hkv = Hkv; prm.Nq = Nq; prm.Nkv = Nkv; prm.D = D;
  prm.nq_pad = (Nq + BT - 1) / BT * BT;
  prm.scale = scale;
  prm.causal = causal;
  prm.status = status;
  prm.wait_limit_ns = wait_limit_ns();
  // per-row vectors, stream-ordered from the library's pool
  const size_t vec_bytes = (size_t)B * Hq * prm.nq_pad * sizeof(float);
  void *ws = nullptr;
  if (scratch_alloc(&ws, 2 * vec_bytes, st) != cudaSuccess || !ws) {
    cudaGetLastError();
    return ATTN_ERR_NOMEM;
  }
  prm.lse2 = static_cast<float *>(ws);
  prm.delta = prm.lse2 + (size_t)B * Hq * prm.nq_pad;
  const auto *qb = static_cast<const __nv_bfloat16 *>(q);
  const auto *kb = static_cast<const __nv_bfloat16 *>(k);
  const auto *vb = static_cast<const __nv_bfloat16 *>(v);
  e = D == 64 ? launch_bwd_d<64>(prm, qb, kb, vb, device, st) : launch_bwd_d<128>(prm, qb, kb, vb, device, st);
  const cudaError_t f = cudaFreeAsync(ws, st);
  if (e == cudaSuccess) e = f;
  return e == cudaSuccess ? ATTN_OK : record_cuda_error(e);
}
