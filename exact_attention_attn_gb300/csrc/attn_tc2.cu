// Exact attention forward for head dims 64 and 128: two 128-row query tiles
// per CTA in ping-pong on the sm_103a tensor cores.
//
// The online softmax is the one of "FlashAttention v1/v2/v3/v4" (lo0.es),
// "El truco que hizo posible todo: online softmax", with the conditional
// rescaling of its "FA4 -- la asimetria de Blackwell" section (rescale only
// when the running max grows by more than TAU in log2 units).  The overlap
// follows the producer/consumer warp specialisation and the two-warpgroup
// ping-pong of its "FA3 -- el momento Hopper" section, rebuilt on tcgen05:
// while warpgroup 0 turns S0 into P0, the tensor core runs P1 V and Q1 K^T
// for the other tile, and the other way round.  Both tiles share every K and
// V block loaded into shared memory.
//
// CTA = 11 warps:
//   warps 0-3 softmax + epilogue of tile 0, warps 4-7 of tile 1
//   (one query row per thread; warp w touches TMEM lanes 32(w%4)..+31)
//   warp 8  TMA producer of Q and K (one thread)
//   warp 9  TMEM allocator and MMA issuer (one thread)
//   warp 10 TMA producer of V (one thread)
//
// TMEM columns: S_t at [128t, 128t+128) fp32, with P_t (bf16 pairs) written
// over its first 64 columns; O_t at [256 + 128t, 256 + 128t + D) fp32.
//
// MMA issue order per block j: PV0_j, S0_{j+1}, PV1_j, S1_{j+1}.  Both the
// overwrite of P_t by S_t,{j+1} and the rescale of O_t rely on tcgen05.mma
// executing in issue order and on tcgen05.commit tracking every earlier MMA of
// the issuing thread: the commit that announces S_t,j also covers PV_t,{j-1},
// so O_t may be rescaled as soon as S_t,j is visible.
#include <math.h>
#include <string.h>

#include <atomic>

#include "attn_internal.h"
#include "attn_mask.cuh"
#include "sm100_ptx.cuh"

// Optional per-role timestamps (clock64) for 8 CTAs starting at
// attn_trace_first, compiled in only when ATTN_TRACE is defined:
// ATTN_TRACE_EV(row, col) stores into the caller-provided buffer
// attn_trace_buf[cta - attn_trace_first][32][64] (pointer read once per thread
// by ATTN_TRACE_SETUP).
#ifdef ATTN_TRACE
__device__ long long *attn_trace_buf;
__device__ unsigned attn_trace_first;
#define ATTN_TRACE_SETUP                                                           \
  const unsigned attn_tcta = blockIdx.x - attn_trace_first;                       \
  long long *const attn_tbuf = (attn_tcta < 8u) ? attn_trace_buf : nullptr
#define ATTN_TRACE_EV(row, col)                                                              \
  do {                                                                                       \
    const long long _t = clock64();                                                          \
    if (attn_tbuf && (col) < 64) attn_tbuf[((long long)attn_tcta * 32 + (row)) * 64 + (col)] = _t; \
  } while (0)
#else
#define ATTN_TRACE_SETUP \
  do {                   \
  } while (0)
#define ATTN_TRACE_EV(row, col) \
  do {                          \
  } while (0)
#endif
// Optional per-CTA start/end stamps (globaltimer ns) and SM id, compiled in
// only when ATTN_TRACE_CTA is defined: attn_cta_buf[cta][4] = {start, end, sm}.
#ifdef ATTN_TRACE_CTA
__device__ long long *attn_cta_buf;
#define ATTN_CTA_EV(slot)                                                                          \
  do {                                                                                             \
    if (threadIdx.x == 0 && attn_cta_buf) {                                                        \
      uint32_t _sm;                                                                                \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(_sm));                                             \
      attn_cta_buf[(long long)blockIdx.x * 4 + (slot)] = (long long)ptx::globaltimer_ns();          \
      attn_cta_buf[(long long)blockIdx.x * 4 + 2] = _sm;                                           \
    }                                                                                              \
  } while (0)
#else
#define ATTN_CTA_EV(slot) \
  do {                    \
  } while (0)
#endif

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128, BN = 128;
constexpr int CHUNK_BYTES = 128 * 128;
#ifdef ATTN_TRACE
constexpr int THREADS = 384;  // + a trace-only observer warp
#else
constexpr int THREADS = 352;
#endif
constexpr int WARP_LOAD_K = 8, WARP_LOAD_V = 10, WARP_MMA = 9;
constexpr uint32_t TMEM_COLS = 512;
constexpr float TAU = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int MAX_KST = 8, MAX_VST = 3;
#ifndef ATTN_TC2_PREFETCH
#define ATTN_TC2_PREFETCH 0
#endif
constexpr int kPrefetch = ATTN_TC2_PREFETCH;  // L2 prefetch distance in blocks
// pairs q with bit (q % 8) set take the FMA-pipe exp2 (none by default: the
// MUFU ex2 alone is faster at the current balance of the softmax warps)
#ifndef ATTN_TC2_POLY_PAIRS
#define ATTN_TC2_POLY_PAIRS 0
#endif
constexpr unsigned kPolyPairs = ATTN_TC2_POLY_PAIRS;
#ifdef ATTN_TC2_MMA_SPIN
#define MMA_WAIT mbar_wait_spin
#else
#define MMA_WAIT mbar_wait
#endif
constexpr int kSmemMax = 232448;

struct Params2 {
  Problem p;
  int npairs;        // tile pairs per head
  int head_chunk;    // (b, hq) heads per chunk of the work order (whole GQA groups)
  int kst, vst;      // K ring (16 KB chunks), V ring (blocks)
  uint32_t off_k, off_v, off_bar;
  uint64_t wait_limit_ns;
};

struct Bars2 {
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

__device__ __forceinline__ void raise_abort(Bars2 *bars, int *status) {
  atomicCAS(status, 0, kStatusTimeout);
  *reinterpret_cast<volatile int *>(&bars->abort) = 1;
}

// One quarter (32 keys) of a masked block for one row: y = s * scale + mask
// (natural-log units) on f32x2 pairs into y2[0..16), the block max in two
// chains.  CUT: keys at or past vis_end give -inf (blocks where some row of
// the warp has such keys).
template <bool CUT>
__device__ __forceinline__ void mask_quarter(const uint32_t (&cur)[32], const uint32_t *mk16, uint64_t *y2,
                                             uint64_t sc2, int key0, int vis_end, float &mx0, float &mx1) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t w = mk16[i];
    uint64_t v = f2_fma(f2_pack(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])), sc2,
                        f2_pack(bf16_lo(w), bf16_hi(w)));
    float y0, y1;
    f2_unpack(v, y0, y1);
    if (CUT) {
      if (key0 + 2 * i >= vis_end) y0 = -INFINITY;
      if (key0 + 2 * i + 1 >= vis_end) y1 = -INFINITY;
      v = f2_pack(y0, y1);
    }
    y2[i] = v;
    if (i & 1)
      mx1 = max3f(mx1, y0, y1);
    else
      mx0 = max3f(mx0, y0, y1);
  }
}

// MODE 0: the scale is positive (scores and their maxima keep their order);
// MODE 1: the scale is zero or negative (block minima of the raw scores);
// MODE 2: an additive mask, either sign (block maxima of the masked, scaled
// scores).  One instantiation per mode keeps each one's code small.
template <int D, int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    attn_tc2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params2 prm) {
  constexpr int NC = D / 64;  // 64-column chunks per row
  constexpr bool POS = MODE == 0, MASK = MODE == 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t *sq = smem;  // Q tile t: its NC chunks at t*NC*16 KB + c*16 KB
  uint8_t *sk = smem + prm.off_k;
  uint8_t *sv = smem + prm.off_v;
  Bars2 *bars = reinterpret_cast<Bars2 *>(smem + prm.off_bar);
  volatile int *abortf = &bars->abort;

  const Problem &p = prm.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t limit = prm.wait_limit_ns;
  ATTN_TRACE_SETUP;
  ATTN_CTA_EV(0);
  if (tid == 0) ATTN_TRACE_EV(19, 0);

  // ---- work unit: heads in chunks of head_chunk; inside a chunk (b, hq)
  //      fastest, then tile pair (heaviest causal pairs first).  A chunk
  //      holds at least three waves of units, so the heaviest-first order
  //      still balances the SMs, while only its heads' K and V are live in
  //      L2 (GQA causal B2 Hq32 Hkv8 N8192: DRAM reads 356 -> 201 MB)
  const int BH = p.B * p.Hq;
  const int nsplit = p.kv_splits;
  const int split = blockIdx.x % nsplit;
  const int unit = blockIdx.x / nsplit;
  const int c_units = prm.head_chunk * prm.npairs;
  const int c_idx = unit / c_units;
  const int c_first = c_idx * prm.head_chunk;
  const int hc_here = min(prm.head_chunk, BH - c_first);  // the last chunk may be short
  const int r_in = unit - c_idx * c_units;
  const int bh = c_first + r_in % hc_here;
  const int t_idx = r_in / hc_here;
  const int pair = p.causal ? (prm.npairs - 1 - t_idx) : t_idx;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int bkv = b * p.Hkv + hq / (p.Hq / p.Hkv);
  const int shift = p.Nkv - p.Nq;
  int nblk_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int q0 = pair * 2 * BM + t * BM;
    int kv_end = p.Nkv;
    if (p.causal) kv_end = max(0, min(p.Nkv, q0 + BM - 1 + shift + 1));
    nblk_t[t] = (q0 < p.Nq) ? (kv_end + BN - 1) / BN : 0;
  }
  // this CTA's key blocks: [jb, jb + nblk) of the pair's range, split evenly;
  // from here on nblk_t[t] counts the blocks tile t takes in that range and
  // every block index j is relative to jb
  const int nall = max(nblk_t[0], nblk_t[1]);
  const int jb = (int)((int64_t)split * nall / nsplit);
  const int je = (int)((int64_t)(split + 1) * nall / nsplit);
#pragma unroll
  for (int t = 0; t < 2; ++t) nblk_t[t] = max(0, min(je, nblk_t[t]) - jb);
  const int nblk = je - jb;

  if (tid == 0) {
    mbar_init(&bars->q_full, 2);  // one Q tile from each producer
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
    // Two independent producer threads (Q0+K and Q1+V), each moving a whole
    // 128-row tile or 128-key block (all D/64 chunks) with one 4-D TMA copy:
    // copies issued by one thread are processed one after the other, so the
    // two query tiles travel in parallel.
    if (lane == 0 && nblk > 0) {
      const bool is_k = warp == WARP_LOAD_K;
      uint32_t ctr = 0;
      int slot = 0;
      uint32_t phase = 0;
      uint32_t skipped = 0xffffffffu;  // a copy never issued (test support)
      bool ok = true;
      tma_prefetch_desc(&tm_q);
      // query tile 0 (K producer) or 1 (V producer), zero-filled past Nq
      const int qt = is_k ? 0 : 1;
      mbar_arrive_expect_tx(&bars->q_full, NC * CHUNK_BYTES);
      tma_load_4d(sq + qt * NC * CHUNK_BYTES, &tm_q, &bars->q_full, 0, pair * 2 * BM + qt * BM, 0, bh);
      if (is_k) {
        tma_prefetch_desc(&tm_k);
        // warm L2 with the first blocks; later ones are prefetched kPrefetch
        // blocks ahead of their shared-memory copy
        for (int j = 0; j < kPrefetch && j < nblk; ++j) tma_prefetch_4d(&tm_k, 0, (jb + j) * BN, 0, bkv);
        for (int j = 0; j < nblk; ++j) {
          if (j + kPrefetch < nblk) tma_prefetch_4d(&tm_k, 0, (jb + j + kPrefetch) * BN, 0, bkv);
          if (!mbar_wait(&bars->k_empty[slot], phase ^ 1u, abortf, limit)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars->k_full[slot], NC * CHUNK_BYTES);
          tma_load_4d(sk + slot * NC * CHUNK_BYTES, &tm_k, &bars->k_full[slot], 0, (jb + j) * BN, 0, bkv);
          ATTN_TRACE_EV(13, j);
          ++ctr;
          if (++slot == prm.kst) {
            slot = 0;
            phase ^= 1u;
          }
        }
      } else {
        tma_prefetch_desc(&tm_v);
        for (int j = 0; j < kPrefetch && j < nblk; ++j) tma_prefetch_4d(&tm_v, 0, (jb + j) * BN, 0, bkv);
        for (int j = 0; j < nblk; ++j) {
          if (j + kPrefetch < nblk) tma_prefetch_4d(&tm_v, 0, (jb + j + kPrefetch) * BN, 0, bkv);
          const int vs = slot;
          if (!mbar_wait(&bars->v_empty[vs], phase ^ 1u, abortf, limit)) { ok = false; break; }
          if (++slot == prm.vst) {
            slot = 0;
            phase ^= 1u;
          }
          if ((p.debug_flags & 1) && j == 1) {  // test support: leave this slot empty
            skipped = ctr;
            ++ctr;
            continue;
          }
          mbar_arrive_expect_tx(&bars->v_full[vs], NC * CHUNK_BYTES);
          tma_load_4d(sv + vs * NC * CHUNK_BYTES, &tm_v, &bars->v_full[vs], 0, (jb + j) * BN, 0, bkv);
          ATTN_TRACE_EV(14, j);
          ++ctr;
        }
      }
      if (!ok) raise_abort(bars, p.status);
      // drain: every copy this thread issued lands before the CTA exits
      mbar_wait_drain(&bars->q_full, 0, limit);
      if (is_k) {
        const uint32_t kn = ctr < (uint32_t)prm.kst ? ctr : (uint32_t)prm.kst;
        for (uint32_t i = ctr - kn; i < ctr; ++i) mbar_wait_drain(&bars->k_full[i % prm.kst], (i / prm.kst) & 1, limit);
      } else {
        const uint32_t vn = ctr < (uint32_t)prm.vst ? ctr : (uint32_t)prm.vst;
        for (uint32_t i = ctr - vn; i < ctr; ++i)
          if (i != skipped) mbar_wait_drain(&bars->v_full[i % prm.vst], (i / prm.vst) & 1, limit);
      }
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nblk > 0) {
      const uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      const uint32_t idesc_pv = idesc_bf16(BM, D, 0, 1);
      bool ok = MMA_WAIT(&bars->q_full, 0, abortf, limit);
      ATTN_TRACE_EV(25, 0);
      // Descriptors of K-major 128B-swizzled chunks (a K=16 step adds 32 bytes,
      // 2 in the >>4 address field): Q tile t chunk c at sq + (t*NC + c)*16 KB;
      // K block in ring slot s at sk + s*NC*16 KB.
      // V (MN-major): a K=16 step is 16 keys, 2048 bytes.
      constexpr uint64_t kChunkD = CHUNK_BYTES >> 4, kBlkD = (uint64_t)(NC * CHUNK_BYTES) >> 4;
      const uint64_t qd_base = smem_desc(smem_u32(sq), 16, 1024);
      const uint64_t kd_base = smem_desc(smem_u32(sk), 16, 1024);
      const uint64_t vd_base = smem_desc(smem_u32(sv), CHUNK_BYTES, 1024);
      // ring positions (slot, phase) of the next K block and of V block j
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      // S_t = Q_t K^T for the K block at the current ring position
      auto issue_s = [&](int t, bool wait_full, bool release) -> bool {
        if (wait_full && !MMA_WAIT(&bars->k_full[ks], kph, abortf, limit)) return false;
        if (wait_full) ATTN_TRACE_EV(12, 0);
        tc_fence_after();
        const uint64_t qd0 = qd_base + (uint64_t)t * kBlkD, kd0 = kd_base + (uint64_t)ks * kBlkD;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + 128 * t, qd0 + (uint64_t)(c * kChunkD + kk * 2), kd0 + (uint64_t)(c * kChunkD + kk * 2),
                   idesc_s, (c | kk) != 0);
        }
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
      // from block 0 on, V_j and K_{j+1} have landed once P of the block's first
      // tile is complete (a softmax thread of that tile waits for both before it
      // arrives), so this thread waits only for P
      for (int j = 0; j < nblk && ok; ++j) {
        ATTN_TRACE_EV(10, j);
        ATTN_TRACE_EV(11, j);
        const uint64_t vd0 = vd_base + (uint64_t)vs * kBlkD;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!act(t, j)) continue;
          if (!MMA_WAIT(&bars->p_full[t], j & 1, abortf, limit)) { ok = false; break; }
          ATTN_TRACE_EV(8 + t, j);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + 256 + 128 * t, tmem + 128 * t + kk * 8, vd0 + (uint64_t)(kk * (2048 >> 4)), idesc_pv,
                   (j > 0 || kk > 0) ? 1u : 0u);
          if (t == 0) ATTN_TRACE_EV(18, j);
          if (j == nblk_t[t] - 1) mma_commit(&bars->o_done[t]);
          if (act(t, j + 1)) {
            const bool last = (t == 1) || !act(1, j + 1);
            if (!issue_s(t, false, last)) { ok = false; break; }
          }
          if (t == 0) ATTN_TRACE_EV(15, j);
        }
        if (!ok) break;
        mma_commit(&bars->v_empty[vs]);
        next_k();
        if (++vs == prm.vst) {
          vs = 0;
          vph ^= 1u;
        }
      }
      if (!ok) raise_abort(bars, p.status);
      mma_commit(&bars->done);
      if (!mbar_wait_drain(&bars->done, 0, limit)) raise_abort(bars, p.status);
    }
#ifdef ATTN_TRACE
  } else if (warp == 11) {
    // trace-only observer: records when each K and V block lands
    if (lane == 0 && nblk > 0) {
      for (int j = 0; j < nblk; ++j) {
        if (!mbar_wait(&bars->k_full[j % prm.kst], (j / prm.kst) & 1, abortf, limit)) break;
        ATTN_TRACE_EV(16, j);
        if (!mbar_wait(&bars->v_full[j % prm.vst], (j / prm.vst) & 1, abortf, limit)) break;
        ATTN_TRACE_EV(17, j);
      }
    }
#endif
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue
    const int t = warp >> 2;          // tile of this warpgroup
    const int row = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + 128 * t;
    const uint32_t tO = tmem + lane_base + 256 + 128 * t;
    const int qi = pair * 2 * BM + t * BM + row;
    const int nb = nblk_t[t];
    const int vis_end = p.causal ? min(p.Nkv, qi + shift + 1) : p.Nkv;
    const float sl2 = p.scale * kLog2e;
    constexpr bool pos = POS;  // sl2 > 0, decided by the host
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    const Exp2Poly exp2_poly;
    const __nv_bfloat16 *mrow = MASK ? mask_row(p, b, hq, qi) : nullptr;

    const bool tr = (tid & 127) == 0;
    // ring positions of V_j and K_{j+1}, followed by thread 0 of the tile in one
    // register: V slot bits 0-7, K slot bits 8-15, V phase bit 16, K phase bit 24
    uint32_t ring = 1u << 8;
    for (int j = 0; j < nb; ++j) {
      const int kbase = (jb + j) * BN;
      const bool full = kbase + BN <= vis_end;  // no masked key in this block for this row
      // the mask values of this row and block, on their way while S_t,j is computed
      uint32_t mk[MASK ? 64 : 1];
      if constexpr (MASK) mask_load<128>(mk, mrow, kbase, p.Nkv);
      if (tr) ATTN_TRACE_EV(4 * t + 0, j);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[t], j & 1, abortf, limit))) { ok = false; break; }
      if (tr) ATTN_TRACE_EV(4 * t + 1, j);
      tc_fence_after();
      float mblk;
      uint64_t y2[MASK ? BN / 2 : 1];
      if constexpr (MASK) {
        // y = s * scale + mask (natural-log units, kept for P) a quarter at a
        // time, so that each quarter's mask values are dead once used; the
        // block max of y times log2 e is the block max of the log2-unit scores
        // (rounding is monotone)
        const bool cut = !__all_sync(0xffffffffu, full);
        const uint64_t sc2 = f2_pack(p.scale, p.scale);
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t cur[32];
          tmem_ld32(tS + 32 * h, cur);
          tmem_wait_ld();
          reg_fence32(cur);
          if (cut)
            mask_quarter<true>(cur, mk + 16 * h, y2 + 16 * h, sc2, kbase + 32 * h, vis_end, mx0, mx1);
          else
            mask_quarter<false>(cur, mk + 16 * h, y2 + 16 * h, sc2, kbase + 32 * h, vis_end, mx0, mx1);
        }
        mblk = fmaxf(mx0, mx1) * kLog2e;
      } else {
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sr[cc]);
      tmem_wait_ld();
      if (tr) ATTN_TRACE_EV(4 * t + 2, j);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) reg_fence32(sr[cc]);
      float x[BN];
#pragma unroll
      for (int c = 0; c < BN; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]);

      if (!full) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (kbase + c >= vis_end) x[c] = pos ? -INFINITY : INFINITY;
      }
      // block max (min when scale < 0) of the raw scores, four chains of 3-input ops
      if (pos) {
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < BN; c += 8) {
          mx0 = max3f(mx0, x[c + 0], x[c + 1]);
          mx1 = max3f(mx1, x[c + 2], x[c + 3]);
          mx2 = max3f(mx2, x[c + 4], x[c + 5]);
          mx3 = max3f(mx3, x[c + 6], x[c + 7]);
        }
        const float ext = max3f(mx0, mx1, fmaxf(mx2, mx3));
        mblk = (ext == -INFINITY) ? -INFINITY : ext * sl2;
      } else {
        float mn[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
#pragma unroll
        for (int c = 0; c < BN; c += 4)
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) mn[k4] = fminf(mn[k4], x[c + k4]);
        const float ext = fminf(fminf(mn[0], mn[1]), fminf(mn[2], mn[3]));
        // ext*sl2 is the block max of the scaled scores; masked-only rows give -inf
        mblk = (ext == INFINITY) ? -INFINITY : (sl2 == 0.f ? 0.f : ext * sl2);
      }
      }  // not MASK
      const float m_new = fmaxf(m_use, mblk);
      if (__any_sync(0xffffffffu, m_new > m_use + TAU)) {
        const float alpha = (m_use == -INFINITY) ? 0.f : ex2_approx(m_use - m_new);
        if (j > 0) {
          // PV_t,{j-1} is complete: the commit that announced S_t,j covers it
#pragma unroll 1
          for (int cc = 0; cc < D / 16; ++cc) {
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
      const float mu = (m_use == -INFINITY) ? 0.f : m_use;
      // the branch must be warp-uniform: both sides end in the warp-collective
      // tcgen05.st, which every lane of the warp has to execute together
      if constexpr (MASK) {
        // P = 2^(y log2 e - mu), a quarter at a time into columns [16h, 16h+16)
        const uint64_t l2e2 = f2_pack(kLog2e, kLog2e), nmu2 = f2_pack(-mu, -mu);
        uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float a0, a1;
            f2_unpack(f2_fma(y2[16 * h + i], l2e2, nmu2), a0, a1);
            const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
            if (i & 1)
              acc1 = f2_add(acc1, f2_pack(p0, p1));
            else
              acc0 = f2_add(acc0, f2_pack(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + h * 16, pk);
        }
        float s0, s1, s2, s3;
        f2_unpack(acc0, s0, s1);
        f2_unpack(acc1, s2, s3);
        l += (s0 + s1) + (s2 + s3);
      } else if (pos && __all_sync(0xffffffffu, full)) {
        // every key visible and scale > 0: y = s*sl2 - mu on f32x2 pairs,
        // exp2 on the MUFU (pairs selected by kPolyPairs on the FMA pipe)
        // The scores are read again from TMEM a quarter at a time (the next
        // quarter's load in flight while this one is turned into P), so only
        // 64 of them are live here: P quarter h lands in columns [16h, 16h+16),
        // already read, while the load in flight reads [32(h+1), 32(h+2)).
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nmu2 = f2_pack(-mu, -mu);
        uint64_t acc0 = 0ull, acc1 = 0ull;
        uint32_t qbuf[2][32];
        tmem_ld32(tS, qbuf[0]);
        tmem_wait_ld();
        reg_fence32(qbuf[0]);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t(&cur)[32] = qbuf[h & 1];
          if (h < 3) tmem_ld32(tS + 32 * (h + 1), qbuf[(h + 1) & 1]);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int q = h * 16 + i;
            const uint64_t y =
                f2_fma(f2_pack(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])), sl2x2, nmu2);
            uint64_t p2;
            if ((kPolyPairs >> (q & 7)) & 1) {
              p2 = exp2_poly(y);
            } else {
              float y0, y1;
              f2_unpack(y, y0, y1);
              p2 = f2_pack(ex2_approx(y0), ex2_approx(y1));
            }
            if (i & 1)
              acc1 = f2_add(acc1, p2);
            else
              acc0 = f2_add(acc0, p2);
            float p0, p1;
            f2_unpack(p2, p0, p1);
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + h * 16, pk);
          if (h < 3) {
            tmem_wait_ld();
            reg_fence32(qbuf[(h + 1) & 1]);
          }
        }
        float a0, a1, b0, b1;
        f2_unpack(acc0, a0, a1);
        f2_unpack(acc1, b0, b1);
        l += (a0 + a1) + (b0 + b1);
      } else {
        // a block with masked keys (or scale <= 0): the scores are read again a
        // quarter at a time as above, and a masked key gives exactly 0.  One
        // quarter's code, looped: unrolling it measured 3 % slower overall
        // (this kernel is sensitive to the size of its code).  A quarter
        // whose keys every row of the warp sees needs no test per key, and
        // one that no row of the warp sees is not read at all (on a causal
        // diagonal block warp w has w of the first kind and 3 - w of the
        // second)
        const int vis_lo = __reduce_min_sync(0xffffffffu, vis_end);
        const int vis_hi = __reduce_max_sync(0xffffffffu, vis_end);
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int h = 0; h < 4; ++h) {
          const int c0 = kbase + 32 * h;
          uint32_t pk[16];
          if (c0 >= vis_hi) {  // warp-uniform: every key hidden
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = 0u;
          } else {
            uint32_t cur[32];
            tmem_ld32(tS + 32 * h, cur);
            tmem_wait_ld();
            reg_fence32(cur);
            if (c0 + 32 <= vis_lo) {  // warp-uniform: every key visible
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float p0 = ex2_approx(fmaf(__uint_as_float(cur[2 * i]), sl2, -mu));
                const float p1 = ex2_approx(fmaf(__uint_as_float(cur[2 * i + 1]), sl2, -mu));
                ls[i & 3] += p0 + p1;
                pk[i] = pack_bf16x2(p0, p1);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float a = __uint_as_float(cur[2 * i]), bb = __uint_as_float(cur[2 * i + 1]);
                const float p0 = (c0 + 2 * i >= vis_end) ? 0.f : ex2_approx(fmaf(a, sl2, -mu));
                const float p1 = (c0 + 2 * i + 1 >= vis_end) ? 0.f : ex2_approx(fmaf(bb, sl2, -mu));
                ls[i & 3] += p0 + p1;
                pk[i] = pack_bf16x2(p0, p1);
              }
            }
          }
          tmem_st16(tS + h * 16, pk);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      }
      tmem_wait_st();
      tc_fence_before();
      // the block's first tile (tile 0, or tile 1 where tile 0 has no keys in
      // this block) vouches for V_j and K_{j+1}: the MMA thread then needs to
      // wait for P alone
      if (row == 0 && (t == 0 || j >= nblk_t[0])) {
        bool got = mbar_wait(&bars->v_full[ring & 0xffu], (ring >> 16) & 1u, abortf, limit);
        if (got && j + 1 < nblk) got = mbar_wait(&bars->k_full[(ring >> 8) & 0xffu], ring >> 24, abortf, limit);
        if (!got) raise_abort(bars, p.status);  // every role stops waiting
      }
      if (row == 0) {
        ring += 1u;
        if ((ring & 0xffu) == (uint32_t)prm.vst) ring = (ring & ~0xffu) ^ (1u << 16);
        ring += 1u << 8;
        if (((ring >> 8) & 0xffu) == (uint32_t)prm.kst) ring = (ring & ~0xff00u) ^ (1u << 24);
      }
      mbar_arrive(&bars->p_full[t]);
      if (tr) ATTN_TRACE_EV(4 * t + 3, j);
    }
    if (!ok) raise_abort(bars, p.status);

    // ---- epilogue
    if (ok && nb > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_done[t], 0, abortf, limit))) {
        raise_abort(bars, p.status);
        ok = false;
      }
      if (tr) ATTN_TRACE_EV(21 + t, 0);
    }
    if (ok) {
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const float lse_val = (m_use == -INFINITY || !(l > 0.f)) ? -INFINITY : (m_use + log2f(l)) * kLn2;
      const int64_t row_idx = (int64_t)bh * p.Nq + qi;
      if (nsplit == 1) {
        __nv_bfloat16 *orow = p.o + row_idx * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t r[32];
          if (nb > 0) {
            tmem_ld32(tO + cc * 32, r);
            tmem_wait_ld();
            reg_fence32(r);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          if (qi < p.Nq) {
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
        if (qi < p.Nq) p.lse[row_idx] = lse_val;
      } else {
        // partial result of this key range: O_s = acc / l_s (fp32), LSE_s
        const int64_t ws_row = (int64_t)split * BH * p.Nq + row_idx;
        float *orow = p.ws_o + ws_row * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t r[32];
          if (nb > 0) {
            tmem_ld32(tO + cc * 32, r);
            tmem_wait_ld();
            reg_fence32(r);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          if (qi < p.Nq) {
            float4 *dst = reinterpret_cast<float4 *>(orow + cc * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(__uint_as_float(r[v4 * 4 + 0]) * inv, __uint_as_float(r[v4 * 4 + 1]) * inv,
                                    __uint_as_float(r[v4 * 4 + 2]) * inv, __uint_as_float(r[v4 * 4 + 3]) * inv);
          }
        }
        if (qi < p.Nq) p.ws_lse[ws_row] = lse_val;
      }
    }
  }

  if ((tid & 127) == 0 && warp < 8) ATTN_TRACE_EV(23 + (warp >> 2), 0);
  tc_fence_before();
  __syncthreads();
  if (tid == 0) ATTN_TRACE_EV(20, 0);
  ATTN_CTA_EV(1);
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Heads per chunk of the work order: as many chunks as the units (head x
// tile pair) fill three waves of one CTA per SM, each of whole GQA groups,
// the groups dealt evenly; one chunk (plain heaviest-first order) when the
// problem is smaller.  Three waves per chunk keep a chunk's heaviest units
// early enough in it that they end with the rest.
int head_chunk(const Problem &p, int npairs, int device) {
  static std::atomic<int> sm_count[64];
  int sms = device >= 0 && device < 64 ? sm_count[device].load(std::memory_order_relaxed) : 0;
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0) sms = 1;
    if (device >= 0 && device < 64) sm_count[device].store(sms, std::memory_order_relaxed);
  }
  const int BH = p.B * p.Hq, g = p.Hq / p.Hkv;
  if (BH <= 0 || g <= 0) return 1;
  const int64_t groups = BH / g;
  int64_t chunks = (int64_t)BH * npairs / (3 * (int64_t)sms);
  if (chunks < 1) chunks = 1;
  if (chunks > groups) chunks = groups;
  return (int)((groups + chunks - 1) / chunks * g);
}

template <int D, int MODE>
cudaError_t launch_tc2_d(const Problem &p, int device, uint64_t wait_limit_ns, cudaStream_t stream) {
  constexpr int NC = D / 64;
  const int avail = kSmemMax - 2048;
  const int qb = 2 * NC * CHUNK_BYTES, blkb = NC * CHUNK_BYTES;
  // K and V rings in whole blocks; at least two of each, the rest to K
  int vst = 2, kst = (avail - qb - vst * blkb) / blkb;
  if (kst > MAX_KST) kst = MAX_KST;
  if (kst > 2 && vst < MAX_VST && kst > vst + 1) {
    const int spare = kst - (vst + 1);
    vst += spare / 2 < MAX_VST - vst ? spare / 2 : MAX_VST - vst;
    kst = (avail - qb - vst * blkb) / blkb;
    if (kst > MAX_KST) kst = MAX_KST;
  }
#ifdef ATTN_TC2_VST
  vst = ATTN_TC2_VST;
  kst = (avail - qb - vst * blkb) / blkb;
  if (kst > MAX_KST) kst = MAX_KST;
#endif
  if (kst < 2 || vst < 2) return cudaErrorInvalidConfiguration;
  Params2 prm;
  memset(&prm, 0, sizeof(prm));
  prm.p = p;
  prm.npairs = ((p.Nq + BM - 1) / BM + 1) / 2;
  // a mask shared by every head is read best with all heads in step (the
  // plain heaviest-first order): every head then reads each mask row at once
  prm.head_chunk = (MODE == 2 && p.mask_sh == 0) ? p.B * p.Hq : head_chunk(p, prm.npairs, device);
  prm.kst = kst;
  prm.vst = vst;
  prm.off_k = qb;
  prm.off_v = qb + kst * blkb;
  prm.off_bar = prm.off_v + vst * blkb;
  prm.wait_limit_ns = wait_limit_ns;
  const int smem = prm.off_bar + (int)sizeof(Bars2) + 1024;
  if (smem > kSmemMax) return cudaErrorInvalidConfiguration;
  CUtensorMap tq, tk, tv;
  if (!make_block_map(&tq, p.q, D, p.Nq, p.B * p.Hq, BM)) return cudaErrorInvalidValue;
  if (!make_block_map(&tk, p.k, D, p.Nkv, p.B * p.Hkv, BN)) return cudaErrorInvalidValue;
  if (!make_block_map(&tv, p.v, D, p.Nkv, p.B * p.Hkv, BN)) return cudaErrorInvalidValue;
  static std::atomic<int> attr_set[64];
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc2_kernel<D, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    attr_set[device].store(1, std::memory_order_release);
  }
  const int64_t grid = (int64_t)prm.npairs * p.B * p.Hq * p.kv_splits;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  attn_tc2_kernel<D, MODE><<<(unsigned)grid, THREADS, smem, stream>>>(tq, tk, tv, prm);
  return cudaGetLastError();
}

}  // namespace

bool tc2_supports(int D) { return D == 64 || D == 128; }

cudaError_t launch_tc2(const Problem &p, int device, uint64_t wait_limit_ns, cudaStream_t stream) {
  // the same product as the kernel's, so that both sides agree on its sign
  const bool pos = p.scale * kLog2e > 0.f;
  if (p.D == 64) {
    if (p.mask) return launch_tc2_d<64, 2>(p, device, wait_limit_ns, stream);
    return pos ? launch_tc2_d<64, 0>(p, device, wait_limit_ns, stream) : launch_tc2_d<64, 1>(p, device, wait_limit_ns, stream);
  }
  if (p.D == 128) {
    if (p.mask) return launch_tc2_d<128, 2>(p, device, wait_limit_ns, stream);
    return pos ? launch_tc2_d<128, 0>(p, device, wait_limit_ns, stream)
               : launch_tc2_d<128, 1>(p, device, wait_limit_ns, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
