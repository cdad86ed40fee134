// Exact attention forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Algorithm: the tiled online softmax of "FlashAttention v1/v2/v3/v4"
// (lo0.es), sections "El truco que hizo posible todo: online softmax" and
// "FA4 -- la asimetria de Blackwell": a 128-row query tile visits the key
// blocks in order; each row keeps a running max m and a running sum l; the
// output accumulator is rescaled by 2^(m_old - m_new) only when the max grows
// by more than TAU (conditional rescaling -- exact, because l, P and O all use
// the same stale max, and P <= 2^TAU stays finite); O is divided by l once at
// the end.  The N x N scores never leave the chip: S lives in TMEM, P is
// written back to TMEM as bf16 and fed to the second MMA from there.
//
// Large head dims follow the FFPA page ("Split-D and TiledMMA"): the D axis is
// cut into 64-column chunks staged one at a time through a fixed-size ring,
// so shared memory holds Br x 64 tiles whatever D is; the output is cut into
// slices of at most 256 columns (the TMEM accumulator budget), each slice a
// separate CTA that recomputes the scores.
//
// CTA = 8 warps:
//   warps 0-3  softmax + correction + epilogue, one query row per thread
//              (warp w may only touch TMEM lanes 32w..32w+31)
//   warps 4, 6 TMA producers of the Q/K ring (one thread each, alternate
//              ring positions; every copy moves two 64-column chunks, 32 KB)
//   warp 5     TMEM allocator and MMA issuer (one thread)
//   warp 7     TMA producer of V (one copy of the block's output slice), idle
//              when V travels through the ring
//
// Shared memory, by head dim: Q resident plus the ring plus a V slot (small
// D); Q resident and V in the ring as 32 KB items next to K (D = 384..512,
// where Q and a V slot do not both fit: streaming Q again for every key
// block would add 128 KB per block to an operand stream that the TMA cannot
// sustain); Q streamed through the ring (D >= 576, Q alone over 144 KB).
//
// TMEM columns: S [0,128) fp32 scores; P0 [128,192) and P1 [192,256) bf16
// pairs (double-buffered); O [256, 256+DV) fp32 output slice.
//
// Synchronisation (mbarriers; every wait is bounded):
//   k_full/k_empty, v_full/v_empty   TMA rings <-> MMA
//   s_full   MMA -> softmax (S_j ready)       s_free  softmax -> MMA (S read)
//   p_full[2] softmax -> MMA (P_j in TMEM)    o_bar[2] MMA -> softmax (PV_j done)
// MMA issue order is S_0, S_1, PV_0, S_2, PV_1, ...; tcgen05.commit after S_j
// therefore also covers PV_{j-2}, which frees P buffer j%2 for P_j and makes
// every parity wait below unambiguous.
#include <math.h>
#include <string.h>

#include <atomic>

#include <cuda.h>

#include "attn_internal.h"
#include "attn_mask.cuh"
#include "sm100_ptx.cuh"

// Optional per-role timestamps (clock64) for 8 CTAs starting at
// attn_tc_trace_first, compiled in only when ATTN_TRACE is defined:
// TC_TRACE_EV(row, col) stores into attn_tc_trace_buf[cta][32][64].
#ifdef ATTN_TRACE
__device__ long long *attn_tc_trace_buf;
__device__ unsigned attn_tc_trace_first;
#define TC_TRACE_SETUP                                                       \
  const unsigned tc_tcta = blockIdx.x - attn_tc_trace_first;                \
  long long *const tc_tbuf = (tc_tcta < 8u) ? attn_tc_trace_buf : nullptr
#define TC_TRACE_EV(row, col)                                                                    \
  do {                                                                                           \
    const long long _t = clock64();                                                              \
    if (tc_tbuf && (col) < 64) tc_tbuf[((long long)tc_tcta * 32 + (row)) * 64 + (col)] = _t;   \
  } while (0)
#else
#define TC_TRACE_SETUP \
  do {                 \
  } while (0)
#define TC_TRACE_EV(row, col) \
  do {                        \
  } while (0)
#endif

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128;                  // query rows per tile (MMA M)
constexpr int BN = 128;                  // keys per block (MMA N of S, K of PV)
constexpr int CHUNK_BYTES = 128 * 128;   // one 128-row x 64-col bf16 tile
constexpr int THREADS = 256;
constexpr int WARP_LOAD_QK0 = 4;
constexpr int WARP_MMA = 5;
constexpr int WARP_LOAD_QK1 = 6;
constexpr int WARP_LOAD_V = 7;
constexpr int SLOT_BYTES = 2 * 128 * 128;  // Q/K ring slot: two 128-row x 64-col chunks
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_P0 = 128, TM_P1 = 192, TM_O = 256;
constexpr float TAU = 8.0f;              // rescale threshold, log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int MAX_KST = 8, MAX_VST = 2;

struct TcParams {
  Problem p;
  int nc;        // contraction chunks = D / 64
  int nslices;   // output slices
  int ntiles;    // query tiles per head
  int kst, vst;  // ring depths (Q/K ring in 32 KB slots; V ring in slices)
  int npairs;    // chunk pairs per block (ceil(nc / 2))
  int qres;      // Q resident in shared memory (else streamed through the K ring)
  int vring;     // V blocks as ring items (2 chunks each) after the next block's K
  int nvitems;   // ring items per V block when vring: ceil(vmax / 2)
  int vmax;      // chunks in the widest output slice
  uint32_t off_q, off_k, off_v, off_m, off_bar;
  uint64_t wait_limit_ns;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[MAX_KST];
  uint64_t k_empty[MAX_KST];
  uint64_t v_full[MAX_VST];
  uint64_t v_empty[MAX_VST];
  uint64_t s_full, s_free;
  uint64_t p_full[2];
  uint64_t o_bar[2];
  uint64_t done;
  uint32_t tmem_slot;
  int abort;
  int slot_item[MAX_KST];  // last Q/K item issued into each ring slot
};

// Ring item i when V travels through the ring: the K pairs of block 0, then
// for each block j the K pairs of block j+1 (while there is one) followed by
// the V items of block j -- the order in which the MMA thread consumes them
// (S_0, then S_{j+1} before P_j V_j).
struct RingItem {
  bool is_v;
  int blk, idx;  // key block; chunk pair (K) or V item
};
__device__ __forceinline__ RingItem vring_item(int i, int np, int nv, int nblk) {
  RingItem r;
  if (i < np) {
    r.is_v = false;
    r.blk = 0;
    r.idx = i;
    return r;
  }
  i -= np;
  const int g = i / (np + nv), m = i % (np + nv);
  if (g < nblk - 1 && m < np) {
    r.is_v = false;
    r.blk = g + 1;
    r.idx = m;
  } else {
    // V items of block g; in the last group (no K after it) only V items exist
    r.is_v = true;
    r.blk = g;
    r.idx = (g < nblk - 1) ? m - np : i - g * (np + nv);
  }
  return r;
}

__device__ __forceinline__ void raise_abort(Bars *bars, int *status) {
  atomicCAS(status, 0, kStatusTimeout);
  *reinterpret_cast<volatile int *>(&bars->abort) = 1;
}

// MASK: an additive mask, staged per block and row (cp.async into shared
// memory, issued before the row's thread waits for the block's scores) and
// added as the scores are scaled.
template <bool MASK>
__global__ void __launch_bounds__(THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const TcParams prm) {
  // tm_q: 128-row boxes of all chunks when Q is resident, else of two chunks;
  // tm_k: 128-row boxes of two chunks; tm_v: 128-row boxes of vmax chunks, or
  // of two chunks when V travels through the ring
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t *sq = smem + prm.off_q;
  uint8_t *sk = smem + prm.off_k;
  uint8_t *sv = smem + prm.off_v;
  uint8_t *smask = smem + prm.off_m;  // [16][128 rows][8 bf16] mask values of one block (MASK)
  Bars *bars = reinterpret_cast<Bars *>(smem + prm.off_bar);
  volatile int *abortf = &bars->abort;

  const Problem &p = prm.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t limit = prm.wait_limit_ns;
  TC_TRACE_SETUP;
  if (tid == 0) TC_TRACE_EV(0, 0);

  // ---- work unit: output slice fastest, then (b, hq), then query tile
  //      (heaviest causal tiles first)
  int bid = blockIdx.x;
  const int nsplit = p.kv_splits;
  const int split = bid % nsplit;
  bid /= nsplit;
  const int slice = bid % prm.nslices;
  bid /= prm.nslices;
  const int BH = p.B * p.Hq;
  const int bh = bid % BH;
  const int t = bid / BH;
  const int tile = p.causal ? (prm.ntiles - 1 - t) : t;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int bkv = b * p.Hkv + hq / (p.Hq / p.Hkv);
  const int q0 = tile * BM;
  const int sbase = prm.nc / prm.nslices, srem = prm.nc % prm.nslices;
  const int s_chunks = sbase + (slice < srem ? 1 : 0);
  const int s_c0 = slice * sbase + (slice < srem ? slice : srem);
  const int DV = s_chunks * 64;
  const int shift = p.Nkv - p.Nq;  // bottom-right causal alignment
  int kv_end = p.Nkv;
  if (p.causal) kv_end = max(0, min(p.Nkv, q0 + BM - 1 + shift + 1));
  // this CTA's key blocks: [jb, jb + nblk) of the tile's range, split evenly;
  // block indices j below are relative to jb
  const int nall = (kv_end + BN - 1) / BN;
  const int jb = (int)((int64_t)split * nall / nsplit);
  const int nblk = (int)((int64_t)(split + 1) * nall / nsplit) - jb;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < prm.kst; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < prm.vst; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 4 * 32);
    mbar_init(&bars->p_full[0], 4 * 32);
    mbar_init(&bars->p_full[1], 4 * 32);
    mbar_init(&bars->o_bar[0], 1);
    mbar_init(&bars->o_bar[1], 1);
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    for (int i = 0; i < MAX_KST; ++i) bars->slot_item[i] = -1;
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

  // Q/K ring items: per block, for each chunk pair c2: [Q pair c2 if Q is
  // streamed], K pair c2.  Item i sits in slot i % kst; producer (i % 2).
  const int items_pb = prm.qres ? prm.npairs : 2 * prm.npairs;  // when V is not in the ring
  if (warp == WARP_LOAD_QK0 || warp == WARP_LOAD_QK1) {
    // ------------------------------------------------------------ Q/K producers
    const int r = (warp == WARP_LOAD_QK0) ? 0 : 1;
    if (lane == 0 && nblk > 0) {
      bool ok = true;
      if (r == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        if (prm.qres) {
          mbar_arrive_expect_tx(&bars->q_full, prm.nc * CHUNK_BYTES);
          tma_load_4d(sq, &tm_q, &bars->q_full, 0, q0, 0, bh);
        }
      }
      const int total = prm.vring ? nblk * (prm.npairs + prm.nvitems) : nblk * items_pb;
      for (int i = r; i < total; i += 2) {
        const int s = i % prm.kst;
        if (!mbar_wait(&bars->k_empty[s], ((i / prm.kst) & 1) ^ 1, abortf, limit)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars->k_full[s], SLOT_BYTES);
        *reinterpret_cast<volatile int *>(&bars->slot_item[s]) = i;
        TC_TRACE_EV(1 + i / 64, i % 64);
        if (prm.vring) {
          const RingItem it = vring_item(i, prm.npairs, prm.nvitems, nblk);
          if (it.is_v)
            tma_load_4d(sk + s * SLOT_BYTES, &tm_v, &bars->k_full[s], 0, (jb + it.blk) * BN, s_c0 + 2 * it.idx, bkv);
          else
            tma_load_4d(sk + s * SLOT_BYTES, &tm_k, &bars->k_full[s], 0, (jb + it.blk) * BN, 2 * it.idx, bkv);
          continue;
        }
        const int j = i / items_pb, m = i % items_pb;
        const bool is_q = !prm.qres && (m & 1) == 0;
        const int c2 = prm.qres ? m : (m >> 1);
        if (is_q)
          tma_load_4d(sk + s * SLOT_BYTES, &tm_q, &bars->k_full[s], 0, q0, 2 * c2, bh);
        else
          tma_load_4d(sk + s * SLOT_BYTES, &tm_k, &bars->k_full[s], 0, (jb + j) * BN, 2 * c2, bkv);
      }
      if (!ok) raise_abort(bars, p.status);
      // drain: copies of this thread that are still the latest in their slot
      // may be in flight; every older one was consumed before its slot refilled
      if (r == 0 && prm.qres) mbar_wait_drain(&bars->q_full, 0, limit);
      for (int s = 0; s < prm.kst; ++s) {
        const int i = *reinterpret_cast<volatile int *>(&bars->slot_item[s]);
        if (i >= 0 && (i & 1) == r) mbar_wait_drain(&bars->k_full[s], (i / prm.kst) & 1, limit);
      }
    }
  } else if (warp == WARP_LOAD_V) {
    // ------------------------------------------------------------ V producer
    if (lane == 0 && nblk > 0 && !prm.vring) {
      tma_prefetch_desc(&tm_v);
      uint32_t vctr = 0;
      bool ok = true;
      for (int j = 0; j < nblk; ++j) {
        const int vs = vctr % prm.vst;
        if (!mbar_wait(&bars->v_empty[vs], ((vctr / prm.vst) & 1) ^ 1, abortf, limit)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars->v_full[vs], prm.vmax * CHUNK_BYTES);
        tma_load_4d(sv + vs * (prm.vmax * CHUNK_BYTES), &tm_v, &bars->v_full[vs], 0, (jb + j) * BN, s_c0, bkv);
        ++vctr;
      }
      if (!ok) raise_abort(bars, p.status);
      const uint32_t vn = vctr < (uint32_t)prm.vst ? vctr : (uint32_t)prm.vst;
      for (uint32_t i = vctr - vn; i < vctr; ++i) mbar_wait_drain(&bars->v_full[i % prm.vst], (i / prm.vst) & 1, limit);
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nblk > 0) {
      const uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      const uint32_t idesc_pv = idesc_bf16(BM, DV, 0, 1);
      // K-major 128B-swizzled chunk descriptors: a K=16 step adds 32 bytes (2 in
      // the >>4 address field), a chunk 16 KB, a ring slot 32 KB
      constexpr uint64_t kChunkD = CHUNK_BYTES >> 4, kSlotD = SLOT_BYTES >> 4;
      const uint64_t qd_res = smem_desc(smem_u32(sq), 16, 1024);
      const uint64_t kd_ring = smem_desc(smem_u32(sk), 16, 1024);
      // V (MN-major): a K=16 step is 16 keys = 2048 bytes; chunks 16 KB apart
      const uint64_t vd_ring = smem_desc(smem_u32(sk), CHUNK_BYTES, 1024);
      const uint64_t vd_sep = smem_desc(smem_u32(sv), CHUNK_BYTES, 1024);
      // ring position of the next Q/K/V item, kept incrementally
      int slot = 0;
      uint32_t phase = 0;
      auto next_item = [&](int &s_out) -> bool {
        s_out = slot;
        const bool r = mbar_wait(&bars->k_full[slot], phase, abortf, limit);
        if (++slot == prm.kst) {
          slot = 0;
          phase ^= 1u;
        }
        return r;
      };
      uint32_t vctr = 0;
      bool ok = true;
      if (prm.qres) ok = mbar_wait(&bars->q_full, 0, abortf, limit);
      auto issue_s = [&]() -> bool {
        for (int c2 = 0; c2 < prm.npairs; ++c2) {
          int qs = -1, ks;
          if (!prm.qres && !next_item(qs)) return false;
          if (!next_item(ks)) return false;
          TC_TRACE_EV(5, c2);
          tc_fence_after();
          const int ncc = min(2, prm.nc - 2 * c2);
          const uint64_t qd = prm.qres ? qd_res + (uint64_t)(2 * c2) * kChunkD : kd_ring + (uint64_t)qs * kSlotD;
          const uint64_t kd = kd_ring + (uint64_t)ks * kSlotD;
          for (int cc = 0; cc < ncc; ++cc) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + TM_S, qd + cc * kChunkD + kk * 2, kd + cc * kChunkD + kk * 2, idesc_s, (c2 | cc | kk) != 0);
          }
          mma_commit(&bars->k_empty[ks]);
          if (qs >= 0) mma_commit(&bars->k_empty[qs]);
        }
        mma_commit(&bars->s_full);
        return true;
      };
      if (ok) ok = issue_s();
      for (int j = 0; j < nblk && ok; ++j) {
        if (j + 1 < nblk) {
          if (!mbar_wait(&bars->s_free, j & 1, abortf, limit)) { ok = false; break; }
          TC_TRACE_EV(8, j);
          tc_fence_after();
          if (!issue_s()) { ok = false; break; }
          TC_TRACE_EV(9, j);
        }
        if (!mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1, abortf, limit)) { ok = false; break; }
        TC_TRACE_EV(10, j);
        const uint32_t pcol = tmem + ((j & 1) ? TM_P1 : TM_P0);
        if (prm.vring) {
          // V_j as ring items of two chunks: O columns [128 v, 128 v + 64 cn)
          for (int v = 0; v < prm.nvitems; ++v) {
            int vs;
            if (!next_item(vs)) { ok = false; break; }
            tc_fence_after();
            const int cn = min(2, s_chunks - 2 * v);
            const uint32_t idesc_v = idesc_bf16(BM, 64 * cn, 0, 1);
            const uint64_t vd = vd_ring + (uint64_t)vs * kSlotD;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ts(tmem + TM_O + 128 * v, pcol + kk * 8, vd + (uint64_t)(kk * (2048 >> 4)), idesc_v,
                     (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bars->k_empty[vs]);
          }
          if (!ok) break;
        } else {
          const int vs = vctr % prm.vst;
          if (!mbar_wait(&bars->v_full[vs], (vctr / prm.vst) & 1, abortf, limit)) { ok = false; break; }
          tc_fence_after();
          const uint64_t vd = vd_sep + (uint64_t)vs * (uint64_t)(prm.vmax * kChunkD);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + TM_O, pcol + kk * 8, vd + (uint64_t)(kk * (2048 >> 4)), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars->v_empty[vs]);
          ++vctr;
        }
        mma_commit(&bars->o_bar[j & 1]);
        TC_TRACE_EV(11, j);
      }
      if (!ok) raise_abort(bars, p.status);
      // every MMA this thread issued completes before TMEM is released
      mma_commit(&bars->done);
      if (!mbar_wait_drain(&bars->done, 0, limit)) raise_abort(bars, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int row = tid;  // 0..127
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int qi = q0 + row;
    const int vis_end = p.causal ? min(p.Nkv, qi + shift + 1) : p.Nkv;  // keys [0, vis_end) are visible
    const float sl2 = p.scale * kLog2e;
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    const __nv_bfloat16 *mrow = MASK ? mask_row(p, b, hq, qi) : nullptr;

    for (int j = 0; j < nblk; ++j) {
      // this row's mask values of the block travel while the scores are computed
      if constexpr (MASK) mask_stage128(smem_u32(smask), BM, row, mrow, (jb + j) * BN, p.Nkv, p.mask);
      // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full, j & 1, abortf, limit))) { ok = false; break; }
      if (tid == 0) TC_TRACE_EV(12, j);
      tc_fence_after();
      uint32_t sr[BN / 32][32];
#pragma unroll
      for (int cc = 0; cc < BN / 32; ++cc) tmem_ld32(tmem + lane_base + TM_S + cc * 32, sr[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < BN / 32; ++cc) reg_fence32(sr[cc]);
      float x[BN];
#pragma unroll
      for (int cc = 0; cc < BN / 32; ++cc)
#pragma unroll
        for (int i = 0; i < 32; ++i) x[cc * 32 + i] = __uint_as_float(sr[cc][i]);
      tc_fence_before();
      mbar_arrive(&bars->s_free);

      // scale to log2 units, mask, block max
      const int kbase = (jb + j) * BN;
      float mblk = -INFINITY;
      if constexpr (MASK) {
        // y = s * sl2 + mask * log2 e, -inf past vis_end (the thread's own
        // copies have landed once its cp.async groups are complete)
        cp_async_wait_all();
        const uint4 *ms = reinterpret_cast<const uint4 *>(smask + row * 16);
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8) {
          const uint4 w = ms[c8 * BM];
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int t4 = 0; t4 < 4; ++t4) {
            const int c = 8 * c8 + 2 * t4;
            x[c] = (kbase + c < vis_end) ? fmaf(x[c], sl2, kLog2e * bf16_lo(wv[t4])) : -INFINITY;
            x[c + 1] = (kbase + c + 1 < vis_end) ? fmaf(x[c + 1], sl2, kLog2e * bf16_hi(wv[t4])) : -INFINITY;
            mblk = max3f(mblk, x[c], x[c + 1]);
          }
        }
      } else if (kbase + BN <= vis_end) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          x[c] *= sl2;
          mblk = fmaxf(mblk, x[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          x[c] = (kbase + c < vis_end) ? x[c] * sl2 : -INFINITY;
          mblk = fmaxf(mblk, x[c]);
        }
      }
      const float m_new = fmaxf(m_use, mblk);
      const bool need = m_new > m_use + TAU;
      if (__any_sync(0xffffffffu, need)) {
        // the whole warp moves to its new maxima (exact for any choice)
        const float alpha = (m_use == -INFINITY) ? 0.f : ex2_approx(m_use - m_new);
        if (j > 0) {
          const int pj = j - 1;
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_bar[pj & 1], (pj >> 1) & 1, abortf, limit))) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int cc = 0; cc < DV / 32; ++cc) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + TM_O + cc * 32, r);
            tmem_wait_ld();
            reg_fence32(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tmem + lane_base + TM_O + cc * 32, r);
          }
          tmem_wait_st();
        }
        l *= alpha;
        m_use = m_new;
      }
      const float mu = (m_use == -INFINITY) ? 0.f : m_use;
      const uint32_t pcol = (j & 1) ? TM_P1 : TM_P0;
      float lsum = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ex2_approx(x[h * 64 + 2 * i] - mu);
          const float p1 = ex2_approx(x[h * 64 + 2 * i + 1] - mu);
          lsum += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tmem + lane_base + pcol + h * 32, pk);
      }
      l += lsum;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[j & 1]);
      if (tid == 0) TC_TRACE_EV(13, j);
    }

    if (!ok) raise_abort(bars, p.status);
    // ---- epilogue: O / l -> bf16, LSE
    __nv_bfloat16 *orow = p.o + ((int64_t)bh * p.Nq + qi) * p.D + s_c0 * 64;
    if (ok && nblk > 0) {
      const int last = nblk - 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_bar[last & 1], (last >> 1) & 1, abortf, limit))) {
        raise_abort(bars, p.status);
        ok = false;
      }
    }
    if (ok) {
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const float lse_val = (m_use == -INFINITY || !(l > 0.f)) ? -INFINITY : (m_use + log2f(l)) * kLn2;
      const int64_t row_idx = (int64_t)bh * p.Nq + qi;
      // split-KV: normalised fp32 partial O_s and LSE_s of this key range
      float *wrow = (nsplit > 1) ? p.ws_o + ((int64_t)split * BH * p.Nq + row_idx) * p.D + s_c0 * 64 : nullptr;
      for (int cc = 0; cc < DV / 32; ++cc) {
        uint32_t r[32];
        if (nblk > 0) {
          tmem_ld32(tmem + lane_base + TM_O + cc * 32, r);
          tmem_wait_ld();
          reg_fence32(r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (qi < p.Nq) {
          if (nsplit == 1) {
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
          } else {
            float4 *dst = reinterpret_cast<float4 *>(wrow + cc * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(__uint_as_float(r[v4 * 4 + 0]) * inv, __uint_as_float(r[v4 * 4 + 1]) * inv,
                                    __uint_as_float(r[v4 * 4 + 2]) * inv, __uint_as_float(r[v4 * 4 + 3]) * inv);
          }
        }
      }
      if (slice == 0 && qi < p.Nq) {
        if (nsplit == 1)
          p.lse[row_idx] = lse_val;
        else
          p.ws_lse[(int64_t)split * BH * p.Nq + row_idx] = lse_val;
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (tid == 0) TC_TRACE_EV(14, 0);
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

constexpr int kSmemMax = 232448;  // opt-in dynamic shared memory per block on sm_100-family
constexpr int kSmemReserve = 2048;
constexpr int kMaxDevicesTc = 64;

}  // namespace

TcConfig tc_config(int D, bool mask) {
  TcConfig c;
  c.nc = D / 64;
  c.nslices = (D + 255) / 256;
  c.vmax = (c.nc + c.nslices - 1) / c.nslices;
  c.mask_bytes = mask ? BM * 256 : 0;  // one block's mask values for the 128 rows
  const int avail = kSmemMax - kSmemReserve - c.mask_bytes;
  const int qb = c.nc * CHUNK_BYTES, vb = c.vmax * CHUNK_BYTES;
  // Q resident when it leaves room for at least three Q/K slots and one V
  // slot (two V slots if three Q/K slots still fit); else Q streams through
  // the ring next to K, with two V slots when four ring slots remain
  c.qres = 0;
  c.vring = 0;
  c.vst = 1;
  if (qb + vb + 3 * SLOT_BYTES <= avail) {
    c.qres = 1;
    c.vst = (qb + 2 * vb + 3 * SLOT_BYTES <= avail) ? 2 : 1;
    c.kst = (avail - qb - c.vst * vb) / SLOT_BYTES;
  } else if (qb + 3 * SLOT_BYTES <= avail) {
    // Q stays resident; V blocks take ring slots between the K pairs
    c.qres = 1;
    c.vring = 1;
    c.vst = 0;
    c.kst = (avail - qb) / SLOT_BYTES;
  } else {
    c.vst = (2 * vb + 4 * SLOT_BYTES <= avail) ? 2 : 1;
    c.kst = (avail - c.vst * vb) / SLOT_BYTES;
  }
  if (c.kst > MAX_KST) c.kst = MAX_KST;
  c.off_q = 0;
  c.off_k = c.qres ? qb : 0;
  c.off_v = c.off_k + c.kst * SLOT_BYTES;
  c.off_m = c.off_v + c.vst * vb;
  c.off_bar = c.off_m + c.mask_bytes;
  c.smem_bytes = c.off_bar + (int)sizeof(Bars) + 1024;  // + alignment slack
  return c;
}

cudaError_t launch_tc(const Problem &p, int device, uint64_t wait_limit_ns, cudaStream_t stream) {
  static_assert(sizeof(Bars) <= kSmemReserve - 1024, "barrier block too large");
  const TcConfig c = tc_config(p.D, p.mask != nullptr);
  if (c.kst < 2 || c.smem_bytes > kSmemMax) return cudaErrorInvalidConfiguration;
  CUtensorMap tq, tk, tv;
  if (!make_chunk_map(&tq, p.q, p.D, p.Nq, p.B * p.Hq, BM, c.qres ? c.nc : 2)) return cudaErrorInvalidValue;
  if (!make_chunk_map(&tk, p.k, p.D, p.Nkv, p.B * p.Hkv, BN, 2)) return cudaErrorInvalidValue;
  if (!make_chunk_map(&tv, p.v, p.D, p.Nkv, p.B * p.Hkv, BN, c.vring ? 2 : c.vmax)) return cudaErrorInvalidValue;
  TcParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.p = p;
  prm.nc = c.nc;
  prm.nslices = c.nslices;
  prm.ntiles = (p.Nq + BM - 1) / BM;
  prm.kst = c.kst;
  prm.vst = c.vst;
  prm.qres = c.qres;
  prm.vring = c.vring;
  prm.nvitems = (c.vmax + 1) / 2;
  prm.vmax = c.vmax;
  prm.npairs = (c.nc + 1) / 2;
  prm.off_q = c.off_q;
  prm.off_k = c.off_k;
  prm.off_v = c.off_v;
  prm.off_m = c.off_m;
  prm.off_bar = c.off_bar;
  prm.wait_limit_ns = wait_limit_ns;
  const int64_t grid = (int64_t)prm.ntiles * p.B * p.Hq * c.nslices * p.kv_splits;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // the opt-in shared-memory limit is a per-device function attribute: raise
  // it to the maximum once per device and variant
  static std::atomic<int> attr_set[2][kMaxDevicesTc];
  if (device < 0 || device >= kMaxDevicesTc) return cudaErrorInvalidDevice;
  const int mk = p.mask ? 1 : 0;
  if (!attr_set[mk][device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(mk ? attn_tc_kernel<true> : attn_tc_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    attr_set[mk][device].store(1, std::memory_order_release);
  }
  if (mk)
    attn_tc_kernel<true><<<(unsigned)grid, THREADS, c.smem_bytes, stream>>>(tq, tk, tv, prm);
  else
    attn_tc_kernel<false><<<(unsigned)grid, THREADS, c.smem_bytes, stream>>>(tq, tk, tv, prm);
  return cudaGetLastError();
}

}  // namespace attn
