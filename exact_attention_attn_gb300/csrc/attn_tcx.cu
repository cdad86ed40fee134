// Exact attention forward for head dims 384 ... 1024 (multiples of 64):
// Split-D across a thread-block cluster, the scores computed once.
//
// The FFPA page's Split-D cuts the D axis into chunks so that on-chip memory
// does not grow with D.  On sm_103a the output accumulator of a 128-row tile
// lives in TMEM, which holds at most 256 fp32 output columns next to S and P,
// so a tile's output is cut into NX slices of at most 256 columns (NX = 2 up
// to D = 512, 4 above; slices of equal width where D/64 divides by NX, else
// widths differing by one 64-column chunk).  Here the NX slices of a tile are
// the NX CTAs of one cluster, and the contraction of S = Q K^T is cut the
// same way: CTA r keeps Q[:, Wr, Wr + W) in shared memory, streams the
// matching columns of K and V, and computes the partial scores
// S_r = Q_r K_r^T on its tensor cores.  The partials are summed across the
// cluster through distributed shared memory: CTA r owns rows
// [rR, rR + R) (R = 128 / NX) of the tile, receives the other CTAs' partial
// rows for them, and runs the online softmax of the "FlashAttention v1/v2/v3/v4"
// page ("El truco que hizo posible todo: online softmax", with the
// conditional rescaling of its FA4 section) on the full scores of its rows.
// P (bf16) and the rescale factors of its rows go back to every CTA, and each
// CTA accumulates O_r += P V_r for its own output slice.  So the
// tensor cores do the useful work once (no CTA recomputes S), at the price of
// moving (NX - 1) R rows of fp32 partial scores and bf16 P per key block
// through the cluster.
//
// CTA = 8 warps:
//   warps 0-3  exchange + softmax + epilogue, one tile row per thread (warp w
//              touches TMEM lanes 32w..32w+31); a warp whose rows this CTA
//              owns runs the softmax and stages its P rows in shared memory;
//              each other warp sends its partial rows to their owner,
//              forwards this CTA's staged P rows to that same CTA, and takes
//              P and the rescale factors of its own rows back
//   warps 4, 6 TMA producers of the ring (one thread each, alternate items)
//   warp 5     TMEM allocator and MMA issuer (one thread)
//   warp 7     idle
//
// Shared memory: Q_r resident (W x 128 bf16 for a slice of W columns); a ring
// of items of two 64-column chunks (W = 256), three (W = 192) or one (uneven
// slices), in the order K_0, K_1, then per block j: K_{j+2}, V_j; xin, the
// partial rows sent to this CTA (NX - 1 slots of R rows x 128 fp32); pin, the
// P rows sent to this CTA ((128 - R) rows x 128 bf16) and their rescale
// factors; the staged P rows and factors of this CTA's own rows; at the end
// the final l and m of every row, in the Q region.
//
// TMEM columns: S [0,128) fp32 partial scores; P0 [128,192) and P1 [192,256)
// bf16 pairs (double-buffered); O [256, 512) fp32 output slice.
//
// Every wait is bounded; a CTA that gives up raises the abort flag of every
// CTA of its cluster, and all of them meet at a final cluster barrier before
// any exits, so that no CTA writes into the shared memory of one that left.
#include <math.h>
#include <string.h>

#include <atomic>

#include <cuda.h>

#include "attn_internal.h"
#include "attn_mask.cuh"
#include "sm100_ptx.cuh"

// Optional per-role timestamps (clock64) of the first cluster, compiled in only
// when ATTN_TRACE is defined: TCX_EV(row, col) stores into
// attn_tcx_trace_buf[cta][16][64].
#ifdef ATTN_TRACE
__device__ long long *attn_tcx_trace_buf;
#define TCX_EV(row, col)                                                                                \
  do {                                                                                                  \
    if (attn_tcx_trace_buf && blockIdx.x < 4 && (col) < 64)                                              \
      attn_tcx_trace_buf[((long long)blockIdx.x * 16 + (row)) * 64 + (col)] = clock64();                 \
  } while (0)
#else
#define TCX_EV(row, col) \
  do {                   \
  } while (0)
#endif

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128, BN = 128;
constexpr int CHUNK_BYTES = 128 * 128;   // one 128-row x 64-column bf16 chunk
constexpr int THREADS = 256;
constexpr int WARP_LOAD0 = 4, WARP_MMA = 5, WARP_LOAD1 = 6;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_P0 = 128, TM_P1 = 192, TM_O = 256;
constexpr float TAU = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int MAX_KST = 8;
constexpr int kSmemMax = 232448;

struct XParams {
  Problem p;
  int ntiles;
  int kst;
  uint32_t off_k, off_x, off_p, off_a, off_s, off_sa, off_m, off_bar;
  uint64_t wait_limit_ns;
};

struct XBars {
  uint64_t q_full;
  uint64_t k_full[MAX_KST];
  uint64_t k_empty[MAX_KST];
  uint64_t s_full, s_free;
  uint64_t p_full[2];
  uint64_t o_bar[2];
  // the *_full barriers count the bytes of the other CTAs' asynchronous
  // stores; one thread of this CTA arrives with the expected byte count
  uint64_t xin_full[3];  // partial rows of the other CTA in slot s have landed here
  uint64_t xin_free;  // every owner has taken this CTA's partial rows
  uint64_t pin_full;  // P rows and rescale factors of every other owner have landed here
  uint64_t pin_free;  // every other CTA has taken this CTA's P rows
  uint64_t stg_full;  // the owner warps have staged this block's P rows (local)
  uint64_t stg_free;  // the other warps have forwarded the staged rows (local)
  uint64_t fin_full;  // final l and m of every other owner's rows have landed here
  uint64_t done;
  uint32_t tmem_slot;
  int abort;
  int slot_item[MAX_KST];
};

// Ring item i, in the order the MMA thread consumes them: K_0 and K_1 (NI
// items each), then for each block g the items of K_{g+2} (while there is
// one) and those of V_g -- S runs two blocks ahead of P V.
struct XItem {
  bool is_v;
  int blk, idx;
};
__device__ __forceinline__ XItem ring_item(int i, int nblk, int NI /* items per K or V block */) {
  XItem r;
  const int head = (nblk > 1 ? 2 : 1) * NI;
  if (i < head) {
    r.is_v = false;
    r.blk = i / NI;
    r.idx = i % NI;
    return r;
  }
  i -= head;
  const int g4 = nblk > 2 ? nblk - 2 : 0;  // groups with a K block
  if (i < 2 * NI * g4) {
    const int g = i / (2 * NI), m = i % (2 * NI);
    r.is_v = m >= NI;
    r.blk = r.is_v ? g : g + 2;
    r.idx = m % NI;
  } else {
    i -= 2 * NI * g4;
    r.is_v = true;
    r.blk = g4 + i / NI;
    r.idx = i % NI;
  }
  return r;
}

template <int NX>
__device__ __forceinline__ void raise_abort_cluster(XBars *bars, int *status, uint32_t me) {
  atomicCAS(status, 0, kStatusTimeout);
  *reinterpret_cast<volatile int *>(&bars->abort) = 1;
  const uint32_t a = smem_u32(&bars->abort);
#pragma unroll
  for (int q = 0; q < NX; ++q)
    if ((uint32_t)q != me) st_cluster_u32(mapa_shared(a, (uint32_t)q), 1u);
}

// NX CTAs per cluster, each with a slice of SC 64-column chunks (D = 64 NX SC),
// K and V travelling through the ring as items of IC chunks -- or, UN, slices
// of SC or SC - 1 chunks (D = 64 nc with nc not a multiple of NX) whose K and
// V travel as one-chunk items.  MASK: an additive mask, staged per block for
// the owner rows (cp.async into shared memory, issued before the owner
// waits for the block's scores) and added as the scores are scaled.
template <int NX, int SC, bool UN, bool MASK>
__global__ void __launch_bounds__(THREADS, 1)
    attn_tcx_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ XParams prm) {
  constexpr int IC = UN ? 1 : SC % 2 == 0 ? 2 : SC;  // chunks per ring item
  constexpr int ITEM_BYTES = IC * CHUNK_BYTES;
  constexpr int R = BM / NX;           // rows owned by each CTA
  constexpr int OWN_WARPS = R / 32;    // warps holding them
  constexpr int NOTHER = BM - R;       // rows owned by the other CTAs
  constexpr int XSLOT = R * 512;       // bytes of one sender's partial rows
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t *sq = smem;
  uint8_t *sk = smem + prm.off_k;
  uint8_t *sx = smem + prm.off_x;
  uint8_t *sp = smem + prm.off_p;
  float *salpha = reinterpret_cast<float *>(smem + prm.off_a);  // [128], by tile row
  uint8_t *sst = smem + prm.off_s;                               // staged own P rows
  uint8_t *smask = smem + prm.off_m;                             // owner rows' mask values (MASK)
  float *sstal = reinterpret_cast<float *>(smem + prm.off_sa);    // staged own rescale factors
  // l[128], m[128] of every row at the end, in the Q region: every CTA's last
  // Q K^T has completed before any owner sends them (it needed their partials)
  float *sfin = reinterpret_cast<float *>(smem);
  XBars *bars = reinterpret_cast<XBars *>(smem + prm.off_bar);
  volatile int *abortf = &bars->abort;

  const Problem &p = prm.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t limit = prm.wait_limit_ns;
  const uint32_t me = cluster_ctarank();

  // ---- work unit (one per cluster): query tile fastest, then (b, hq); the
  //      CTA's rank is its D slice
  int cid = (int)(blockIdx.x / NX);
  const int nsplit = p.kv_splits;
  const int split = cid % nsplit;
  cid /= nsplit;
  const int BH = p.B * p.Hq;
  // the tiles of one head one after the other (heaviest causal tiles first),
  // so that a wave of clusters streams the K/V of few heads and each block
  // comes from L2 to every tile of its head: on B1 H8 N4096 D512 the DRAM
  // reads fall from 2.1x to 1.0x the algorithmic bytes (head-fastest order)
  const int bh = cid / prm.ntiles;
  const int tt = cid % prm.ntiles;
  const int tile = p.causal ? (prm.ntiles - 1 - tt) : tt;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int bkv = b * p.Hkv + hq / (p.Hq / p.Hkv);
  const int q0 = tile * BM;
  const int nc = p.D / 64;
  const int sc = UN ? nc / NX + ((int)me < nc % NX ? 1 : 0) : SC;  // chunks of this CTA's slice
  const int c0 = UN ? (int)me * (nc / NX) + min((int)me, nc % NX) : SC * (int)me;  // its first chunk
  const int NI = sc / IC;      // ring items per K or V block
  const int OCOLS = sc * 64;   // output columns of the slice
  const int shift = p.Nkv - p.Nq;
  int kv_end = p.Nkv;
  if (p.causal) kv_end = max(0, min(p.Nkv, q0 + BM - 1 + shift + 1));
  const int nall = (kv_end + BN - 1) / BN;
  const int jb = (int)((int64_t)split * nall / nsplit);
  const int nblk = (int)((int64_t)(split + 1) * nall / nsplit) - jb;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < prm.kst; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 128);
    mbar_init(&bars->p_full[0], 128);
    mbar_init(&bars->p_full[1], 128);
    mbar_init(&bars->o_bar[0], 1);
    mbar_init(&bars->o_bar[1], 1);
    for (int sl = 0; sl < NX - 1; ++sl) mbar_init(&bars->xin_full[sl], 1);
    mbar_init(&bars->xin_free, (NX - 1) * OWN_WARPS);
    mbar_init(&bars->pin_full, 1);
    mbar_init(&bars->pin_free, (NX - 1) * OWN_WARPS);
    mbar_init(&bars->stg_full, R);
    mbar_init(&bars->stg_free, 4 - OWN_WARPS);
    mbar_init(&bars->fin_full, 1);
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
  // every CTA's barriers exist before any CTA of the cluster touches them
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  if (warp == WARP_LOAD0 || warp == WARP_LOAD1) {
    // ------------------------------------------------------------ producers
    const int r = (warp == WARP_LOAD0) ? 0 : 1;
    if (lane == 0 && nblk > 0) {
      bool ok = true;
      if (r == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(&bars->q_full, sc * CHUNK_BYTES);
        if constexpr (UN) {
          for (int c = 0; c < sc; ++c) tma_load_4d(sq + c * CHUNK_BYTES, &tm_q, &bars->q_full, 0, q0, c0 + c, bh);
        } else {
          tma_load_4d(sq, &tm_q, &bars->q_full, 0, q0, c0, bh);
        }
      }
      const int total = 2 * NI * nblk;
      for (int i = r; i < total; i += 2) {
        const int s = i % prm.kst;
        if (!mbar_wait(&bars->k_empty[s], ((i / prm.kst) & 1) ^ 1, abortf, limit)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars->k_full[s], ITEM_BYTES);
        *reinterpret_cast<volatile int *>(&bars->slot_item[s]) = i;
        const XItem it = ring_item(i, nblk, NI);
        tma_load_4d(sk + s * ITEM_BYTES, it.is_v ? &tm_v : &tm_k, &bars->k_full[s], 0, (jb + it.blk) * BN,
                    c0 + IC * it.idx, bkv);
      }
      if (!ok) raise_abort_cluster<NX>(bars, p.status, me);
      // drain: copies of this thread that are still the latest in their slot
      // may be in flight; every older one was consumed before its slot refilled
      if (r == 0) mbar_wait_drain(&bars->q_full, 0, limit);
      for (int s = 0; s < prm.kst; ++s) {
        const int i = *reinterpret_cast<volatile int *>(&bars->slot_item[s]);
        if (i >= 0 && (i & 1) == r) mbar_wait_drain(&bars->k_full[s], (i / prm.kst) & 1, limit);
      }
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nblk > 0) {
      const uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      const uint32_t idesc_v = idesc_bf16(BM, IC * 64, 0, 1);
      constexpr uint64_t kChunkD = CHUNK_BYTES >> 4, kItemD = ITEM_BYTES >> 4;
      const uint64_t qd = smem_desc(smem_u32(sq), 16, 1024);
      const uint64_t kd_ring = smem_desc(smem_u32(sk), 16, 1024);
      const uint64_t vd_ring = smem_desc(smem_u32(sk), CHUNK_BYTES, 1024);
      int slot = 0;
      uint32_t phase = 0;
      auto next_item = [&](int &s_out) -> bool {
        s_out = slot;
        const bool got = mbar_wait(&bars->k_full[slot], phase, abortf, limit);
        if (++slot == prm.kst) {
          slot = 0;
          phase ^= 1u;
        }
        return got;
      };
      bool ok = mbar_wait(&bars->q_full, 0, abortf, limit);
      int nissued = 0;
      (void)nissued;
      // S_r = Q_r K_r^T over this CTA's 256 columns: two items of two chunks
      auto issue_s = [&]() -> bool {
        for (int it = 0; it < NI; ++it) {
          int ks;
          if (!next_item(ks)) return false;
          tc_fence_after();
          const uint64_t kd = kd_ring + (uint64_t)ks * kItemD;
#pragma unroll
          for (int cc = 0; cc < IC; ++cc)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + TM_S, qd + (uint64_t)((IC * it + cc) * kChunkD + kk * 2),
                     kd + (uint64_t)(cc * kChunkD + kk * 2), idesc_s, (it | cc | kk) != 0);
          mma_commit(&bars->k_empty[ks]);
        }
        mma_commit(&bars->s_full);
        TCX_EV(6, nissued);
        ++nissued;
        return true;
      };
      // S_0, S_1, then per block j: S_{j+2} (once every thread has read S_{j+1})
      // and P_j V_j -- so that a late P_j holds back no scores
      if (ok) ok = issue_s();
      if (ok && nblk > 1) {
        ok = mbar_wait(&bars->s_free, 0, abortf, limit);
        if (ok) {
          tc_fence_after();
          ok = issue_s();
        }
      }
      for (int j = 0; j < nblk && ok; ++j) {
        if (j + 2 < nblk) {
          if (!mbar_wait(&bars->s_free, (j + 1) & 1, abortf, limit)) { ok = false; break; }
          tc_fence_after();
          if (!issue_s()) { ok = false; break; }
        }
        if (!mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1, abortf, limit)) { ok = false; break; }
        TCX_EV(8, j);
        const uint32_t pcol = tmem + ((j & 1) ? TM_P1 : TM_P0);
        // O_r += P V_r: NI items of IC * 64 output columns
        for (int v = 0; v < NI && ok; ++v) {
          int vs;
          if (!next_item(vs)) { ok = false; break; }
          tc_fence_after();
          const uint64_t vd = vd_ring + (uint64_t)vs * kItemD;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + TM_O + IC * 64 * v, pcol + kk * 8, vd + (uint64_t)(kk * (2048 >> 4)), idesc_v,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars->k_empty[vs]);
        }
        if (!ok) break;
        mma_commit(&bars->o_bar[j & 1]);
        TCX_EV(7, j);
      }
      if (!ok) raise_abort_cluster<NX>(bars, p.status, me);
      mma_commit(&bars->done);
      if (!mbar_wait_drain(&bars->done, 0, limit)) raise_abort_cluster<NX>(bars, p.status, me);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ exchange / softmax / epilogue
    const int row = tid;                       // tile row = TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int owner = warp / OWN_WARPS;        // CTA that owns this warp's rows
    const bool is_owner = owner == (int)me;
    const int orow = row - owner * R;          // row index within its owner's R rows
    const int qi = q0 + row;
    const int vis_end = p.causal ? min(p.Nkv, qi + shift + 1) : p.Nkv;
    const float sl2 = p.scale * kLog2e;
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    // this CTA's slot among the senders into `owner`, and `owner`'s slot among
    // the P senders into this CTA
    const int xslot_out = (int)me < owner ? (int)me : (int)me - 1;
    // the sender warp that announces the P bytes expected per block, and the count
    const int first_sender = me == 0 ? OWN_WARPS : 0;
    constexpr uint32_t PBYTES = (uint32_t)NOTHER * (256 + 4);
    const int pslot_in = owner < (int)me ? owner : owner - 1;
    const uint32_t sx_u = smem_u32(sx), sp_u = smem_u32(sp), sa_u = smem_u32(salpha), sf_u = smem_u32(sfin);

    // A sender warp forwards this CTA's staged P rows of block jj (one row per
    // lane, with its rescale factor) to the CTA that owns the warp's own rows:
    // at D=1024 each of the three sender warps serves one other CTA, at D=512
    // the two serve halves of the rows.  The owner warps only stage them.
    auto forward_p = [&](int jj) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->stg_full, jj & 1, abortf, limit))) return false;
      if (jj > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->pin_free, (jj - 1) & 1, abortf, limit))) return false;
      const int fr = (warp % OWN_WARPS) * 32 + lane;  // row among this CTA's owned rows
      const int ps = (int)me < owner ? (int)me : (int)me - 1;  // this CTA's slot among the target's P senders
      const uint32_t dst = mapa_shared(sp_u, (uint32_t)owner) + (uint32_t)((ps * R + fr) * 16);
      const uint32_t rbar = mapa_shared(smem_u32(&bars->pin_full), (uint32_t)owner);
      const uint4 *src = reinterpret_cast<const uint4 *>(sst + fr * 16);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 w4 = src[c * R];
        st_async_v4(dst + (uint32_t)(c * NOTHER * 16), w4.x, w4.y, w4.z, w4.w, rbar);
      }
      st_async_u32(mapa_shared(sa_u + (uint32_t)((int)me * R + fr) * 4u, (uint32_t)owner), __float_as_uint(sstal[fr]),
                   rbar);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->stg_free);
      return true;
    };

    // a sender warp takes P of block jj from its owner: the rescale factor
    // (applied to its O rows once P_{jj-1} V has completed) and the P rows,
    // into TMEM P buffer jj % 2 once P_{jj-2} V has read it
    auto take_p = [&](int jj) -> bool {
      if (lane == 0 && warp == first_sender) mbar_arrive_expect_tx(&bars->pin_full, PBYTES);
      if (!__all_sync(0xffffffffu, mbar_wait_cluster(&bars->pin_full, jj & 1, abortf, limit))) return false;
      const float alpha = salpha[row];
      if (__any_sync(0xffffffffu, alpha != 1.f) && jj > 0) {
        const int pj = jj - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_bar[pj & 1], (pj >> 1) & 1, abortf, limit))) return false;
        tc_fence_after();
        for (int cc = 0; cc < OCOLS / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + TM_O + cc * 32, r);
          tmem_wait_ld();
          reg_fence32(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tmem + lane_base + TM_O + cc * 32, r);
        }
      }
      const uint32_t pc = (jj & 1) ? TM_P1 : TM_P0;
      if (jj >= 2) {  // P buffer jj % 2 was read by P_{jj-2} V
        const int pj = jj - 2;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_bar[pj & 1], (pj >> 1) & 1, abortf, limit))) return false;
        tc_fence_after();
      }
      const uint4 *src = reinterpret_cast<const uint4 *>(sp + (pslot_in * R + orow) * 16);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w4 = src[(h * 8 + c) * NOTHER];
          pk[4 * c + 0] = w4.x;
          pk[4 * c + 1] = w4.y;
          pk[4 * c + 2] = w4.z;
          pk[4 * c + 3] = w4.w;
        }
        tmem_st32(tmem + lane_base + pc + h * 32, pk);
      }
      __syncwarp();
      if (lane == 0 && jj + 1 < nblk)  // P_{jj+1} may be written here
        mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&bars->pin_free), (uint32_t)owner));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[jj & 1]);
      if (lane == 0 && (warp & (OWN_WARPS - 1)) == 0) TCX_EV(5, jj);
      return true;
    };

    const __nv_bfloat16 *mrow = MASK ? mask_row(p, b, hq, qi) : nullptr;
    for (int j = 0; j < nblk && ok; ++j) {
      // an owner's mask values of this block travel while it waits for the scores
      if (MASK && is_owner) mask_stage128(smem_u32(smask), R, orow, mrow, (jb + j) * BN, p.Nkv, p.mask);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full, j & 1, abortf, limit))) { ok = false; break; }
      tc_fence_after();
      const uint32_t pcol = (j & 1) ? TM_P1 : TM_P0;

      if (!is_owner) {
        uint32_t sr[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tmem + lane_base + TM_S + cc * 32, sr[cc]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) reg_fence32(sr[cc]);
        tc_fence_before();
        mbar_arrive(&bars->s_free);  // S may be overwritten by the next block's partial
        if (lane == 0 && (warp & (OWN_WARPS - 1)) == 0) TCX_EV(3, j);
        // -------- sender: partial rows to their owner; the P of the block
        // before is taken afterwards, so that this block's rows are already on
        // their way while the owner works on the previous one
        if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->xin_free, (j - 1) & 1, abortf, limit))) {
          ok = false;
          break;
        }
        const uint32_t dst = mapa_shared(sx_u, (uint32_t)owner) + (uint32_t)(xslot_out * XSLOT + orow * 16);
        const uint32_t rbar = mapa_shared(smem_u32(&bars->xin_full[xslot_out]), (uint32_t)owner);
#pragma unroll
        for (int c4 = 0; c4 < 32; ++c4)
          st_async_v4(dst + (uint32_t)(c4 * R * 16), sr[c4 >> 3][(c4 & 7) * 4 + 0], sr[c4 >> 3][(c4 & 7) * 4 + 1],
                      sr[c4 >> 3][(c4 & 7) * 4 + 2], sr[c4 >> 3][(c4 & 7) * 4 + 3], rbar);
        if (lane == 0 && (warp & (OWN_WARPS - 1)) == 0) TCX_EV(4, j);
        if (j > 0 && !(forward_p(j - 1) && take_p(j - 1))) {
          ok = false;
          break;
        }
        if (j + 1 == nblk && !(forward_p(j) && take_p(j))) {
          ok = false;
          break;
        }
        continue;
      }

      // -------- owner: full scores of its rows, online softmax, P to everyone
      // this CTA's own partial first, a quarter at a time, so that S may be
      // overwritten by the next block's while the other CTAs' partials travel
      float x[BN];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + TM_S + cc * 32, r);
        tmem_wait_ld();
        reg_fence32(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[cc * 32 + i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      mbar_arrive(&bars->s_free);
      if (lane == 0 && (warp & (OWN_WARPS - 1)) == 0) TCX_EV(0, j);
      if (lane == 0 && warp % OWN_WARPS == 0)
        for (int sl = 0; sl < NX - 1; ++sl) mbar_arrive_expect_tx(&bars->xin_full[sl], XSLOT);
      {
        // plus the other CTAs' partials in rank order, each as soon as it has
        // landed (the order of the additions stays fixed)
        const float4 *slots = reinterpret_cast<const float4 *>(sx + orow * 16);
#pragma unroll
        for (int sl = 0; sl < NX - 1; ++sl) {
          if (!__all_sync(0xffffffffu, mbar_wait_cluster(&bars->xin_full[sl], j & 1, abortf, limit))) {
            ok = false;
            break;
          }
          if (sl == 0 && lane == 0 && (warp & (OWN_WARPS - 1)) == 0) TCX_EV(1, j);
#pragma unroll
          for (int c4 = 0; c4 < 32; ++c4) {
            const float4 v = slots[sl * (XSLOT / 16) + c4 * R];
            x[4 * c4 + 0] += v.x;
            x[4 * c4 + 1] += v.y;
            x[4 * c4 + 2] += v.z;
            x[4 * c4 + 3] += v.w;
          }
        }
      }
      if (!ok) break;
      if (lane == 0 && (warp & (OWN_WARPS - 1)) == 0) TCX_EV(9, j);
      __syncwarp();
      if (lane == 0 && j + 1 < nblk) {
        // the partial slots may be refilled (every lane's reads of them have
        // returned: their values are in the sums above)
#pragma unroll
        for (int q = 0; q < NX; ++q)
          if (q != (int)me) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&bars->xin_free), (uint32_t)q));
      }
      // scale to log2 units, mask, block max
      const int kbase = (jb + j) * BN;
      if constexpr (MASK) {
        // y = s * sl2 + mask * log2 e, -inf past vis_end; this thread's own
        // copies have landed once its cp.async groups are complete
        cp_async_wait_all();
        const uint4 *ms = reinterpret_cast<const uint4 *>(smask + orow * 16);
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8) {
          const uint4 w = ms[c8 * R];
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int c = 8 * c8 + 2 * t;
            x[c] = (kbase + c < vis_end) ? fmaf(x[c], sl2, kLog2e * bf16_lo(wv[t])) : -INFINITY;
            x[c + 1] = (kbase + c + 1 < vis_end) ? fmaf(x[c + 1], sl2, kLog2e * bf16_hi(wv[t])) : -INFINITY;
          }
        }
      } else if (kbase + BN <= vis_end) {
#pragma unroll
        for (int c = 0; c < BN; ++c) x[c] *= sl2;
      } else {
#pragma unroll
        for (int c = 0; c < BN; ++c) x[c] = (kbase + c < vis_end) ? x[c] * sl2 : -INFINITY;
      }
      // block max in four independent chains of 3-input maxima
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < BN; c += 8)
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) mx[k4] = max3f(mx[k4], x[c + 2 * k4], x[c + 2 * k4 + 1]);
      const float mblk = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const float m_new = fmaxf(m_use, mblk);
      if (lane == 0 && (warp & (OWN_WARPS - 1)) == 0) TCX_EV(10, j);
      float alpha = 1.f;
      if (__any_sync(0xffffffffu, m_new > m_use + TAU)) {
        // the whole warp moves to its new maxima (exact for any choice)
        alpha = (m_use == -INFINITY) ? 0.f : ex2_approx(m_use - m_new);
        if (j > 0) {
          const int pj = j - 1;
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_bar[pj & 1], (pj >> 1) & 1, abortf, limit))) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int cc = 0; cc < OCOLS / 32; ++cc) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + TM_O + cc * 32, r);
            tmem_wait_ld();
            reg_fence32(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tmem + lane_base + TM_O + cc * 32, r);
          }
        }
        l *= alpha;
        m_use = m_new;
      }
      const float mu = (m_use == -INFINITY) ? 0.f : m_use;
      if (j >= 2) {  // P buffer j % 2 was read by P_{j-2} V
        const int pj = j - 2;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_bar[pj & 1], (pj >> 1) & 1, abortf, limit))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      // P rows are staged for the other warps to forward: the previous block's
      // have been forwarded
      if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->stg_free, (j - 1) & 1, abortf, limit))) {
        ok = false;
        break;
      }
      if (lane == 0 && (warp & (OWN_WARPS - 1)) == 0) TCX_EV(11, j);
      float lsum = 0.f;
      uint4 *stg = reinterpret_cast<uint4 *>(sst + orow * 16);
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
#pragma unroll
        for (int c = 0; c < 8; ++c) stg[(h * 8 + c) * R] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        if (lane == 0 && (warp & (OWN_WARPS - 1)) == 0) TCX_EV(12 + h, j);
      }
      l += lsum;
      sstal[orow] = alpha;
      mbar_arrive(&bars->stg_full);
      if (lane == 0 && (warp & (OWN_WARPS - 1)) == 0) TCX_EV(2, j);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[j & 1]);
    }
    if (!ok) raise_abort_cluster<NX>(bars, p.status, me);

    // ---- final l and m of every row: owners tell the other CTAs
    if (ok && nblk > 0) {
      if (is_owner) {
#pragma unroll
        for (int q = 0; q < NX; ++q) {
          if (q == (int)me) continue;
          const uint32_t rbar = mapa_shared(smem_u32(&bars->fin_full), (uint32_t)q);
          st_async_u32(mapa_shared(sf_u + (uint32_t)row * 4u, (uint32_t)q), __float_as_uint(l), rbar);
          st_async_u32(mapa_shared(sf_u + (uint32_t)(BM + row) * 4u, (uint32_t)q), __float_as_uint(m_use), rbar);
        }
      } else {
        if (lane == 0 && warp == first_sender) mbar_arrive_expect_tx(&bars->fin_full, (uint32_t)NOTHER * 8u);
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(&bars->fin_full, 0, abortf, limit))) {
          ok = false;
          raise_abort_cluster<NX>(bars, p.status, me);
        } else {
          l = sfin[row];
          m_use = sfin[BM + row];
        }
      }
    }
    // ---- epilogue: O_r / l -> bf16 (or the fp32 partial of this key range), LSE by the owner
    if (ok && nblk > 0) {
      const int last = nblk - 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_bar[last & 1], (last >> 1) & 1, abortf, limit))) {
        raise_abort_cluster<NX>(bars, p.status, me);
        ok = false;
      }
    }
    if (ok) {
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const float lse_val = (m_use == -INFINITY || !(l > 0.f)) ? -INFINITY : (m_use + log2f(l)) * kLn2;
      const int64_t row_idx = (int64_t)bh * p.Nq + qi;
      __nv_bfloat16 *obase = p.o + row_idx * p.D + c0 * 64;
      float *wbase = (nsplit > 1) ? p.ws_o + ((int64_t)split * BH * p.Nq + row_idx) * p.D + c0 * 64 : nullptr;
      for (int cc = 0; cc < OCOLS / 32; ++cc) {
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
            uint4 *dst = reinterpret_cast<uint4 *>(obase + cc * 32);
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
            float4 *dst = reinterpret_cast<float4 *>(wbase + cc * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(__uint_as_float(r[v4 * 4 + 0]) * inv, __uint_as_float(r[v4 * 4 + 1]) * inv,
                                    __uint_as_float(r[v4 * 4 + 2]) * inv, __uint_as_float(r[v4 * 4 + 3]) * inv);
          }
        }
      }
      if (is_owner && qi < p.Nq) {
        if (nsplit == 1)
          p.lse[row_idx] = lse_val;
        else
          p.ws_lse[(int64_t)split * BH * p.Nq + row_idx] = lse_val;
      }
    }
  }

  // ---- teardown: no CTA leaves while another may still write into it
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int NX, int SC, bool UN, bool MASK>
struct XLayout {
  static constexpr int R = BM / NX;
  static constexpr int QB = SC * CHUNK_BYTES;
  static constexpr int IC = UN ? 1 : SC % 2 == 0 ? 2 : SC;
  static constexpr int ITEM_BYTES = IC * CHUNK_BYTES;
  static constexpr int XB = (NX - 1) * R * 512;
  static constexpr int PB = (BM - R) * 256;
  static constexpr int AB = BM * 4;
  static constexpr int SB = R * 256;
  static constexpr int SAB = 512;
  static constexpr int MB = MASK ? R * 256 : 0;  // owner rows' mask values of one block
};

template <int NX, int SC, bool UN, bool MASK>
cudaError_t launch_tcx_n(const Problem &p, int device, uint64_t wait_limit_ns, cudaStream_t stream) {
  using L = XLayout<NX, SC, UN, MASK>;
  constexpr int ITEM_BYTES = L::ITEM_BYTES;
  static_assert(sizeof(XBars) <= 1024, "barrier block too large");
  constexpr int kBarBytes = (int)((sizeof(XBars) + 127) / 128 * 128);
  const int fixed = L::QB + L::XB + L::PB + L::AB + L::SB + L::SAB + L::MB + kBarBytes + 1024 /* alignment */;
  int kst = (kSmemMax - fixed) / ITEM_BYTES;
  if (kst > MAX_KST) kst = MAX_KST;
  if (kst < 2) return cudaErrorInvalidConfiguration;
  XParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.p = p;
  prm.ntiles = (p.Nq + BM - 1) / BM;
  prm.kst = kst;
  prm.off_k = L::QB;
  prm.off_x = prm.off_k + kst * ITEM_BYTES;
  prm.off_p = prm.off_x + L::XB;
  prm.off_a = prm.off_p + L::PB;
  prm.off_s = prm.off_a + L::AB;
  prm.off_sa = prm.off_s + L::SB;
  prm.off_m = prm.off_sa + L::SAB;
  prm.off_bar = prm.off_m + L::MB;
  prm.wait_limit_ns = wait_limit_ns;
  const int smem = (int)prm.off_bar + kBarBytes + 1024;
  if (smem > kSmemMax) return cudaErrorInvalidConfiguration;
  CUtensorMap tq, tk, tv;
  if (!make_chunk_map(&tq, p.q, p.D, p.Nq, p.B * p.Hq, BM, UN ? 1 : SC)) return cudaErrorInvalidValue;
  if (!make_chunk_map(&tk, p.k, p.D, p.Nkv, p.B * p.Hkv, BN, L::IC)) return cudaErrorInvalidValue;
  if (!make_chunk_map(&tv, p.v, p.D, p.Nkv, p.B * p.Hkv, BN, L::IC)) return cudaErrorInvalidValue;
  static std::atomic<int> attr_set[64];
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(attn_tcx_kernel<NX, SC, UN, MASK>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    attr_set[device].store(1, std::memory_order_release);
  }
  const int64_t grid = (int64_t)NX * prm.ntiles * p.B * p.Hq * p.kv_splits;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NX;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // a device that cannot hold one such cluster at a time (a partitioned GPU,
  // say) gets cudaErrorNotSupported, and the caller the per-slice kernel
  static std::atomic<int> fits[64];  // 0 unknown, 1 yes, 2 no
  int f = fits[device].load(std::memory_order_relaxed);
  if (f == 0) {
    int nclusters = 0;
    cudaError_t q = cudaOccupancyMaxActiveClusters(&nclusters, attn_tcx_kernel<NX, SC, UN, MASK>, &cfg);
    if (q != cudaSuccess) {
      cudaGetLastError();
      nclusters = 0;
    }
    f = nclusters > 0 ? 1 : 2;
    fits[device].store(f, std::memory_order_relaxed);
  }
  if (f != 1) return cudaErrorNotSupported;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_tcx_kernel<NX, SC, UN, MASK>, tq, tk, tv, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int tcx_slices(int D) {
  if (!tcx_supports(D)) return 0;
  return D <= 512 ? 2 : 4;
}

bool tcx_supports(int D) {
#ifdef ATTN_NO_TCX
  (void)D;
  return false;
#else
  // from D = 384: at D = 320 the per-slice kernel measured faster (578 against
  // 540 TFLOP/s on B1 H8 N4096), at 448 the two tie
  return D % 64 == 0 && D >= 384 && D <= 1024;
#endif
}

template <bool MASK>
cudaError_t launch_tcx_m(const Problem &p, int device, uint64_t wait_limit_ns, cudaStream_t stream) {
  if (p.D == 384) return launch_tcx_n<2, 3, false, MASK>(p, device, wait_limit_ns, stream);
  if (p.D == 512) return launch_tcx_n<2, 4, false, MASK>(p, device, wait_limit_ns, stream);
  if (p.D == 768) return launch_tcx_n<4, 3, false, MASK>(p, device, wait_limit_ns, stream);
  if (p.D == 1024) return launch_tcx_n<4, 4, false, MASK>(p, device, wait_limit_ns, stream);
  // uneven slices: 2 CTAs up to D = 512, 4 above, at most four chunks each
  const int nc = p.D / 64;
  if (nc == 7) return launch_tcx_n<2, 4, true, MASK>(p, device, wait_limit_ns, stream);
  if (nc >= 9 && nc <= 11) return launch_tcx_n<4, 3, true, MASK>(p, device, wait_limit_ns, stream);
  if (nc >= 13 && nc <= 15) return launch_tcx_n<4, 4, true, MASK>(p, device, wait_limit_ns, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_tcx(const Problem &p, int device, uint64_t wait_limit_ns, cudaStream_t stream) {
  return p.mask ? launch_tcx_m<true>(p, device, wait_limit_ns, stream)
                : launch_tcx_m<false>(p, device, wait_limit_ns, stream);
}

}  // namespace attn
