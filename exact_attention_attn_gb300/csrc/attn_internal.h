// Internal declarations shared by the host launcher and the kernel
// translation units of libattn_gb300.so.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace attn {

// One attention forward problem, as validated by attn_fwd.
struct Problem {
  const __nv_bfloat16 *q;  // [B, Hq, Nq, D]
  const __nv_bfloat16 *k;  // [B, Hkv, Nkv, D]
  const __nv_bfloat16 *v;  // [B, Hkv, Nkv, D]
  __nv_bfloat16 *o;        // [B, Hq, Nq, D]
  float *lse;              // [B, Hq, Nq]
  int B, Hq, Hkv, Nq, Nkv, D;
  float scale;
  int causal;
  int *status;             // device status word (first error wins)
  // split-KV: kv_splits CTAs share each query tile, each over a contiguous
  // range of key blocks; with kv_splits > 1 the kernels write normalised fp32
  // partial outputs ws_o [kv_splits, B*Hq, Nq, D] and partial natural-log
  // LSEs ws_lse [kv_splits, B*Hq, Nq] instead of o and lse.
  int kv_splits;
  float *ws_o;
  float *ws_lse;
  // test support (attn_set_debug): bit 0 makes the V producer of the
  // two-tile kernel skip its copy of the second key block, so that the MMA
  // thread's bounded wait for it runs out
  int debug_flags;
  // optional additive mask (null: none): bf16 value for (b, hq, query row i,
  // key j) at mask[b * mask_sb + hq * mask_sh + i * mask_sq + j]; the strides
  // are element counts, multiples of 8 (0 broadcasts that dimension)
  const __nv_bfloat16 *mask;
  int64_t mask_sb, mask_sh, mask_sq;
};

// Device status codes written by kernels (same values as the public ATTN_ERR_*).
constexpr int kStatusTimeout = -5;
constexpr int kStatusDevice = -7;

// TMA map of a [planes, rows, cols] bf16 tensor (cols contiguous) with
// 128-row x 64-column boxes and the 128-byte swizzle.  False on failure.
bool make_tile_map(CUtensorMap *m, const void *base, int cols, int rows, int planes);

// TMA map of the same tensor whose box is box_rows rows x all of its columns,
// landing in shared memory as cols/64 consecutive [box_rows x 64] chunks with
// the 128-byte swizzle.  One copy moves a whole K or V block: large copies
// keep more bytes in flight per TMA operation.
bool make_block_map(CUtensorMap *m, const void *base, int cols, int rows, int planes, int box_rows);
// Same view, box of box_chunks chunks starting at the chunk coordinate given
// to the copy (chunks past the last one read as zeros).
bool make_chunk_map(CUtensorMap *m, const void *base, int cols, int rows, int planes, int box_rows, int box_chunks);

// TMA map of a [planes, rows, inner] byte tensor (inner contiguous, at least
// 128 and a multiple of 16) with 128 x 128-byte boxes and the 128-byte swizzle.
bool make_u8_map(CUtensorMap *m, const void *base, int inner, int rows, int planes);

// Shared-memory plan of the tensor-core kernel for head dim D.
struct TcConfig {
  int nc;       // 64-column chunks of D
  int nslices;  // output slices (each <= 256 columns)
  int vmax;     // chunks in the widest slice
  int qres;     // Q tile resident in shared memory (else streamed through the ring)
  int vring;    // V blocks travel through the Q/K ring too (Q resident, no V slot)
  int kst;      // Q/K ring depth (32 KB slots of two chunks)
  int vst;      // V-ring depth (slices)
  int mask_bytes;  // shared memory for one block's mask values (0 without a mask)
  uint32_t off_q, off_k, off_v, off_m, off_bar;
  int smem_bytes;
};
TcConfig tc_config(int D, bool mask = false);

// Tensor-core kernel (tcgen05/TMEM/TMA): every D multiple of 64 up to 1024,
// Nkv >= 1.  Bounded waits give up after wait_limit_ns.
cudaError_t launch_tc(const Problem &p, int device, uint64_t wait_limit_ns, cudaStream_t stream);

// Cluster Split-D kernel for head dims 384 ... 1024: the output
// slices of a tile (2 or 4) are the CTAs of one cluster, which compute the
// scores once (partial products over their slices, summed through
// distributed shared memory).
bool tcx_supports(int D);
int tcx_slices(int D);  // CTAs per cluster (D-slices per tile), 0 when not supported
cudaError_t launch_tcx(const Problem &p, int device, uint64_t wait_limit_ns, cudaStream_t stream);

// Two-tile ping-pong tensor-core kernel for head dims 64 and 128.
bool tc2_supports(int D);
cudaError_t launch_tc2(const Problem &p, int device, uint64_t wait_limit_ns, cudaStream_t stream);

// Merge kv_splits partial results into o (bf16) and lse: LSE = ln sum_s
// exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.  Memory-bound, one pass.
cudaError_t launch_combine(const Problem &p, cudaStream_t stream);

// Stream-ordered scratch from the current device's library pool (the one the
// split-KV workspace comes from; cudaMallocAsync while `st` is captured).
// Free with cudaFreeAsync on the same stream.
cudaError_t scratch_alloc(void **ptr, size_t bytes, cudaStream_t st);

// Waits for every device whose host-copy pool (attn_fwd_host) holds memory
// and returns that pool's unused memory to the driver; leaves the current
// device changed (the caller restores it).
cudaError_t release_host_copy_memory();

// Bound on device-side waits and debug flags currently set by attn_set_debug.
uint64_t wait_limit_ns();
int debug_flags();

// Current device (as attn_fwd sees it): index, SM count, status word.
int current_device(int *device, int *sm_count, int **status);
// Records a CUDA error for attn_last_cuda_error; returns ATTN_ERR_LAUNCH.
int record_cuda_error(cudaError_t e);
// The size and flag checks of attn_fwd (ATTN_OK or ATTN_ERR_ARG), no device work.
int check_problem(int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal);

// Problems with no keys: O = 0 and LSE = -inf everywhere (grid of at most
// 8 CTAs per SM, grid-stride).
cudaError_t launch_nokeys(const Problem &p, int sm_count, cudaStream_t stream);

// Most key-range splits attn_fwd_splitkv accepts.
constexpr int kMaxSplits = 64;

// The tensor-core kernel for the head dim, as attn_fwd picks it: two-tile
// (D 64, 128), cluster Split-D (D 384 ... 1024, unless ATTN_DEBUG_NO_CLUSTER
// is set or the device cannot hold one cluster), else the per-slice kernel.
// p.kv_splits > 1 writes the partials to p.ws_o / p.ws_lse.
cudaError_t launch_tensor(const Problem &p, int device, cudaStream_t stream);

}  // namespace attn
