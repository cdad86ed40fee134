/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact attention forward library
 * (libattn_gb300.so).
 *
 * The operation.  For every batch b and query head hq, with key/value head
 * kv = hq / (Hq / Hkv):
 *
 *     S   = scale * Q[b,hq] K[b,kv]^T                      (Nq x Nkv)
 *     S_ij = -inf where causal and j > i + (Nkv - Nq)
 *     O   = softmax_rows(S) V[b,kv]                        (Nq x D)
 *     LSE_i = ln sum_j exp(S_ij)
 *
 * Sources (page title, section):
 *   - "FlashAttention: Fast and Memory-Efficient Exact Attention with
 *     IO-Awareness" (summary card): exact attention computed in SRAM-sized
 *     tiles; the N x N score matrix is never written to HBM.
 *   - "FlashAttention v1/v2/v3/v4: el bibliotecario que nunca despeja la mesa"
 *     (lo0.es), "El truco que hizo posible todo: online softmax": the running
 *     max m and running sum l; the result equals the standard softmax.
 *   - "ffpa-attn 0.2.3" (FFPA README), feature table and "Quick Start":
 *     (B, H, N, D) layout, self-attention, cross-attention (Nq != Nkv),
 *     GQA/MQA (Hq != Hkv), causal masking, head dims up to 1024;
 *     "Split-D and TiledMMA": the D axis is split so on-chip staging does not
 *     grow with D.
 *   - "ZYFA: FP8 FlashAttention Kernels for AMD MI355X", "The details that
 *     make it production-grade" and "Getting started with ZYFA": LSE for
 *     merging partial results over key ranges; a call that never waits on
 *     the host.
 *
 * Conventions the pages leave open (chosen here): LSE is the natural log;
 * causal masking with Nq != Nkv is bottom-right aligned; a query row that
 * sees no key gets O = 0 and LSE = -inf; GQA groups are consecutive query
 * heads.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *attn_stream_t;

/* Return codes.  0 is success; every error is negative. */
#define ATTN_OK 0
#define ATTN_ERR_ARG (-1)     /* a null pointer, a bad size, Hq % Hkv != 0, an unsupported D, a non-finite scale */
#define ATTN_ERR_ALIGN (-2)   /* a tensor base address not 16-byte aligned */
#define ATTN_ERR_ARCH (-3)    /* the current device is not a compute capability 10.3 GPU (sm_103) */
#define ATTN_ERR_LAUNCH (-4)  /* a CUDA runtime or driver call failed; attn_last_cuda_error() has its text */
#define ATTN_ERR_TIMEOUT (-5) /* a kernel's bounded wait ran out (reported by attn_fwd_status) */
#define ATTN_ERR_NOMEM (-6)   /* the split-KV workspace could not be allocated */
#define ATTN_ERR_DEVICE (-7)  /* a kernel's own consistency check failed (reported by attn_fwd_status) */
#define ATTN_ERR_SCRATCH (-8) /* attn_fwd_splitkv_noalloc: the partials need more than ATTN_NOALLOC_SCRATCH_BYTES */

#define ATTN_MAX_HEAD_DIM 1024

/*
 * attn_fwd -- exact scaled-dot-product attention forward, bf16 in, bf16 O and
 * fp32 LSE out.
 *
 * q    device pointer, bf16, [B, Hq, Nq, D], contiguous (D fastest).
 * k, v device pointers, bf16, [B, Hkv, Nkv, D], contiguous.
 * o    device pointer, bf16, [B, Hq, Nq, D], contiguous; fully written.
 * lse  device pointer, fp32, [B, Hq, Nq]; fully written (natural log).
 * B, Nq, Nkv >= 0; Hq >= 1, Hkv >= 1, Hq % Hkv == 0.  B * Nq == 0 is an empty
 *      problem (returns ATTN_OK without launching).  Nkv == 0 gives O = 0 and
 *      LSE = -inf everywhere.
 * D    head dim: a multiple of 64 in [64, 1024].
 * scale  finite multiplier of Q K^T (1/sqrt(D) is the usual choice).
 * causal  0 or 1; 1 masks key j for query i when j > i + (Nkv - Nq).
 * stream  the CUDA stream to run on.
 *
 * All pointers are owned by the caller and must stay valid until the stream
 * reaches the work.  o must not overlap q, k, v or lse.  Every base address
 * must be 16-byte aligned.  The call validates its arguments on the host,
 * launches asynchronously on `stream` and returns without waiting.  It may
 * take a stream-ordered split-KV workspace (see attn_fwd_splitkv) when the
 * problem has too few query tiles to fill the GPU.  Bounded device-side waits that run out are not
 * reported here: call attn_fwd_status.
 *
 * CUDA graphs: the call keeps no state between calls that a graph replay
 * would miss (the tensor maps are kernel parameters, the workspace is
 * stream-ordered), so it may be captured into a graph once the same sizes
 * have run outside capture on that device (the first call of a size does
 * one-time set-up that capture forbids: device facts, kernel attributes, the
 * cluster-fit query).  A replay reads and writes the captured pointers.
 *
 * Returns ATTN_OK or a negative ATTN_ERR_* code; on error nothing is launched.
 */
ATTN_API int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int Hq, int Hkv, int Nq, int Nkv, int D,
             float scale, int causal, attn_stream_t stream);

/*
 * attn_fwd_splitkv -- attn_fwd with an explicit number of key-range splits.
 *
 * The key blocks of every query tile are cut into kv_splits contiguous
 * ranges, each handled by its own CTA, which writes a normalised fp32 partial
 * output and a partial LSE; a second kernel merges them (LSE = ln sum_s
 * exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s) -- the merge of partial results
 * over key ranges through their LSE described on the ZYFA page ("The details
 * that make it production-grade").  This spreads a problem with few query
 * tiles and many keys over all SMs.
 *
 * kv_splits: 0 chooses automatically (what attn_fwd does); 1 disables the
 *   split; 2..64 forces that many ranges (ranges left empty are harmless).
 * Workspace: kv_splits * B * Hq * Nq * (D + 1) * 4 bytes, stream-ordered on
 *   `stream` (allocated before the kernels, freed after the merge) from a
 *   memory pool of the library's that keeps its memory between calls (a
 *   device holds up to the largest workspace asked for, until the process
 *   exits); while `stream` is being captured into a CUDA graph it is taken
 *   with cudaMallocAsync instead (a graph memory node).  ATTN_ERR_NOMEM if it
 *   cannot be had.
 * Everything else (arguments, layouts, asynchrony, errors) is as attn_fwd.
 */
ATTN_API int attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                              float scale, int causal, int kv_splits, attn_stream_t stream);

/*
 * attn_fwd_masked -- attn_fwd with an additive attention mask.
 *
 * The FFPA README's feature table lists a mask besides the causal one
 * ("Causal/Mask"); it is read here as SDPA's additive float mask.  With
 * M[b, hq, i, j] the mask value, the scores become
 *
 *     S_ij = scale * Q[b,hq]_i . K[b,kv]_j + M[b, hq, i, j]
 *
 * before the row softmax; an entry of -inf hides key j from query i, and the
 * causal flag, if set, hides j > i + (Nkv - Nq) on top.  LSE is ln sum_j
 * exp(S_ij) over the visible keys; a row whose keys are all hidden gets
 * O = 0 and LSE = -inf.
 *
 * mask   device pointer, bf16; the value for (b, hq, i, j) is at element
 *        b * mask_stride_b + hq * mask_stride_h + i * mask_stride_q + j.
 *        Keys (j) are contiguous.  Strides are element counts >= 0 and
 *        multiples of 8 (16 bytes); a stride of 0 broadcasts that dimension
 *        (e.g. one [Nq, Nkv] mask for every batch and head, or a key-padding
 *        mask [B, 1, 1, Nkv] with mask_stride_h = mask_stride_q = 0).  The
 *        base must be 16-byte aligned.  Values must be finite or -inf
 *        (+inf and NaN give undefined results).  Every element the strides
 *        address for j < Nkv must be readable; nothing past Nkv is read.
 * Everything else (arguments, layouts, automatic key splits, asynchrony,
 * errors, CUDA-graph capture) is as attn_fwd.  Returns ATTN_ERR_ARG for a
 * null mask or a negative stride, ATTN_ERR_ALIGN for a stride that is not a
 * multiple of 8 or a misaligned base.
 */
ATTN_API int attn_fwd_masked(const void *q, const void *k, const void *v, const void *mask,
                             long long mask_stride_b, long long mask_stride_h, long long mask_stride_q,
                             void *o, float *lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                             float scale, int causal, attn_stream_t stream);

/*
 * attn_fwd_host -- attn_fwd on host buffers.
 *
 * q, k, v, o and lse are HOST pointers with the layouts of attn_fwd
 * (contiguous [B, H, N, D] bf16, lse [B, Hq, Nq] fp32; no alignment needed).
 * The call copies the inputs to the current device, runs the same kernels as
 * attn_fwd (the same key split count, so O and LSE are bit-identical to
 * attn_fwd's), copies O and LSE back and returns when they are in host
 * memory: the caller may reuse every buffer at once.
 *
 * The work is cut by (b, kv head) group -- independent attention problems
 * whose rows are contiguous -- into chunks of about 25 MiB of inputs (at most
 * 8, at most one per group; measured best on GB300 for 100-200 MB problems,
 * where more chunks lost to the copies of the two directions sharing the
 * host link); a chunk's inputs go up
 * on a copy stream of the library's, its kernels run on a compute stream of
 * the library's (one per chunk) as soon as they have landed, and its outputs
 * come down on a second copy stream, so that the copies of one chunk overlap
 * the kernels and the copies of the others, and chunks too small to fill the
 * GPU compute side by side.  The work starts after what `stream` holds at the
 * call and the call returns when all of it is done.
 * The copies overlap only when the host buffers are page-locked
 * (cudaHostAlloc / cudaHostRegister); with pageable memory the call is still
 * correct but the copies run one after the other.
 *
 * Device memory: one stream-ordered block on `stream` for the device copies
 * of all five tensors (plus what attn_fwd itself may take for key splits),
 * freed before the call returns into a memory pool of the library's that keeps
 * it for the next call (a device holds up to the largest block asked for).
 * The library's streams are created on a device's first call and reused;
 * calls on the same device serialise on them
 * (the call is synchronous anyway).  Errors: those of attn_fwd, plus
 * ATTN_ERR_NOMEM when the device block cannot be allocated.
 *
 * The pages describe no host-buffer entry point; this one exists so that the
 * library can be measured, and used, end to end from host memory.
 */
ATTN_API int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                           float scale, int causal, attn_stream_t stream);

/*
 * attn_fwd_splitkv_noalloc -- attn_fwd_splitkv that allocates nothing.
 *
 * The pages have no counterpart of this call; it exists for callers that may
 * not allocate device memory while they run attention: code that owns every
 * byte of the GPU through its own allocator or memory budget (a serving
 * process that pins its KV cache and activations up front and must not have
 * a library take memory behind its back), hard-latency paths where an
 * allocation -- even a stream-ordered one from a pool that may have to grow --
 * is an unbounded stall, and callers in contexts where the CUDA allocator
 * may not be used at all.  Instead of a per-call workspace it uses one
 * fixed, file-scope device array of ATTN_NOALLOC_SCRATCH_BYTES bytes that
 * every GPU which loads this library holds until the process exits.
 *
 * Arguments, checks, kernels, the device-side wait bound and the debug flags
 * of attn_set_debug are those of attn_fwd_splitkv, except that kv_splits must
 * be an explicit count from 2 to 64 (ATTN_ERR_ARG otherwise).  The partials need
 * kv_splits * B * Hq * Nq * (D + 1) * 4 bytes; a larger problem is refused
 * with ATTN_ERR_SCRATCH before anything is launched.  Nkv == 0 needs no
 * partials and runs the plain no-key path.
 *
 * Set-up: the first call on a device looks up the array's device address
 * with cudaGetSymbolAddress (with that device current); make that first call
 * outside any stream capture.  No call of this function allocates or frees
 * device memory.  The address is kept for the life of the process, like the
 * library's other per-device facts: do not call the library on a device
 * again after cudaDeviceReset has destroyed its context.
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents.  Nothing in it has to start at zero -- each call writes
 * every partial it later reads -- but two calls whose kernels overlap on the
 * GPU (different streams, or a second call before the first one's kernels
 * have finished on another stream) race on the array and corrupt each
 * other's results; serialise them, e.g. on one stream.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (16u << 20)
ATTN_API int attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                                      int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                                      float scale, int causal, int kv_splits, attn_stream_t stream);

/*
 * attn_bwd -- exact attention backward: the gradients of attn_fwd's O with
 * respect to q, k and v, given the upstream gradient dout of O.
 *
 * With P the row softmax of S = scale * Q K^T (causal entries hidden as in
 * attn_fwd; P = 0 where hidden) and O = P V, the chain rule through the row
 * softmax gives
 *     dV = P^T dO,   dP = dO V^T,   Delta_i = sum_d dO_id O_id,
 *     dS = P * (dP - Delta),   dQ = scale * dS K,   dK = scale * dS^T Q,
 * and a key/value head shared by a GQA group receives the sum over its query
 * heads.  As the FlashAttention pages describe the backward pass ("FlashAttention
 * v1/v2/v3/v4", "FA1 -- el cambio de orden de las operaciones"; the
 * FlashAttention summary card), S is recomputed block by block from Q, K and
 * the forward's row statistics (here LSE); nothing N x N is stored.
 *
 * q, k, v   the forward's inputs (layouts of attn_fwd).
 * o, lse    the forward's outputs for these inputs (attn_fwd's O and LSE).
 * dout      bf16 [B, Hq, Nq, D], the gradient of the loss with respect to O.
 * dq        bf16 [B, Hq, Nq, D]; dk, dv bf16 [B, Hkv, Nkv, D]: fully written.
 * D         64 or 128 (other head dims: ATTN_ERR_ARG).
 * Every other argument, the checks, alignment (16 bytes for every pointer)
 * and asynchrony are as attn_fwd.  Rows that see no key get dq = 0; keys
 * that no query sees get dk = dv = 0.  The result is deterministic (no
 * atomics: one kernel accumulates dK, dV per key tile over the queries of
 * the whole GQA group, another dQ per query tile over the keys).  A
 * stream-ordered scratch of 2 * B * Hq * ceil(Nq / 128) * 128 * 4 bytes is
 * taken from the library's pool (see attn_fwd_splitkv); ATTN_ERR_NOMEM if it
 * cannot be had.  CUDA graphs: as attn_fwd (while the stream is captured the
 * scratch becomes a graph memory node).  The additive mask of
 * attn_fwd_masked has no backward here.
 */
ATTN_API int attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                      const float *lse, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Nq, int Nkv,
                      int D, float scale, int causal, attn_stream_t stream);

/*
 * attn_fp8_quantize / attn_fwd_fp8 -- FP8 (e4m3) attention forward, head
 * dim 128.
 *
 * The FP8 scheme of the FlashAttention blog ("FlashAttention v1/v2/v3/v4",
 * "FA3 -- el momento Hopper": per-tile scales and a Hadamard-based rotation
 * before quantising) and of the ZYFA page (a Hadamard rotation of Q and K,
 * power-of-two descales, probabilities scaled by a power of two before they
 * are rounded to FP8).  attn_fp8_quantize turns bf16 q, k, v into:
 *   q8   uint8 [B, Hq, Nq, 128]: e4m3 codes of (q_row H / sqrt(128)) / sq,
 *        H the Sylvester Hadamard matrix, per 128-row block of one head;
 *   sq   float [B, Hq, ceil(Nq/128)]: the blocks' scales, powers of two, the
 *        smallest 2^k with max |x| <= 448 * 2^k;
 *   k8, sk  the same for k: [B, Hkv, Nkv, 128] and [B, Hkv, ceil(Nkv/128)];
 *   vt8  uint8 [B, Hkv, 128, nkv_pad], nkv_pad = 128 * ceil(Nkv / 128): e4m3
 *        codes of v / sv, transposed (keys contiguous), code 0 past Nkv;
 *   sv   float [B, Hkv]: one power-of-two scale per (b, kv head).
 * attn_fwd_fp8 computes O (bf16 [B, Hq, Nq, 128]) and LSE (fp32 [B, Hq, Nq])
 * from them: S = sq sk (q8 k8^T) on the FP8 tensor cores (the rotation
 * cancels: (qH)(kH)^T = q k^T), the online softmax of attn_fwd with a lazy
 * rescale threshold of 6.5 (log2 units), P rounded to e4m3 as 2^2 p, and
 * O = sv (P8 v8) / (2^2 l) with l the fp32 sum of p.  The result approximates
 * attn_fwd's; it equals exact attention on the dequantised inputs up to the
 * e4m3 rounding of P.
 *
 * D must be 128; attn_fwd_fp8 also needs a finite scale > 0 (ATTN_ERR_ARG
 * otherwise).  Every pointer is a device pointer owned by the caller, 16-byte
 * aligned; sizes, causal masking (bottom-right), rows with no key, GQA,
 * asynchrony, errors and CUDA-graph capture are as attn_fwd (neither call
 * allocates).  No key-range splits.
 */
ATTN_API int attn_fp8_quantize(const void *q, const void *k, const void *v, void *q8, void *k8, void *vt8,
                               float *sq, float *sk, float *sv, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                               attn_stream_t stream);
ATTN_API int attn_fwd_fp8(const void *q8, const void *k8, const void *vt8, const float *sq, const float *sk,
                          const float *sv, void *o, float *lse, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                          float scale, int causal, attn_stream_t stream);

/*
 * attn_fwd_status -- synchronise `stream`, then read and clear the device
 * status word of the current device.  Returns ATTN_OK, ATTN_ERR_TIMEOUT (a
 * bounded mbarrier wait inside a kernel gave up; that kernel's outputs are
 * undefined), ATTN_ERR_DEVICE, or ATTN_ERR_LAUNCH if the synchronisation
 * itself reported a CUDA error.
 */
ATTN_API int attn_fwd_status(attn_stream_t stream);

/*
 * attn_set_debug -- test support for the failure path; process-wide, read at
 * every later launch.
 *
 * flags: an OR of
 *   ATTN_DEBUG_DROP_V_COPY, which makes the V producer of the head-dim-64/128
 *     kernel skip its copy of each CTA's second key block, so the MMA
 *     thread's wait for it runs out: the kernel then records ATTN_ERR_TIMEOUT
 *     in the status word, every role of the CTA stops waiting, drains its own
 *     copies and MMAs, frees its tensor memory and exits (no trap, no hang;
 *     outputs of that call are undefined);
 *   ATTN_DEBUG_NO_CLUSTER, which runs head dims 384 ... 1024 on the
 *     per-slice Split-D kernel (each output slice recomputes the scores)
 *     instead of the cluster kernel, the path a device takes when it cannot
 *     hold one cluster; results agree within the parity tolerances;
 *   ATTN_DEBUG_HOST_CHUNKS, which makes attn_fwd_host cut every problem into
 *     one chunk per (b, kv head) group (up to its most, 8), whatever its size,
 *     so that small problems take the chunked copy path; results stay
 *     bit-identical to attn_fwd.
 * wait_limit_ns: bound on every device-side wait; 0 restores the default
 *   (2 s).
 * Returns ATTN_OK or ATTN_ERR_ARG.
 */
#define ATTN_DEBUG_DROP_V_COPY 1
#define ATTN_DEBUG_NO_CLUSTER 2
#define ATTN_DEBUG_HOST_CHUNKS 4
ATTN_API int attn_set_debug(int flags, long long wait_limit_ns);

/* Static description of a return code. */
ATTN_API const char *attn_strerror(int code);

/* Text of the last CUDA error seen by this library on the calling thread
 * ("" if none). */
ATTN_API const char *attn_last_cuda_error(void);

/*
 * attn_fwd_plan -- describe, without launching anything, the kernels attn_fwd
 * (automatic split choice) would run for these sizes on the current device.  Sizes are checked as in
 * attn_fwd (pointers are not involved).  Fills *plan and returns ATTN_OK, or
 * returns a negative ATTN_ERR_* code.
 */
#define ATTN_PATH_NONE 0      /* empty problem: nothing is launched */
#define ATTN_PATH_NOKEYS 1    /* no keys (Nkv == 0): a fill kernel writes O = 0, LSE = -inf */
#define ATTN_PATH_TC 2        /* tcgen05 tensor-core kernel */
#define ATTN_PATH_TC_SPLITKV 3 /* tcgen05 kernel over key splits + LSE merge kernel */

typedef struct attn_plan {
  int path;                  /* ATTN_PATH_* */
  int launches;              /* kernel launches per attn_fwd call */
  int grid;                  /* CTAs of the main kernel */
  int kv_splits;             /* key-range splits (1 = none) */
  int d_slices;              /* output head-dim slices per query tile */
  long long workspace_bytes; /* split-KV workspace allocated per call */
} attn_plan;

ATTN_API int attn_fwd_plan(int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, attn_plan *plan);

/* Library version as major * 10000 + minor * 100 + patch. */
ATTN_API int attn_version(void);

/*
 * attn_shutdown -- give back the device memory the library's pools hold.
 *
 * The split-KV workspace (attn_fwd, attn_fwd_splitkv, attn_fwd_masked,
 * attn_bwd's per-row vectors) and the device copies of attn_fwd_host come
 * from memory pools of the library's that keep their memory between calls.
 * This call waits until every device the library has used for them is idle
 * (cudaDeviceSynchronize on each, so also for work that is not the
 * library's), then trims each pool to nothing.  The library stays usable:
 * later calls grow the pools again.  The fixed 16 MiB scratch of
 * attn_fwd_splitkv_noalloc is part of the loaded module and stays.
 * Call it when no other thread is calling the library.
 * Returns ATTN_OK, or ATTN_ERR_LAUNCH with the first CUDA error (see
 * attn_last_cuda_error); the current device is restored.
 */
ATTN_API int attn_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
