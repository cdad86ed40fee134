"""Oracle for the FP8 forward path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module; the product path never does.  It shares no code with
the CUDA path.

What the pages fix, by page title and section:

* "FlashAttention v1/v2/v3/v4" (lo0.es), "FA3 -- el momento Hopper": FP8
  attention quantises Q and K (and V) to FP8 with one scale per tile of rows
  (64 x d there) instead of one per tensor, after multiplying by a
  Hadamard-based orthogonal matrix that spreads outliers.
* "ZYFA: FP8 FlashAttention Kernels for AMD MI355X", "The ZYFA accuracy work
  is the sleeper contribution" and "Getting started with ZYFA": a Hadamard
  rotation of Q and K before quantisation; power-of-two descales; "The
  three techniques" (per-block scaling): probabilities are multiplied by a
  power of two before they are rounded to FP8 and the factor is divided
  back out.

Readings where the pages leave the details open (also listed in the design
notes):

1. FP8 format: e4m3 (4 exponent bits, bias 7, 3 mantissa bits, no
   infinities, largest finite 448, subnormals down to 2^-9), rounding to
   nearest with ties to even, saturating at +-448.
2. Rotation: the Sylvester Hadamard matrix H (H_1 = [1], H_2n = [[H, H],
   [H, -H]]) scaled by 1/sqrt(D), applied to every row of Q and of K (not to
   V): (Q H)(K H)^T = Q K^T because H H^T = I.  Computed as the fast
   transform in float32 (butterflies of stride 1, 2, 4, ..., D/2, then one
   multiply by the float32 value of 1/sqrt(D)), the same order and precision
   the kernel uses, because its result decides the FP8 codes.
3. Scales: powers of two.  Q and K: one per block of 128 rows of one head
   (the kernel's tile); V: one per (b, kv head).  The scale of a block with
   largest magnitude a is 2^k for the smallest integer k with a <= 448 2^k
   (k = 0 for an all-zero block); codes are e4m3(x / 2^k).
4. The reference for the kernel is exact attention (the float64 oracle) on
   the dequantised inputs 2^k e4m3(x / 2^k).  The kernel also rounds P to
   e4m3 (times a power of two, divided back out); that rounding is an approximation
   the tolerance accounts for, not part of this reference.
"""
from __future__ import annotations

import math

import numpy as np

from .attention import attention

E4M3_MAX = 448.0
BLOCK_ROWS = 128


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value of each element (ties to even), saturated at
    +-448; float64 in, float64 out.  A binade [2^e, 2^(e+1)) with e >= -6
    holds 8 values 2^(e-3) apart; below 2^-6 the spacing stays 2^-9."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, E = np.frexp(np.where(a > 0, a, 1.0))     # a = m 2^E, m in [0.5, 1)
    e = np.clip(E - 1, -6, 8)                     # binade exponent, subnormals share -6
    step = np.ldexp(1.0, e - 3)
    q = np.minimum(np.round(a / step) * step, E4M3_MAX)   # np.round: ties to even
    return np.where(x < 0, -q, q)


def fwht_f32(x) -> np.ndarray:
    """Unnormalised Sylvester Walsh-Hadamard transform of the last axis
    (length a power of two) in float32: butterflies (a, b) -> (a + b, a - b)
    of stride 1, 2, 4, ...  Equals x @ H for the Sylvester matrix H."""
    y = np.array(x, dtype=np.float32)
    D = y.shape[-1]
    if D & (D - 1):
        raise ValueError("length must be a power of two")
    lead = y.shape[:-1]
    h = 1
    while h < D:
        z = y.reshape(lead + (D // (2 * h), 2, h))
        a, b = z[..., 0, :], z[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(lead + (D,))
        h *= 2
    return y


def rotate_f32(x) -> np.ndarray:
    """x H / sqrt(D) in float32 (reading 2)."""
    D = np.asarray(x).shape[-1]
    return fwht_f32(x) * np.float32(1.0 / math.sqrt(D))


def pow2_scale(amax) -> np.ndarray:
    """2^k for the smallest integer k with amax <= 448 2^k (reading 3); 1 for
    amax == 0.  With amax = m 2^E, m in [0.5, 1), and 448 = 0.875 2^9:
    k = E - 9, plus one when m > 0.875."""
    a = np.asarray(amax, dtype=np.float64)
    m, E = np.frexp(np.where(a > 0, a, 1.0))
    k = E - 9 + (m > 0.875)
    return np.where(a > 0, np.ldexp(1.0, k), 1.0)


def quantize_row_blocks(x, block: int = BLOCK_ROWS):
    """x [..., N, D] (float32 values): per block of `block` rows, the scale
    s = pow2_scale(max |x|) and the dequantised values s e4m3(x / s).
    Returns (dequantised float64 [..., N, D], scales [..., ceil(N/block)])."""
    x = np.asarray(x, dtype=np.float64)
    N = x.shape[-2]
    nb = (N + block - 1) // block
    out = np.empty_like(x)
    scales = np.empty(x.shape[:-2] + (nb,))
    for j in range(nb):
        blk = x[..., j * block:(j + 1) * block, :]
        s = pow2_scale(np.abs(blk).max(axis=(-2, -1)) if blk.size else np.zeros(x.shape[:-2]))
        scales[..., j] = s
        out[..., j * block:(j + 1) * block, :] = s[..., None, None] * e4m3_round(blk / s[..., None, None])
    return out, scales


def quantize_heads(x):
    """x [B, H, N, D]: one scale per (b, h) head.  Returns (dequantised, scales [B, H])."""
    x = np.asarray(x, dtype=np.float64)
    s = pow2_scale(np.abs(x).max(axis=(-2, -1)) if x.size else np.zeros(x.shape[:2]))
    return s[..., None, None] * e4m3_round(x / s[..., None, None]), s


def fp8_inputs(q, k, v, block: int = BLOCK_ROWS):
    """The FP8 path's view of bf16 inputs (any float arrays whose values are
    exact in float32): Q and K rotated (reading 2) and quantised per block of
    rows, V quantised per head.  Returns dequantised float64 (q, k, v) and
    the scales (sq [B, Hq, nqb], sk [B, Hkv, nkb], sv [B, Hkv])."""
    qd, sq = quantize_row_blocks(rotate_f32(q), block)
    kd, sk = quantize_row_blocks(rotate_f32(k), block)
    vd, sv = quantize_heads(np.asarray(v, dtype=np.float32))
    return (qd, kd, vd), (sq, sk, sv)


def attention_fp8(q, k, v, scale: float, causal: bool, rows=None):
    """Exact attention (float64) on the FP8 path's dequantised inputs."""
    (qd, kd, vd), _ = fp8_inputs(q, k, v)
    return attention(qd, kd, vd, scale, causal, rows)
