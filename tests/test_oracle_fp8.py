"""Pins for the FP8 oracle (oracle/fp8.py): each piece against something
other than itself, and planted mistakes that must fail a pin.

Sources: "FlashAttention v1/v2/v3/v4" (lo0.es), "FA3 -- el momento Hopper"
(FP8 with per-tile scales and a Hadamard-based rotation); "ZYFA: FP8
FlashAttention Kernels for AMD MI355X" (Hadamard rotation of Q and K before
quantisation, power-of-two descales).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def rnd(shape, seed, amp=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * amp


def torch_e4m3(x):
    """torch's float8_e4m3fn cast (round to nearest even; used below 448 only)."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# checks: each returns a deviation (0 is perfect) for a candidate function set

def check_e4m3_vs_torch(round_fn):
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(4000) * 30, rng.standard_normal(2000) * 1e-2, rng.uniform(-448, 448, 2000),
        # ties: midpoints between neighbouring codes, normal and subnormal
        np.array([1.0625, 1.1875, 2.125, 0.0029296875, 0.0009765625, 0.00146484375, 464.0 - 1e-9, 240.0, 248.0]),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    return float(np.abs(round_fn(x) - torch_e4m3(x)).max())


def check_e4m3_codes_fixed(round_fn):
    """Every finite e4m3 code (all 256 bit patterns but NaN) is a fixed
    point, and values past 448 saturate."""
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    codes = codes[np.isfinite(codes)]
    dev = np.abs(round_fn(codes) - codes).max()
    sat = np.abs(round_fn(np.array([449.0, 500.0, 1e6, -470.0])) - np.array([448.0, 448.0, 448.0, -448.0])).max()
    return float(max(dev, sat))


def check_fwht(fwht):
    """Against scipy's Sylvester Hadamard matrix: x @ H (float64 reference,
    float32 transform), and the normalised transform keeps the norm."""
    sl = pytest.importorskip("scipy.linalg")
    worst = 0.0
    for D in (2, 8, 64, 128):
        x = rnd((5, D), D).astype(np.float32)
        H = sl.hadamard(D).astype(np.float64)
        ref = x.astype(np.float64) @ H
        worst = max(worst, np.abs(fwht(x) - ref).max() / np.abs(ref).max())
        y = fwht(x).astype(np.float64) / math.sqrt(D)
        worst = max(worst, np.abs(np.linalg.norm(y, axis=1) - np.linalg.norm(x, axis=1)).max())
    return float(worst)


def check_scale_rule(scale_fn):
    """pow2_scale(a) is a power of two s with a/s <= 448 < 2 a/s (the
    smallest such), and 1 for a = 0."""
    a = np.concatenate([np.abs(rnd(2000, 3, 50.0)), [448.0, 448.0 * 2, 448.0 * 2 ** -5, 392.0, 393.0, 1e-30]])
    s = scale_fn(a)
    m, _ = np.frexp(s)
    bad = (m != 0.5) | (a / s > 448.0) | (2 * a / s <= 448.0)
    return float(bad.sum() + abs(float(scale_fn(np.array([0.0]))[0]) - 1.0))


def check_rotation_invariance(rotate):
    """Rotating Q and K (not V) by an orthogonal H leaves attention unchanged."""
    q, k, v = rnd((1, 2, 9, 16), 4), rnd((1, 2, 13, 16), 5), rnd((1, 2, 13, 16), 6)
    q32, k32 = q.astype(np.float32).astype(np.float64), k.astype(np.float32).astype(np.float64)
    worst = 0.0
    for causal in (False, True):
        O0, L0 = oracle.attention(q32, k32, v, 0.25, causal)
        Hq = rotate(q32).astype(np.float64)
        Hk = rotate(k32).astype(np.float64)
        O1, L1 = oracle.attention(Hq, Hk, v, 0.25, causal)
        worst = max(worst, np.abs(O1 - O0).max(), np.abs(L1 - L0).max())
    return float(worst)


def check_block_quantisation(qfn):
    """Each block of 128 rows gets its own scale: its largest code lies in
    (224, 448] (or the block is zero), and every dequantised value is within
    half a step of e4m3 of the input."""
    x = rnd((2, 300, 8), 7).astype(np.float32)
    x[:, 130:256] *= 100.0   # the second block is much larger than the others
    x[1, 256:] = 0.0         # and one block is zero
    deq, s = qfn(x)
    worst = 0.0
    for b in range(2):
        for j in range(3):
            blk = deq[b, j * 128:(j + 1) * 128] / s[b, j]
            top = np.abs(blk).max()
            if np.abs(x[b, j * 128:(j + 1) * 128]).max() == 0:
                worst = max(worst, top, abs(s[b, j] - 1.0))
            elif not (224.0 < top <= 448.0):
                worst = max(worst, 1.0)
    rel = np.abs(deq - x) / np.maximum(np.abs(x), 1e-30)
    worst = max(worst, float(rel[np.abs(x) / np.repeat(s, 128, axis=1)[:, :300, None] >= 2 ** -6].max()) - 2 ** -4)
    return max(worst, 0.0)


def _all_checks(e4m3=fp8.e4m3_round, fwht=fp8.fwht_f32, scale=fp8.pow2_scale, rotate=fp8.rotate_f32,
                qblocks=fp8.quantize_row_blocks):
    return [check_e4m3_vs_torch(e4m3), check_e4m3_codes_fixed(e4m3), check_fwht(fwht), check_scale_rule(scale),
            check_rotation_invariance(rotate), check_block_quantisation(qblocks)]


def test_fp8_oracle_pins():
    errs = _all_checks()
    assert max(errs) < 1e-6, errs


def test_fp8_inputs_shapes_and_identity():
    q, k, v = rnd((1, 2, 200, 128), 8), rnd((1, 1, 300, 128), 9), rnd((1, 1, 300, 128), 10)
    (qd, kd, vd), (sq, sk, sv) = fp8.fp8_inputs(q, k, v)
    assert qd.shape == q.shape and kd.shape == k.shape and vd.shape == v.shape
    assert sq.shape == (1, 2, 2) and sk.shape == (1, 1, 3) and sv.shape == (1, 1)
    O, L = fp8.attention_fp8(q, k, v, 0.1, True)
    O2, L2 = oracle.attention(qd, kd, vd, 0.1, True)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    # the FP8 result stays close to exact attention on the original inputs
    O3, _ = oracle.attention(q, k, v, 0.1, True)
    assert np.abs(O - O3).mean() < 0.05


# planted mistakes ------------------------------------------------------------

def _e4m3_two_mantissa_bits(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    step = np.ldexp(1.0, np.clip(E - 1, -6, 8) - 2)
    return np.sign(x) * np.minimum(np.round(a / step) * step, 448.0)


def _e4m3_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    step = np.ldexp(1.0, np.clip(E - 1, -6, 8) - 3)
    return np.sign(x) * np.minimum(np.floor(a / step) * step, 448.0)


def _e4m3_flush_subnormals(x):
    y = fp8.e4m3_round(x)
    return np.where(np.abs(y) < 2 ** -6, 0.0, y)


def _e4m3_no_saturation(x):
    y = fp8.e4m3_round(np.clip(x, -448, 448))
    return np.where(np.abs(x) > 448, x, y)


def _fwht_wrong_sign(x):
    y = fp8.fwht_f32(x)
    return np.concatenate([y[..., :1], -y[..., 1:]], axis=-1)


def _scale_not_minimal(a):
    return fp8.pow2_scale(a) * 2.0


def _rotate_unnormalised(x):
    return fp8.fwht_f32(x)


def _per_tensor_blocks(x, block=128):
    x = np.asarray(x, dtype=np.float64)
    s = fp8.pow2_scale(np.abs(x).max(axis=(-2, -1)))
    nb = (x.shape[-2] + block - 1) // block
    S = np.repeat(s[..., None], nb, axis=-1)
    return s[..., None, None] * fp8.e4m3_round(x / s[..., None, None]), S


MUTANTS = {
    "two_mantissa_bits": dict(e4m3=_e4m3_two_mantissa_bits),
    "truncating": dict(e4m3=_e4m3_truncate),
    "flush_subnormals": dict(e4m3=_e4m3_flush_subnormals),
    "no_saturation": dict(e4m3=_e4m3_no_saturation),
    "fwht_sign": dict(fwht=_fwht_wrong_sign),
    "scale_not_minimal": dict(scale=_scale_not_minimal),
    "rotation_unnormalised": dict(rotate=_rotate_unnormalised),
    "per_tensor_scale": dict(qblocks=_per_tensor_blocks),
}


@pytest.mark.parametrize("kind", list(MUTANTS))
def test_fp8_pins_catch_planted_mistake(kind):
    with np.errstate(all="ignore"):
        errs = _all_checks(**MUTANTS[kind])
    assert max(errs) > 1e-6, f"FP8 mutant {kind} passed every pin"
