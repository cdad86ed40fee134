"""GPU parity of the FP8 path (attn_fp8_quantize, attn_fwd_fp8) against the
FP8 oracle (oracle/fp8.py), through the C ABI.

Quantisation decides integer codes, so both sides take it in float32 in the
same butterfly order and the codes and scales must match exactly.  The
attention output is compared with exact (float64) attention on the
dequantised inputs; the kernel also rounds P to e4m3 (as 2^2 p), which the
tolerance covers: max|dO| <= 0.1, mean|dO| <= 1e-2, max|dLSE| <= 1e-3.
Derivation: e4m3 keeps 3 mantissa bits, so each probability carries a
relative error of up to 2^-4; an emulation of exactly that rounding on the
oracle's side gives max|dO| up to 5.1e-2 (rows that see 8 keys) and
mean|dO| up to 5.7e-3 on these shapes, so the bound keeps a 2x margin.
LSE does not go through the rounded P (l sums the fp32 probabilities).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from exact_attention_attn_gb300 import attn_fp8_quantize, attn_fwd_fp8, attn_fwd_status
from exact_attention_attn_gb300.workloads import make_qkv, sample_rows, to_f64

pytestmark = pytest.mark.gpu

MAX_O, MEAN_O, MAX_LSE = 1e-1, 1e-2, 1e-3


def codes_to_f64(u8):
    return u8.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.mark.parametrize("shape", [(1, 2, 1, 300, 333), (2, 1, 1, 128, 1), (1, 3, 3, 1, 257)])
def test_quantisation_matches_oracle_bit_for_bit(shape):
    B, Hq, Hkv, Nq, Nkv = shape
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nkv, 128, seed=Nq + Nkv, amp=3.0)
    # a few large values so that blocks get different scales
    q[..., :1, :7] *= 40
    k[..., -1:, 5:9] *= 25
    qz = attn_fp8_quantize(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    (qd, kd, vd), (sq, sk, sv) = fp8.fp8_inputs(to_f64(q), to_f64(k), to_f64(v))
    assert np.array_equal(qz["sq"].cpu().numpy(), sq) and np.array_equal(qz["sk"].cpu().numpy(), sk)
    assert np.array_equal(qz["sv"].cpu().numpy(), sv)
    nqb = sq.shape[-1]
    q_dev = codes_to_f64(qz["q8"]) * np.repeat(sq, 128, axis=-1)[..., :Nq, None]
    k_dev = codes_to_f64(qz["k8"]) * np.repeat(sk, 128, axis=-1)[..., :Nkv, None]
    assert np.array_equal(q_dev, qd), np.abs(q_dev - qd).max()
    assert np.array_equal(k_dev, kd), np.abs(k_dev - kd).max()
    vt = codes_to_f64(qz["vt8"])                      # [B, Hkv, 128, nkv_pad]
    assert np.all(vt[..., Nkv:] == 0)
    v_dev = np.swapaxes(vt[..., :Nkv], -1, -2) * sv[..., None, None]
    assert np.array_equal(v_dev, vd), np.abs(v_dev - vd).max()
    assert nqb == (Nq + 127) // 128


def test_quantisation_many_units_bit_for_bit():
    # more (head, 128-row block) units than the rotation kernel keeps resident
    # (three CTAs per SM), so each CTA walks several units through both of its
    # buffers; ragged last blocks on both sides
    B, Hq, Hkv, Nq, Nkv = 1, 8, 8, 8192 + 37, 8192 - 5
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nkv, 128, seed=11, amp=2.0)
    q[:, :, ::97, :3] *= 30
    qz = attn_fp8_quantize(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    (qd, kd, _), (sq, sk, _) = fp8.fp8_inputs(to_f64(q), to_f64(k), to_f64(v))
    assert np.array_equal(qz["sq"].cpu().numpy(), sq) and np.array_equal(qz["sk"].cpu().numpy(), sk)
    q_dev = codes_to_f64(qz["q8"]) * np.repeat(sq, 128, axis=-1)[..., :Nq, None]
    k_dev = codes_to_f64(qz["k8"]) * np.repeat(sk, 128, axis=-1)[..., :Nkv, None]
    assert np.array_equal(q_dev, qd) and np.array_equal(k_dev, kd)


def run_fp8(B, Hq, Hkv, Nq, Nkv, causal, seed, nrows=0):
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nkv, 128, seed)
    scale = 1.0 / math.sqrt(128)
    qz = attn_fp8_quantize(q.cuda(), k.cuda(), v.cuda())
    out = torch.full((B, Hq, Nq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device="cuda")
    attn_fwd_fp8(qz, scale=scale, causal=causal, out=out, lse=lse)
    torch.cuda.synchronize()
    assert attn_fwd_status() == 0
    rows = sample_rows(Nq, nrows, seed) if nrows else None
    O_ref, L_ref = fp8.attention_fp8(to_f64(q), to_f64(k), to_f64(v), scale, causal, rows)
    og, lg = to_f64(out.cpu()), to_f64(lse.cpu())
    if rows is not None:
        og, lg = og[:, :, rows], lg[:, :, rows]
    assert not np.isnan(og).any() and not np.isnan(lg).any()
    dead = np.isneginf(L_ref)
    assert np.array_equal(dead, np.isneginf(lg)) and np.all(og[dead] == 0)
    d = np.abs(og - O_ref)
    dl = np.abs(lg[~dead] - L_ref[~dead]) if (~dead).any() else np.zeros(1)
    assert d.max() <= MAX_O and d.mean() <= MEAN_O, (d.max(), d.mean())
    assert dl.max() <= MAX_LSE, dl.max()
    # and the FP8 result stays close to exact attention on the bf16 inputs
    O_x, _ = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, causal, rows)
    assert np.abs(og - O_x).mean() <= 2e-2
    return d.max(), d.mean(), dl.max()


CASES = [
    # B, Hq, Hkv, Nq, Nkv, causal
    (1, 2, 2, 128, 128, False),
    (1, 2, 2, 128, 128, True),
    (2, 4, 2, 300, 333, False),
    (2, 4, 2, 300, 333, True),
    (1, 4, 1, 257, 1000, False),
    (1, 2, 2, 500, 200, True),      # rows with no key
    (1, 2, 2, 200, 700, True),      # causal cross
    (1, 2, 1, 1, 300, False),
    (1, 2, 2, 260, 8, False),
    (1, 8, 2, 1024, 1024, True),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_fp8_forward_matches_oracle(case):
    run_fp8(*case, seed=sum(case[:5]))


def test_fp8_forward_gqa_causal_n8192_sampled():
    run_fp8(2, 32, 8, 8192, 8192, True, seed=2, nrows=64)


def test_fp8_deterministic():
    q, k, v = (t.cuda() for t in make_qkv(1, 4, 2, 700, 700, 128, 9))
    qz = attn_fp8_quantize(q, k, v)
    o1, l1 = attn_fwd_fp8(qz, causal=True)
    o2, l2 = attn_fwd_fp8(qz, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fp8_rejects_bad_arguments():
    from exact_attention_attn_gb300.binding import AttnError
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 1, 64, 64, 128, 3))
    qz = attn_fp8_quantize(q, k, v)
    with pytest.raises(AttnError):
        attn_fwd_fp8(qz, scale=-0.1)
    q2, k2, v2 = (t.cuda() for t in make_qkv(1, 1, 1, 64, 64, 64, 3))
    with pytest.raises(AttnError):
        attn_fp8_quantize(q2, k2, v2)
