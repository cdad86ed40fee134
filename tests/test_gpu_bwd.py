"""GPU parity of the backward pass (attn_bwd) against the float64 oracle's
gradient, through the C ABI.

The forward O and LSE the backward consumes come from attn_fwd, as a user's
would.  Tolerance (per gradient tensor, relative to the reference's scale):
max|d| <= 1e-2 * max|ref| and mean|d| <= 5e-3 * mean|ref|.  It follows from
the arithmetic: P and dS are rounded to bf16 before their tensor-core
products and dQ, dK, dV are rounded to bf16 once (unit roundoff 2^-9); a
float32 emulation of exactly these roundings lands at <= 4.5e-3 (max) and
2.3e-3 (mean) of the reference scale on these shapes, so the bound keeps a
2x margin while a dropped term, a wrong sign or a missing scale (errors of
order 1) fail it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_attn_gb300 import attn_bwd, attn_fwd, attn_fwd_status
from exact_attention_attn_gb300.workloads import make_qkv, to_f64

pytestmark = pytest.mark.gpu

MAX_REL, MEAN_REL = 1e-2, 5e-3


def grads(B, Hq, Hkv, Nq, Nkv, D, causal, seed, scale=None):
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed)
    do = make_qkv(B, Hq, Hq, Nq, 1, D, seed + 1000)[0]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq_, dk_, dv_ = (t.cuda() for t in (q, k, v))
    o, lse = attn_fwd(dq_, dk_, dv_, scale=scale, causal=causal)
    gq = torch.full_like(dq_, float("nan"))
    gk = torch.full_like(dk_, float("nan"))
    gv = torch.full_like(dv_, float("nan"))
    attn_bwd(dq_, dk_, dv_, o, lse, do.cuda(), scale=scale, causal=causal, dq=gq, dk=gk, dv=gv)
    torch.cuda.synchronize()
    assert attn_fwd_status() == 0
    return (q, k, v, do, scale), (gq.cpu(), gk.cpu(), gv.cpu())


def check(B, Hq, Hkv, Nq, Nkv, D, causal, seed, scale=None):
    (q, k, v, do, scale), got = grads(B, Hq, Hkv, Nq, Nkv, D, causal, seed, scale)
    ref = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = to_f64(g)
        assert not np.isnan(g).any(), f"{name}: unwritten values"
        d = np.abs(g - r)
        rmax, rmean = np.abs(r).max(), np.abs(r).mean()
        if rmax == 0:
            # an exactly zero gradient (one key: dS = dP - Delta vanishes) is
            # met up to the rounding of Delta, which uses the bf16 O
            assert d.max() <= 1e-4, (name, d.max())
            continue
        assert d.max() <= MAX_REL * rmax, (name, d.max() / rmax)
        assert d.mean() <= MEAN_REL * rmean, (name, d.mean() / rmean)
    return got


CASES = [
    # B, Hq, Hkv, Nq, Nkv, D, causal
    (1, 2, 2, 128, 128, 64, False),
    (1, 2, 2, 128, 128, 128, True),
    (2, 4, 2, 300, 333, 64, False),
    (2, 4, 2, 300, 333, 64, True),
    (1, 4, 1, 257, 515, 128, False),
    (1, 8, 2, 384, 384, 128, True),
    (1, 2, 2, 500, 200, 128, True),     # Nq > Nkv: the first rows see no key
    (1, 2, 2, 200, 700, 128, True),     # Nkv > Nq: causal cross
    (1, 2, 1, 1, 300, 128, False),      # one query
    (1, 2, 2, 260, 1, 64, False),       # one key
    (1, 2, 2, 1000, 1000, 128, True),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_backward_matches_oracle(case):
    check(*case, seed=sum(case[:6]))


@pytest.mark.parametrize("scale", [0.0, -0.09, 0.3])
def test_backward_scale_values(scale):
    check(1, 2, 2, 200, 260, 128, True, seed=7, scale=scale)


def test_backward_large_gqa_causal():
    check(1, 4, 1, 2048, 2048, 128, True, seed=12)


def test_backward_deterministic():
    _, a = grads(1, 4, 2, 700, 700, 128, True, seed=5)
    _, b = grads(1, 4, 2, 700, 700, 128, True, seed=5)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_empty_sides():
    # no queries: no key is seen, dk = dv = 0; no keys: dq = 0
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 2, 64, 96, 128, 3))
    o, lse = attn_fwd(q[:, :, :0].contiguous(), k, v)
    dk, dv = torch.full_like(k, 7.0), torch.full_like(v, 7.0)
    dq = torch.empty_like(q[:, :, :0])
    attn_bwd(q[:, :, :0].contiguous(), k, v, o, lse, o.clone(), dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)
    k0 = k[:, :, :0].contiguous()
    o, lse = attn_fwd(q, k0, k0)
    dq = torch.full_like(q, 7.0)
    attn_bwd(q, k0, k0.clone(), o, lse, torch.randn_like(o), dq=dq, dk=torch.empty_like(k0), dv=torch.empty_like(k0))
    torch.cuda.synchronize()
    assert torch.all(dq == 0)


def test_backward_rejects_unsupported_head_dim():
    from exact_attention_attn_gb300.binding import AttnError
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 1, 64, 64, 256, 3))
    o, lse = attn_fwd(q, k, v)
    with pytest.raises(AttnError):
        attn_bwd(q, k, v, o, lse, o.clone())
