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


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def emulated_sampled(q, k, v, do, scale, rows, keys, block=1024):
    """The sampled causal gradients of one head with exactly the kernels'
    documented roundings applied to the float64 quantities: Delta from the
    bf16 O, dS = P (dP - Delta) rounded to bf16 before both products, P
    rounded to bf16 before dV's, dq, dk, dv rounded to bf16 once."""
    N = q.shape[0]
    dq = np.zeros((len(rows), q.shape[1]))
    dk = np.zeros((len(keys), k.shape[1]))
    dv = np.zeros((len(keys), v.shape[1]))
    for r0 in range(0, N, block):
        idx = np.arange(r0, min(N, r0 + block))
        P = oracle.probs_head(q, k, scale, True, idx)
        delta = (do[idx] * _bf16(P @ v)).sum(axis=1)
        dSk = _bf16(P[:, keys] * (do[idx] @ v[keys].T - delta[:, None]))
        dv += _bf16(P[:, keys]).T @ do[idx]
        dk += scale * (dSk.T @ q[idx])
        for s_, r in enumerate(rows):
            if idx[0] <= r <= idx[-1]:
                i = r - r0
                dq[s_] = scale * (_bf16(P[i] * (do[r] @ v.T - delta[i])) @ k)
    return dq, dk, dv


def test_backward_bench_shape_sampled():
    # the backward at the size bench.py --path bwd times (GQA causal B2 Hq32
    # Hkv8 N8192 D128, the same launches), checked on entries the oracle
    # computes without N x N matrices: dq at sampled rows of the four query
    # heads of one (b, kv head) group, dk and dv at sampled keys of that kv
    # head (the group's sum).  Rows of 8192 keys sum 8192 rounded dS terms
    # whose row sums cancel, so the small shapes' fixed bound does not carry
    # over: here each error may be at most twice that of an emulation of the
    # kernels' roundings (emulated_sampled) on the same entries.
    B, Hq, Hkv, N, D = 2, 32, 8, 8192, 128
    (q, k, v, do, scale), (gq, gk, gv) = grads(B, Hq, Hkv, N, N, D, True, seed=81)
    b, kvh, g = 1, 5, Hq // Hkv
    rng = np.random.default_rng(82)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 4095, N - 1], rng.integers(0, N, 10)]))
    keys = np.unique(np.concatenate([[0, 1, 127, 128, 4096, N - 2, N - 1], rng.integers(0, N, 9)]))
    kk, vv = to_f64(k[b, kvh]), to_f64(v[b, kvh])
    ref_k, emu_k = np.zeros((2, len(keys), D)), np.zeros((2, len(keys), D))

    def within(name, got, ref, emu):
        e_got, e_emu = np.abs(got - ref), np.abs(_bf16(emu) - ref)
        tiny = 1e-6 * np.abs(ref).max()
        assert e_got.max() <= 2 * e_emu.max() + tiny, (name, e_got.max(), e_emu.max())
        assert e_got.mean() <= 2 * e_emu.mean() + tiny, (name, e_got.mean(), e_emu.mean())

    for h in range(kvh * g, kvh * g + g):
        qh, doh = to_f64(q[b, h]), to_f64(do[b, h])
        dq_ref, dk_h, dv_h = oracle.attention_backward_sampled(qh, kk, vv, doh, scale, True, rows, keys)
        dq_emu, dke, dve = emulated_sampled(qh, kk, vv, doh, scale, rows, keys)
        ref_k += (dk_h, dv_h)
        emu_k += (dke, dve)
        within(f"dq head {h}", to_f64(gq[b, h])[rows], dq_ref, dq_emu)
    within("dk", to_f64(gk[b, kvh])[keys], ref_k[0], emu_k[0])
    within("dv", to_f64(gv[b, kvh])[keys], ref_k[1], emu_k[1])
