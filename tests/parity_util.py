"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI binding and the float64 oracle on the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle
from exact_attention_attn_gb300 import attn_fwd
from exact_attention_attn_gb300.workloads import make_qkv, sample_rows, to_f64

# tolerances for bf16 O and fp32 LSE against the float64 oracle
MAX_ABS_O = 2e-2
MEAN_ABS_O = 2e-3
MAX_ABS_LSE = 1e-3


def run_gpu(q, k, v, scale, causal, poison=True):
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    B, Hq, Nq, D = q.shape
    out = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    if poison:  # catch rows the kernel forgets to write
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
    attn_fwd(dq, dk, dv, scale=scale, causal=causal, out=out, lse=lse)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def compare(o_gpu, lse_gpu, q, k, v, scale, causal, rows=None):
    """Return (max|dO|, mean|dO|, max|dLSE|) over the chosen rows (all rows
    when rows is None).  Rows with LSE = -inf on the oracle side must be
    -inf on the GPU side, with O = 0."""
    O_ref, L_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, causal, rows)
    og = to_f64(o_gpu)
    lg = to_f64(lse_gpu)
    if rows is not None:
        og = og[:, :, rows]
        lg = lg[:, :, rows]
    assert not np.isnan(og).any(), "NaN in O (unwritten or poisoned rows)"
    assert not np.isnan(lg).any(), "NaN in LSE"
    dead = np.isneginf(L_ref)
    assert np.array_equal(dead, np.isneginf(lg)), "fully-masked rows disagree"
    d_o = np.abs(og - O_ref)
    d_l = np.abs(lg[~dead] - L_ref[~dead]) if (~dead).any() else np.zeros(1)
    return float(d_o.max(initial=0.0)), float(d_o.mean()) if d_o.size else 0.0, float(d_l.max(initial=0.0))


def check_case(B, Hq, Hkv, Nq, Nkv, D, causal, seed, amp=1.0, scale=None, nrows=0):
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed, amp)
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    o, l = run_gpu(q, k, v, scale, causal)
    rows = sample_rows(Nq, nrows, seed) if nrows else None
    mx, mean, dl = compare(o, l, q, k, v, scale, causal, rows)
    assert mx <= MAX_ABS_O, f"max|dO| {mx}"
    assert mean <= MEAN_ABS_O, f"mean|dO| {mean}"
    assert dl <= MAX_ABS_LSE, f"max|dLSE| {dl}"
    return mx, mean, dl
