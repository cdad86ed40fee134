"""attn_fwd_splitkv_noalloc: the split-KV path for callers that may not
allocate device memory (their own allocator or budget owns the GPU, or an
allocation would be an unbounded stall on a hard-latency path).  It keeps its
partial results in one fixed device array instead of a per-call workspace.

Checked through the C ABI: on two calls in a row (the second reuses the
array the first one left behind) the output matches the allocating entry
point, attn_fwd_splitkv with the same split count, within the parity
tolerances of the other GPU tests; oversize problems are refused.  This file
sorts last so that a run stopping at the first failure has run every other
test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_attn_gb300 import attn_fwd
from exact_attention_attn_gb300.binding import load_library
from exact_attention_attn_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu

ATTN_ERR_SCRATCH = -8
SCRATCH_BYTES = 16 << 20


def _noalloc(q, k, v, out, lse, scale, causal, splits):
    lib = load_library()
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    return lib.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                        B, Hq, Hkv, Nq, Nkv, D, ctypes.c_float(scale), int(causal), splits,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    # B, Hq, Hkv, Nq, Nkv, D, causal, splits
    (1, 4, 2, 300, 2000, 128, True, 4),
    (2, 2, 2, 129, 1500, 64, False, 3),
    (1, 2, 1, 200, 900, 512, True, 5),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_noalloc_matches_allocating_entry_point(case):
    B, Hq, Hkv, Nq, Nkv, D, causal, splits = case
    assert splits * B * Hq * Nq * (D + 1) * 4 <= SCRATCH_BYTES
    scale = 1.0 / np.sqrt(D)
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=splits + D))
    o_ref, l_ref = attn_fwd(q, k, v, scale=scale, causal=causal, kv_splits=splits)
    for call in range(2):
        out = torch.full((B, Hq, Nq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(q, k, v, out, lse, scale, causal, splits)
        assert rc == 0, rc
        torch.cuda.synchronize()
        d_o = (out.float() - o_ref.float()).abs()
        d_l = (lse - l_ref).abs()
        assert not torch.isnan(out).any() and not torch.isnan(lse).any(), f"call {call}: unwritten outputs"
        assert d_o.max().item() <= 2e-2 and d_o.mean().item() <= 2e-3, (call, d_o.max().item())
        assert d_l.max().item() <= 1e-3, (call, d_l.max().item())


def test_noalloc_refuses_oversize_and_bad_splits():
    B, Hq, Hkv, Nq, Nkv, D = 1, 8, 8, 4096, 512, 128
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=1))
    out = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    assert 2 * B * Hq * Nq * (D + 1) * 4 > SCRATCH_BYTES
    assert _noalloc(q, k, v, out, lse, 0.1, False, 2) == ATTN_ERR_SCRATCH
    assert _noalloc(q, k, v, out, lse, 0.1, False, 1) == -1
    assert _noalloc(q, k, v, out, lse, 0.1, False, 65) == -1
