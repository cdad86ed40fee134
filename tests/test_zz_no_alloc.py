"""attn_fwd_splitkv_noalloc: the split-KV path for callers that may not
allocate device memory (their own allocator or budget owns the GPU, or an
allocation would be an unbounded stall on a hard-latency path).  It keeps its
partial results in one fixed device array instead of a per-call workspace.

Checked through the C ABI: on two calls in a row, the second one on other
inputs (so that partials left behind by the first call would show), the
output is bit-identical to the allocating entry point, attn_fwd_splitkv with
the same split count (the same kernels run, only the partials live
elsewhere); every kernel family is covered, the per-slice one also through
ATTN_DEBUG_NO_CLUSTER; problems without keys, oversize problems and bad
split counts; and the bounded-wait failure path reaches this entry point
too.  This file sorts last so that a run stopping at the first failure has
run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_attn_gb300 import attn_fwd, attn_fwd_status, attn_set_debug
from exact_attention_attn_gb300.binding import load_library
from exact_attention_attn_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu

ATTN_ERR_SCRATCH = -8
ATTN_ERR_TIMEOUT = -5
ATTN_DEBUG_DROP_V_COPY = 1
ATTN_DEBUG_NO_CLUSTER = 2
SCRATCH_BYTES = 16 << 20


def _noalloc(q, k, v, out, lse, scale, causal, splits):
    lib = load_library()
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    return lib.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                        B, Hq, Hkv, Nq, Nkv, D, ctypes.c_float(scale), int(causal), splits,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    # B, Hq, Hkv, Nq, Nkv, D, causal, splits, debug flags
    (1, 4, 2, 300, 2000, 128, True, 4, 0),          # two-tile kernel
    (2, 2, 2, 129, 1500, 64, False, 3, 0),          # two-tile kernel
    (1, 2, 2, 200, 900, 256, False, 3, 0),          # per-slice kernel (D 192 ... 320)
    (1, 2, 1, 200, 900, 512, True, 5, 0),           # cluster kernel
    (1, 2, 1, 150, 700, 512, False, 3, ATTN_DEBUG_NO_CLUSTER),  # per-slice kernel at D 512
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_noalloc_matches_allocating_entry_point(case):
    B, Hq, Hkv, Nq, Nkv, D, causal, splits, flags = case
    assert splits * B * Hq * Nq * (D + 1) * 4 <= SCRATCH_BYTES
    scale = 1.0 / np.sqrt(D)
    try:
        attn_set_debug(flags, 0)
        for call in range(2):
            q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=splits + D + 101 * call))
            o_ref, l_ref = attn_fwd(q, k, v, scale=scale, causal=causal, kv_splits=splits)
            out = torch.full((B, Hq, Nq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
            lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device="cuda")
            rc = _noalloc(q, k, v, out, lse, scale, causal, splits)
            assert rc == 0, rc
            torch.cuda.synchronize()
            assert attn_fwd_status() == 0
            assert torch.equal(out, o_ref), (call, (out.float() - o_ref.float()).abs().max().item())
            assert torch.equal(lse, l_ref), (call, (lse - l_ref).abs().max().item())
    finally:
        attn_set_debug(0, 0)


def test_noalloc_no_keys():
    q, _, _ = make_qkv(1, 2, 1, 70, 1, 128, 3)
    q = q.cuda()
    k = torch.zeros((1, 1, 0, 128), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        out = torch.full((1, 2, 70, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((1, 2, 70), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(q, k, k, out, lse, 0.1, False, 2) == 0
        torch.cuda.synchronize()
        assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_noalloc_refuses_oversize_and_bad_splits():
    B, Hq, Hkv, Nq, Nkv, D = 1, 8, 8, 4096, 512, 128
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=1))
    out = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    assert 2 * B * Hq * Nq * (D + 1) * 4 > SCRATCH_BYTES
    assert _noalloc(q, k, v, out, lse, 0.1, False, 2) == ATTN_ERR_SCRATCH
    assert _noalloc(q, k, v, out, lse, 0.1, False, 1) == -1
    assert _noalloc(q, k, v, out, lse, 0.1, False, 65) == -1
    assert _noalloc(q, k, v, out, lse, 0.1, 2, 4) == -1        # causal flag not 0/1
    assert _noalloc(q[:, :, :, :96].contiguous(), k, v, out, lse, 0.1, False, 4) == -1  # D not a multiple of 64


def test_noalloc_bounded_wait_reaches_this_entry_point():
    """attn_set_debug's wait bound and fault-free failure injection apply here
    as in attn_fwd: the V producer skips a copy, the wait runs out after 20 ms,
    the status word reports it, and the next call is correct."""
    B, Hq, Hkv, Nq, Nkv, D = 1, 2, 2, 256, 1024, 128
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=3))
    out = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    assert attn_fwd_status() == 0
    try:
        attn_set_debug(ATTN_DEBUG_DROP_V_COPY, 20_000_000)
        assert _noalloc(q, k, v, out, lse, D ** -0.5, False, 2) == 0
        assert attn_fwd_status() == ATTN_ERR_TIMEOUT
    finally:
        attn_set_debug(0, 0)
    assert _noalloc(q, k, v, out, lse, D ** -0.5, False, 2) == 0
    o_ref, l_ref = attn_fwd(q, k, v, kv_splits=2)
    torch.cuda.synchronize()
    assert attn_fwd_status() == 0
    assert torch.equal(out, o_ref) and torch.equal(lse, l_ref)
