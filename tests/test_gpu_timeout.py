"""Failure path without a GPU fault: a device-side wait that runs out.

attn_set_debug(ATTN_DEBUG_DROP_V_COPY, short limit) makes the V producer of
the head-dim-128 kernel leave one shared-memory slot empty; the MMA thread's
bounded wait for it runs out, the kernel records ATTN_ERR_TIMEOUT and every
role of the CTA stops, drains its copies and MMAs and frees tensor memory.
The host reads the status; the context stays usable for the next call.
"""
import numpy as np
import pytest
import torch

from exact_attention_attn_gb300 import attn_fwd, attn_fwd_status, attn_set_debug
from exact_attention_attn_gb300.workloads import make_qkv

from parity_util import compare

pytestmark = pytest.mark.gpu

ATTN_ERR_TIMEOUT = -5


def test_bounded_wait_runs_out_and_context_survives():
    q, k, v = make_qkv(1, 2, 2, 256, 1024, 128, seed=3)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    assert attn_fwd_status() == 0
    try:
        attn_set_debug(1, 20_000_000)  # 20 ms bound on every device-side wait
        attn_fwd(dq, dk, dv)
        assert attn_fwd_status() == ATTN_ERR_TIMEOUT
        assert attn_fwd_status() == 0  # read clears
    finally:
        attn_set_debug(0, 0)
    # the same context computes correctly afterwards
    o, l = attn_fwd(dq, dk, dv)
    torch.cuda.synchronize()
    assert attn_fwd_status() == 0
    mx, mean, dl = compare(o.cpu(), l.cpu(), q, k, v, 1.0 / np.sqrt(128), False)
    assert mx <= 2e-2 and mean <= 2e-3 and dl <= 1e-3
