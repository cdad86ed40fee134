"""CUDA graph capture of attn_fwd.

attn_fwd keeps nothing between calls that a replay would miss: the tensor
maps travel as kernel parameters and the split-KV workspace is allocated and
freed on the caller's stream.  So one call, after a warm-up call has done the
first-use setup (device facts, kernel attributes, the cluster-fit query),
captures into a CUDA graph as a plain stream capture, and replaying the graph
on new inputs written into the captured buffers gives the same bits as a
direct call on them.  Covers each kernel family: the two-tile kernel, the
per-slice Split-D kernel, the cluster Split-D kernel (even and uneven
slices), and the split-KV path with its workspace allocated inside the graph.
"""
import numpy as np
import pytest
import torch

from exact_attention_attn_gb300 import attn_fwd, attn_fwd_plan, attn_fwd_status
from exact_attention_attn_gb300.workloads import make_qkv

from parity_util import MAX_ABS_LSE, MAX_ABS_O, MEAN_ABS_O, compare

pytestmark = pytest.mark.gpu

# B, Hq, Hkv, Nq, Nkv, D, causal, kv_splits (None = automatic)
GRAPH_CASES = [
    (2, 4, 2, 300, 300, 128, True, None),
    (1, 2, 2, 129, 257, 64, False, None),
    (1, 2, 1, 200, 330, 256, False, None),
    (1, 2, 2, 200, 260, 512, True, None),
    (1, 2, 1, 150, 300, 896, False, None),
    (1, 2, 1, 256, 16384, 128, False, None),
    (1, 2, 2, 150, 600, 1024, True, 3),
    (4, 16, 16, 2048, 2048, 128, True, None),
]


@pytest.mark.parametrize("case", GRAPH_CASES, ids=[str(c) for c in GRAPH_CASES])
def test_graph_replay_matches_direct_call(case):
    B, Hq, Hkv, Nq, Nkv, D, causal, splits = case
    scale = 1.0 / np.sqrt(D)
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=D + Nkv))
    out = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")

    attn_fwd(q, k, v, scale=scale, causal=causal, out=out, lse=lse, kv_splits=splits)  # first-use setup
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        attn_fwd(q, k, v, scale=scale, causal=causal, out=out, lse=lse, kv_splits=splits)

    for seed in (101, 202):
        q2, k2, v2 = make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=seed + D)
        q.copy_(q2)
        k.copy_(k2)
        v.copy_(v2)
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        o_ref, l_ref = attn_fwd(q, k, v, scale=scale, causal=causal, kv_splits=splits)
        torch.cuda.synchronize()
        assert torch.equal(out, o_ref) and torch.equal(lse, l_ref), seed
    assert attn_fwd_status() == 0

    # the replayed result against the oracle (rows sampled on the large case)
    rows = np.array([0, 1, 777, Nq - 1]) if Nq >= 2048 else None
    mx, mean, dl = compare(out.cpu(), lse.cpu(), q2, k2, v2, scale, causal, rows)
    assert mx <= MAX_ABS_O and mean <= MEAN_ABS_O and dl <= MAX_ABS_LSE, (mx, mean, dl)


def test_graph_case_paths():
    # the cases above reach the kernel families they are meant to
    names = {c: attn_fwd_plan(*c[:7])["path_name"] for c in GRAPH_CASES}
    assert names[GRAPH_CASES[5]] == "tc_splitkv"
    assert all(n in ("tc", "tc_splitkv") for n in names.values())
