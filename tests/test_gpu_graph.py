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


def _replay_check(capture, direct, refill):
    """Warm up, capture one call into a graph, then twice: write new inputs
    into the captured buffers, replay, and compare with a direct call."""
    capture()  # first-use setup outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = capture()
    for seed in (11, 22):
        refill(seed)
        for t in outs:
            t.fill_(float("nan")) if t.is_floating_point() else None
        g.replay()
        refs = direct()
        torch.cuda.synchronize()
        for a, b in zip(outs, refs):
            assert torch.equal(a, b), seed
    assert attn_fwd_status() == 0


@pytest.mark.parametrize("D", [128, 512])
def test_graph_masked_forward(D):
    from exact_attention_attn_gb300 import attn_fwd
    B, Hq, Hkv, Nq, Nkv = 1, 2, 1, 200, 300
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=5))
    mask = torch.zeros((Nq, 304), dtype=torch.bfloat16, device="cuda")[:, :Nkv]
    out = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")

    def refill(seed):
        q2, k2, v2 = make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=seed)
        q.copy_(q2), k.copy_(k2), v.copy_(v2)
        mask.copy_(torch.randn((Nq, Nkv), generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16))

    _replay_check(lambda: attn_fwd(q, k, v, causal=True, out=out, lse=lse, mask=mask),
                  lambda: attn_fwd(q, k, v, causal=True, mask=mask), refill)


def test_graph_backward():
    from exact_attention_attn_gb300 import attn_bwd
    B, Hq, Hkv, Nq, Nkv, D = 1, 4, 2, 300, 300, 128
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=6))
    o, lse = attn_fwd(q, k, v, causal=True)
    do = torch.randn_like(o)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def refill(seed):
        q2, k2, v2 = make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=seed)
        q.copy_(q2), k.copy_(k2), v.copy_(v2)
        attn_fwd(q, k, v, causal=True, out=o, lse=lse)

    _replay_check(lambda: attn_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv),
                  lambda: attn_bwd(q, k, v, o, lse, do, causal=True), refill)


def test_graph_fp8_forward():
    from exact_attention_attn_gb300 import attn_fp8_quantize, attn_fwd_fp8
    B, Hq, Hkv, Nq, Nkv, D = 1, 4, 2, 300, 333, 128
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=7))
    qz = attn_fp8_quantize(q, k, v)
    out = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    import ctypes
    from exact_attention_attn_gb300.binding import load_library
    lib = load_library()

    def quantize_into():  # quantisation into the same buffers every time
        rc = lib.attn_fp8_quantize(q.data_ptr(), k.data_ptr(), v.data_ptr(), qz["q8"].data_ptr(), qz["k8"].data_ptr(),
                                   qz["vt8"].data_ptr(), qz["sq"].data_ptr(), qz["sk"].data_ptr(), qz["sv"].data_ptr(),
                                   B, Hq, Hkv, Nq, Nkv, D, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0

    def capture():
        quantize_into()
        return attn_fwd_fp8(qz, causal=True, out=out, lse=lse)

    def refill(seed):
        q2, k2, v2 = make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=seed)
        q.copy_(q2), k.copy_(k2), v.copy_(v2)

    _replay_check(capture, lambda: attn_fwd_fp8(attn_fp8_quantize(q, k, v), causal=True), refill)
