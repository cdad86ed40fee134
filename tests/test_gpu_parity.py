"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Tolerances (bf16 O, fp32 LSE): max|dO| <= 2e-2, mean|dO| <= 2e-3,
max|dLSE| <= 1e-3.  The five named workloads run at their full sizes (rows
sampled for the three large ones), plus a sweep over head dims, ragged
lengths, GQA ratios, cross-attention and causal masking, and the edge cases.
"""
import numpy as np
import pytest
import torch

from exact_attention_attn_gb300 import attn_fwd, attn_fwd_status
from exact_attention_attn_gb300.workloads import WORKLOADS, WORKLOAD_ORDER, make_qkv, make_workload_inputs, \
    sample_rows

from parity_util import check_case, compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert attn_fwd_status() == 0


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_named_workload(name):
    w = WORKLOADS[name]
    q, k, v = make_workload_inputs(w)
    o, l = run_gpu(q, k, v, w.scale, w.causal)
    rows = sample_rows(w.Nq, w.sample_rows, w.seed) if w.sample_rows else None
    mx, mean, dl = compare(o, l, q, k, v, w.scale, w.causal, rows)
    print(f"{name}: max|dO|={mx:.3e} mean|dO|={mean:.3e} max|dLSE|={dl:.3e}")
    assert mx <= 2e-2 and mean <= 2e-3 and dl <= 1e-3, (mx, mean, dl)


@pytest.mark.parametrize("D", [64, 128, 192, 256, 320, 384, 448, 512, 576, 640, 704, 768, 832, 896, 960, 1024])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dims(D, causal):
    check_case(1, 2, 1, 200, 200, D, causal, seed=D + causal)


@pytest.mark.parametrize("Nq,Nkv", [(1, 1), (1, 300), (63, 63), (128, 128), (129, 129), (257, 100), (100, 257),
                                    (1000, 1000), (128, 1), (3, 700)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_ragged_lengths(Nq, Nkv, causal, D):
    check_case(2, 2, 2, Nq, Nkv, D, causal, seed=Nq * 7 + Nkv)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (8, 2), (8, 1), (32, 1), (6, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_ratios(Hq, Hkv, causal):
    check_case(2, Hq, Hkv, 300, 300, 128, causal, seed=Hq * 10 + Hkv)


# D = 384 ... 1024 run on clusters of 2 or 4 CTAs that exchange partial scores
# and P; these cases cover single-row and single-key problems, key counts
# below one block, ragged tails, GQA, rows that see no key, and a negative
# and a zero scale.
CLUSTER_CASES = [
    (1, 1, 1, 1, 1, False, None),
    (1, 2, 2, 129, 3, False, None),
    (1, 2, 1, 300, 100, True, None),
    (2, 4, 2, 200, 260, True, None),
    (1, 1, 1, 64, 700, False, None),
    (1, 2, 2, 150, 300, False, -0.04),
    (1, 2, 2, 150, 300, True, 0.0),
]


@pytest.mark.parametrize("D", [384, 448, 512, 640, 768, 896, 1024])
@pytest.mark.parametrize("case", CLUSTER_CASES, ids=[str(c) for c in CLUSTER_CASES])
def test_cluster_splitd_cases(D, case):
    B, Hq, Hkv, Nq, Nkv, causal, scale = case
    check_case(B, Hq, Hkv, Nq, Nkv, D, causal, seed=Nq + Nkv + D, scale=scale)


@pytest.mark.parametrize("D", [384, 448, 512, 640, 768, 1024])
@pytest.mark.parametrize("causal", [False, True])
def test_per_slice_path(D, causal):
    # the path taken where a cluster does not fit: each output slice recomputes S
    from exact_attention_attn_gb300 import attn_set_debug
    attn_set_debug(2)  # ATTN_DEBUG_NO_CLUSTER
    try:
        check_case(1, 2, 1, 200, 330, D, causal, seed=D + 3 * causal)
    finally:
        attn_set_debug(0)


@pytest.mark.parametrize("D", [384, 448, 512, 640, 768, 1024])
def test_cluster_splitd_deterministic(D):
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 2, 300, 500, D, 23))
    o1, l1 = attn_fwd(q, k, v, causal=True)
    o2, l2 = attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# large and lopsided shapes: one query against 128 Ki keys (automatic key
# splits), few queries against long keys on the cluster kernel, a grid of
# 4096 (b, hq) heads, causal cross-attention with Nkv far above Nq, and a
# 32 Ki causal self-attention (rows sampled).
LARGE_CASES = [
    (1, 8, 1, 1, 131072, 128, False, 0),
    (1, 4, 2, 64, 65536, 512, False, 0),
    (256, 16, 16, 128, 128, 64, True, 0),
    (1, 4, 4, 1000, 9000, 128, True, 0),
    (1, 2, 2, 1000, 9000, 768, True, 0),
    (1, 2, 1, 32768, 32768, 128, True, 256),
]


@pytest.mark.parametrize("case", LARGE_CASES, ids=[str(c) for c in LARGE_CASES])
def test_large_shapes(case):
    B, Hq, Hkv, Nq, Nkv, D, causal, nrows = case
    check_case(B, Hq, Hkv, Nq, Nkv, D, causal, seed=Nq + Nkv + D, nrows=nrows)


@pytest.mark.parametrize("scale", [-0.09, 0.0])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128, 192, 256, 320])
def test_nonpositive_scale(D, causal, scale):
    # scale <= 0 runs the kernels' other instantiation (block minimum of the
    # raw scores instead of the maximum); scale 0 gives uniform weights
    check_case(1, 4, 2, 300, 333, D, causal, seed=D + 17 * causal, scale=scale)


@pytest.mark.parametrize("scale", [-0.09, 0.0])
def test_nonpositive_scale_splitkv(scale):
    q, k, v = make_qkv(1, 2, 1, 200, 1500, 128, seed=9)
    out = torch.full((1, 2, 200, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 2, 200), float("nan"), dtype=torch.float32, device="cuda")
    attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=True, out=out, lse=lse, kv_splits=3)
    torch.cuda.synchronize()
    mx, mean, dl = compare(out.cpu(), lse.cpu(), q, k, v, scale, True)
    assert mx <= 2e-2 and mean <= 2e-3 and dl <= 1e-3, (mx, mean, dl)


@pytest.mark.parametrize("D", [128, 512])
def test_large_scores(D):
    # scale 1 on amp-2 inputs: scores of order 2*sqrt(D)*2; stresses the running max
    check_case(1, 2, 2, 256, 600, D, False, seed=5, amp=2.0, scale=1.0)


def test_empty_problems():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 1, 4, 4, 64, 0))
    o, l = attn_fwd(q[:0], k[:0], v[:0])
    assert o.shape == (0, 2, 4, 64)
    o, l = attn_fwd(q[:, :, :0], k, v)
    assert o.shape == (1, 2, 0, 64)
    torch.cuda.synchronize()


def test_no_keys():
    q, _, _ = make_qkv(1, 2, 1, 70, 1, 128, 3)
    k = torch.zeros((1, 1, 0, 128), dtype=torch.bfloat16)
    o, l = run_gpu(q, k, k.clone(), 0.1, False)
    assert torch.all(o == 0) and torch.all(torch.isneginf(l))
    from exact_attention_attn_gb300 import attn_fwd_plan
    plan = attn_fwd_plan(1, 2, 1, 70, 0, 128, False)
    assert plan["path_name"] == "nokeys" and plan["launches"] == 1 and plan["grid"] >= 1


def test_fully_masked_rows():
    # causal with Nq > Nkv: the first Nq - Nkv rows see no key
    check_case(1, 2, 2, 300, 100, 128, True, seed=11)
    q, k, v = make_qkv(1, 1, 1, 300, 100, 64, 12)
    o, l = run_gpu(q, k, v, 0.125, True)
    assert torch.all(o[:, :, :200] == 0) and torch.all(torch.isneginf(l[:, :, :200]))


@pytest.mark.parametrize("Nq", [1, 129, 300])
@pytest.mark.parametrize("D", [64, 128])
def test_no_write_past_output(Nq, D):
    # O and LSE as the leading slice of larger sentinel-filled buffers: the
    # kernel's stores (row-clipped tile copies for O) must stay inside them
    B, Hq, Hkv = 2, 2, 1
    q, k, v = make_qkv(B, Hq, Hkv, Nq, 257, D, seed=Nq + D)
    big_o = torch.full((B + 1, Hq, Nq, D), 7.0, dtype=torch.bfloat16, device="cuda")
    big_l = torch.full((B + 1, Hq, Nq), 7.0, dtype=torch.float32, device="cuda")
    out, lse = big_o[:B], big_l[:B]
    attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=D ** -0.5, causal=True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(big_o[B] == 7.0) and torch.all(big_l[B] == 7.0)
    mx, mean, dl = compare(out.cpu(), lse.cpu(), q, k, v, D ** -0.5, True)
    assert mx <= 2e-2 and mean <= 2e-3 and dl <= 1e-3, (mx, mean, dl)


def test_deterministic():
    q, k, v = (t.cuda() for t in make_qkv(2, 4, 2, 777, 777, 128, 21))
    o1, l1 = attn_fwd(q, k, v, causal=True)
    o2, l2 = attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_stream_argument():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 2, 256, 256, 64, 22))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o1, _ = attn_fwd(q, k, v, stream=s)
    s.synchronize()
    o2, _ = attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


# ---------------------------------------------------------------------------
# split-KV: key ranges merged through their LSE

SPLIT_CASES = [
    (1, 2, 2, 200, 1000, 64, False),
    (1, 2, 1, 300, 700, 128, True),
    (2, 4, 2, 129, 1500, 128, False),
    (1, 2, 2, 256, 300, 128, True),     # fewer key blocks than some split counts: empty ranges
    (1, 1, 1, 100, 900, 192, False),
    (1, 2, 2, 150, 600, 512, True),
    (1, 1, 1, 128, 700, 1024, False),
    (1, 2, 1, 150, 700, 448, True),     # cluster kernel, uneven slices (4 + 3 chunks)
    (1, 2, 2, 200, 600, 640, False),    # uneven slices over four CTAs
    (1, 1, 1, 128, 900, 896, False),
    (1, 2, 1, 300, 100, 128, True),     # causal, Nq > Nkv: fully masked rows in every range
]


@pytest.mark.parametrize("splits", [2, 3, 7])
@pytest.mark.parametrize("case", SPLIT_CASES, ids=[str(c) for c in SPLIT_CASES])
def test_splitkv_forced(case, splits):
    B, Hq, Hkv, Nq, Nkv, D, causal = case
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=splits * 31 + D)
    scale = 1.0 / np.sqrt(D)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    out = torch.full((B, Hq, Nq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device="cuda")
    attn_fwd(dq, dk, dv, scale=scale, causal=causal, out=out, lse=lse, kv_splits=splits)
    torch.cuda.synchronize()
    mx, mean, dl = compare(out.cpu(), lse.cpu(), q, k, v, scale, causal)
    assert mx <= 2e-2 and mean <= 2e-3 and dl <= 1e-3, (mx, mean, dl)


def test_splitkv_auto_for_few_tiles():
    from exact_attention_attn_gb300 import attn_fwd_plan
    B, Hq, Hkv, Nq, Nkv, D = 1, 2, 1, 256, 16384, 128
    plan = attn_fwd_plan(B, Hq, Hkv, Nq, Nkv, D, False)
    assert plan["path_name"] == "tc_splitkv" and plan["kv_splits"] > 1 and plan["launches"] == 2
    assert plan["workspace_bytes"] == plan["kv_splits"] * B * Hq * Nq * (D + 1) * 4
    check_case(B, Hq, Hkv, Nq, Nkv, D, False, seed=77, nrows=64)


def test_splitkv_deterministic():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 2, 300, 2000, 128, 5))
    o1, l1 = attn_fwd(q, k, v, causal=True, kv_splits=5)
    o2, l2 = attn_fwd(q, k, v, causal=True, kv_splits=5)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_workload_plans():
    from exact_attention_attn_gb300 import attn_fwd_plan
    for name in WORKLOAD_ORDER:
        w = WORKLOADS[name]
        plan = attn_fwd_plan(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D, w.causal)
        assert plan["path_name"] in ("tc", "tc_splitkv"), (name, plan)
        assert plan["grid"] > 0
