"""attn_fwd_host (host buffers, copies overlapped with the kernels by chunks of
(b, kv head) groups) against attn_fwd on the device: bit-identical O and LSE,
and the oracle's tolerances on one case.  These problems are small enough to
go in one chunk by size; ATTN_DEBUG_HOST_CHUNKS makes the same calls take one
chunk per group, so both forms are checked."""
import pytest
import torch

from exact_attention_attn_gb300 import attn_fwd, attn_fwd_host, attn_fwd_status, attn_set_debug
from exact_attention_attn_gb300.workloads import make_qkv

from parity_util import compare

pytestmark = pytest.mark.gpu

ATTN_DEBUG_HOST_CHUNKS = 4

CASES = [
    # B, Hq, Hkv, Nq, Nkv, D, causal
    (2, 8, 2, 300, 300, 128, True),     # GQA; chunked: four chunks of one group
    (1, 3, 3, 129, 200, 64, False),     # chunked: three chunks; LSE rows of 129 floats per head
    (2, 10, 10, 200, 200, 64, True),    # chunked: twenty groups in eight chunks of two or three
    (2, 4, 4, 1000, 5000, 128, False),  # few row tiles: the key split count of the whole problem
    (1, 2, 1, 100, 0, 128, False),      # no keys
    (1, 4, 4, 256, 300, 512, True),     # Split-D kernel
    (3, 2, 1, 1, 77, 64, True),         # single query row
]


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert attn_fwd_status() == 0


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("chunked", [False, True])
def test_host_matches_device(case, pinned, chunked):
    B, Hq, Hkv, Nq, Nkv, D, causal = case
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed=Nq + Nkv + D)
    scale = D ** -0.5
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    attn_set_debug(ATTN_DEBUG_HOST_CHUNKS if chunked else 0, 0)
    try:
        o_h, l_h = attn_fwd_host(q, k, v, scale=scale, causal=causal)
    finally:
        attn_set_debug(0, 0)
    o_d, l_d = attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert o_h.device.type == "cpu" and l_h.device.type == "cpu"
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(l_h, l_d.cpu())


def test_host_parity_with_oracle():
    q, k, v = make_qkv(2, 4, 2, 333, 333, 128, seed=5)
    o, l = attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), scale=128 ** -0.5, causal=True)
    mx, mean, dl = compare(o, l, q, k, v, 128 ** -0.5, True)
    assert mx <= 2e-2 and mean <= 2e-3 and dl <= 1e-3, (mx, mean, dl)


def test_host_outputs_in_place():
    q, k, v = (t.pin_memory() for t in make_qkv(1, 2, 2, 200, 200, 64, seed=9))
    out = torch.full((1, 2, 200, 64), float("nan"), dtype=torch.bfloat16).pin_memory()
    lse = torch.full((1, 2, 200), float("nan"), dtype=torch.float32).pin_memory()
    o, l = attn_fwd_host(q, k, v, causal=False, out=out, lse=lse)
    assert o.data_ptr() == out.data_ptr() and l.data_ptr() == lse.data_ptr()
    assert not torch.isnan(out.float()).any() and not torch.isnan(lse).any()


def test_shutdown_gives_back_pools_and_library_stays_usable():
    # a split-KV call (few row tiles, many keys) and a host-buffer call fill
    # the library's two pools; attn_shutdown trims them, and the same calls
    # afterwards give the same bits
    from exact_attention_attn_gb300 import attn_fwd_plan, attn_shutdown
    q, k, v = make_qkv(1, 2, 2, 64, 16384, 128, seed=21)
    assert attn_fwd_plan(1, 2, 2, 64, 16384, 128, False)["kv_splits"] > 1
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o1, l1 = attn_fwd(q.cuda(), k.cuda(), v.cuda())
    oh1, lh1 = attn_fwd_host(qp, kp, vp)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    attn_shutdown()
    assert torch.cuda.mem_get_info()[0] >= free_before
    o2, l2 = attn_fwd(q.cuda(), k.cuda(), v.cuda())
    oh2, lh2 = attn_fwd_host(qp, kp, vp)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(oh1, oh2) and torch.equal(lh1, lh2)
    assert torch.equal(oh1, o1.cpu())
