"""GPU parity of the additive mask (attn_fwd_masked) against the float64
oracle, through the C ABI, on every kernel family.

The mask is the FFPA README's "Causal/Mask" feature read as SDPA's additive
float mask: added to the scaled scores before the row softmax, -inf hides a
key.  The oracle takes the same bf16 mask values, upcast exactly.  Cases:
the two-tile kernel (D 64, 128), the per-slice Split-D kernel (D 256, and
D 512 with ATTN_DEBUG_NO_CLUSTER), the cluster Split-D kernel (D 384, 512,
448 with uneven slices, 1024); causal and not; full, per-batch, broadcast
and key-padding masks; GQA; ragged lengths; rows and whole heads hidden;
automatic key splits; and a mask of zeros giving attn_fwd's bits.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_attn_gb300 import attn_fwd, attn_fwd_plan, attn_fwd_status, attn_set_debug
from exact_attention_attn_gb300.workloads import make_qkv, sample_rows, to_f64

from parity_util import MAX_ABS_LSE, MAX_ABS_O, MEAN_ABS_O

pytestmark = pytest.mark.gpu

ATTN_DEBUG_NO_CLUSTER = 2


def make_mask(shape, seed, p_hide=0.15, amp=2.0, pad_to=8):
    """bf16 mask of `shape` (last dim = Nkv), N(0, amp^2) values with a share
    p_hide of -inf, stored with the key dimension padded to a multiple of 8
    (the padding holds NaN: it must never be read)."""
    g = torch.Generator().manual_seed(seed)
    vals = torch.randn(shape, generator=g) * amp
    vals[torch.rand(shape, generator=g) < p_hide] = float("-inf")
    nkv = shape[-1]
    padded = (nkv + pad_to - 1) // pad_to * pad_to
    store = torch.full(tuple(shape[:-1]) + (padded,), float("nan"), dtype=torch.bfloat16)
    store[..., :nkv] = vals.to(torch.bfloat16)
    return store, store[..., :nkv]


def run_case(B, Hq, Hkv, Nq, Nkv, D, causal, mask_shape, seed, nrows=0, amp=1.0, p_hide=0.15):
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nkv, D, seed, amp)
    store, mask = make_mask(mask_shape, seed + 7, p_hide=p_hide)
    scale = 1.0 / np.sqrt(D)
    dm = store.cuda()[..., :Nkv]
    out = torch.full((B, Hq, Nq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device="cuda")
    attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal, out=out, lse=lse, mask=dm)
    torch.cuda.synchronize()
    assert attn_fwd_status() == 0
    rows = sample_rows(Nq, nrows, seed) if nrows else None
    M = to_f64(mask)
    O_ref, L_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, causal, rows, mask=M)
    og, lg = to_f64(out.cpu()), to_f64(lse.cpu())
    if rows is not None:
        og, lg = og[:, :, rows], lg[:, :, rows]
    assert not np.isnan(og).any() and not np.isnan(lg).any(), "unwritten or NaN outputs"
    dead = np.isneginf(L_ref)
    assert np.array_equal(dead, np.isneginf(lg)), "rows with no visible key disagree"
    assert np.all(og[dead] == 0)
    d_o = np.abs(og - O_ref)
    d_l = np.abs(lg[~dead] - L_ref[~dead]) if (~dead).any() else np.zeros(1)
    assert d_o.max() <= MAX_ABS_O and d_o.mean() <= MEAN_ABS_O, (d_o.max(), d_o.mean())
    assert d_l.max() <= MAX_ABS_LSE, d_l.max()
    return out, lse


FAMILY_CASES = [
    # B, Hq, Hkv, Nq, Nkv, D, causal, mask shape (built from the sizes)
    (2, 4, 2, 300, 333, 64, False, "full"),
    (2, 4, 2, 300, 333, 64, True, "full"),
    (1, 4, 1, 257, 515, 128, False, "heads1"),
    (2, 2, 2, 384, 384, 128, True, "full"),
    (1, 2, 2, 200, 301, 256, False, "full"),
    (1, 2, 2, 200, 301, 256, True, "batch1"),
    (1, 2, 1, 130, 260, 384, True, "full"),
    (1, 2, 2, 129, 300, 448, False, "full"),
    (1, 2, 2, 256, 389, 512, False, "keypad"),
    (1, 2, 2, 256, 389, 512, True, "full"),
    (1, 2, 1, 140, 270, 1024, False, "full"),
]


def _shape(kind, B, Hq, Nq, Nkv):
    return {"full": (B, Hq, Nq, Nkv), "heads1": (B, 1, Nq, Nkv), "batch1": (1, Hq, Nq, Nkv),
            "keypad": (B, 1, 1, Nkv)}[kind]


@pytest.mark.parametrize("case", FAMILY_CASES, ids=[str(c) for c in FAMILY_CASES])
def test_mask_kernel_families(case):
    B, Hq, Hkv, Nq, Nkv, D, causal, kind = case
    run_case(B, Hq, Hkv, Nq, Nkv, D, causal, _shape(kind, B, Hq, Nq, Nkv), seed=D + Nq)


@pytest.mark.parametrize("D", [512, 1024])
def test_mask_per_slice_path(D):
    try:
        attn_set_debug(ATTN_DEBUG_NO_CLUSTER, 0)
        run_case(1, 2, 2, 150, 300, D, True, (1, 2, 150, 300), seed=D + 3)
    finally:
        attn_set_debug(0, 0)


@pytest.mark.parametrize("D", [128, 256, 512])
def test_mask_hides_rows_and_heads(D):
    """Rows whose every key is hidden (and a whole head) give O = 0, LSE = -inf."""
    B, Hq, Nq, Nkv = 1, 2, 160, 200
    q, k, v = make_qkv(B, Hq, Hq, Nq, Nkv, D, seed=D)
    store, mask = make_mask((B, Hq, Nq, Nkv), D + 1, p_hide=0.3)
    store[:, :, 5] = float("-inf")          # one row hidden in both heads
    store[:, :, 130:140] = float("-inf")    # rows in the second tile
    store[:, 1, 150:] = float("-inf")
    out, lse = attn_fwd(q.cuda(), k.cuda(), v.cuda(), mask=store.cuda()[..., :Nkv])
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), 1 / np.sqrt(D), False, mask=to_f64(mask))
    lg = to_f64(lse.cpu())
    assert np.array_equal(np.isneginf(lg), np.isneginf(L_ref))
    assert np.isneginf(lg[:, :, 5]).all() and torch.all(out[:, :, 5] == 0)
    live = ~np.isneginf(L_ref)
    assert np.abs(to_f64(out.cpu()) - O_ref).max() <= MAX_ABS_O
    assert np.abs(lg[live] - L_ref[live]).max() <= MAX_ABS_LSE


@pytest.mark.parametrize("D", [128, 512])
def test_mask_with_automatic_key_splits(D):
    B, Hq, Hkv, Nq, Nkv = 1, 2, 1, 256, 9000
    plan = attn_fwd_plan(B, Hq, Hkv, Nq, Nkv, D, False)
    assert plan["kv_splits"] > 1
    run_case(B, Hq, Hkv, Nq, Nkv, D, False, (B, Hq, Nq, Nkv), seed=D + 11, nrows=64)


@pytest.mark.parametrize("D", [64, 128, 256, 512, 1024])
def test_zero_mask_matches_unmasked(D):
    """A mask of zeros adds exactly 0 to every score.  The Split-D kernels
    (D >= 192) scale a score the same way with and without a mask (one
    rounding of s * scale*log2e, then y - m), so O and LSE match attn_fwd's
    bit for bit; the two-tile kernel's unmasked path fuses the subtraction
    of the running max into the same rounding, so there they agree within
    the parity tolerances."""
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 2, 200, 300, D, seed=D + 5))
    zero = torch.zeros((1, 1, 200, 304), dtype=torch.bfloat16, device="cuda")[..., :300]
    for causal in (False, True):
        o0, l0 = attn_fwd(q, k, v, causal=causal)
        o1, l1 = attn_fwd(q, k, v, causal=causal, mask=zero)
        torch.cuda.synchronize()
        if D >= 192:
            assert torch.equal(l0, l1) and torch.equal(o0, o1), (D, causal)
        else:
            assert (o0.float() - o1.float()).abs().max().item() <= MAX_ABS_O
            assert (l0 - l1).abs().max().item() <= MAX_ABS_LSE


def test_mask_large_workload_sampled():
    # the causal GQA N2048 D128 shape with one mask shared by every head
    run_case(2, 8, 2, 2048, 2048, 128, True, (1, 1, 2048, 2048), seed=31, nrows=128)


def test_mask_bench_shape_sampled():
    # the size bench.py --path mask times: GQA causal B2 Hq32 Hkv8 N8192 D128,
    # one [Nq, Nkv] mask shared by every head, 64 sampled rows per head
    run_case(2, 32, 8, 8192, 8192, 128, True, (1, 1, 8192, 8192), seed=41, nrows=64)
