"""Host-side checks of the seeded input generator and the workload table."""
import numpy as np
import torch

from exact_attention_attn_gb300 import workloads as W


def test_inputs_are_seeded_and_bf16():
    a = W.make_qkv(1, 2, 1, 5, 7, 64, seed=3)
    b = W.make_qkv(1, 2, 1, 5, 7, 64, seed=3)
    c = W.make_qkv(1, 2, 1, 5, 7, 64, seed=4)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    assert not torch.equal(a[0], c[0])
    assert a[0].shape == (1, 2, 5, 64) and a[1].shape == (1, 1, 7, 64)


def test_amp_scales_before_rounding():
    full = W.make_qkv(1, 1, 1, 4, 4, 64, seed=9)
    half = W.make_qkv(1, 1, 1, 4, 4, 64, seed=9, amp=0.5)
    # multiplying by 0.5 is exact in float32 and commutes with the bf16 cast
    for x, y in zip(full, half):
        assert torch.equal(x.float() * 0.5, y.float())


def test_sample_rows():
    r = W.sample_rows(8192, 256, 2)
    assert len(r) == 256 and r[0] == 0 and r[-1] == 8191
    assert len(np.unique(r)) == 256 and np.all(np.diff(r) > 0)
    assert np.array_equal(r, W.sample_rows(8192, 256, 2))
    assert np.array_equal(W.sample_rows(100, 0, 1), np.arange(100))


def test_flop_counts():
    # 4*B*Hq*Nq*Nkv*D, halved when causal
    got = [W.WORKLOADS[n].flops() for n in W.WORKLOAD_ORDER]
    assert got == [4194304.0, 68719476736.0, 1099511627776.0, 274877906944.0, 137438953472.0]
    assert W.WORKLOADS[W.BENCH_WORKLOAD].causal
