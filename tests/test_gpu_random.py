"""Seeded random shapes through every path, against the oracle: the forward
(every kernel family), the additive mask (with broadcast batch and head
dimensions), the backward and the FP8 forward.  The hand-picked cases in the
other files aim at the edges they name; these mix GQA ratios, batch sizes,
ragged and unequal lengths, causal and not, and head dims at random (fixed
seeds), each at its path's tolerance, on sampled rows where the oracle
would be slow."""
import numpy as np
import pytest

from parity_util import check_case
from test_gpu_bwd import check as check_bwd
from test_gpu_fp8 import run_fp8
from test_gpu_mask import run_case as run_mask_case

pytestmark = pytest.mark.gpu


def _shapes(seed, n, dims, max_n):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        g = int(rng.choice([1, 2, 4, 8]))
        hkv = int(rng.integers(1, 4))
        b = int(rng.integers(1, 4))
        d = int(rng.choice(dims))
        nq = int(rng.integers(1, max_n))
        nkv = nq if rng.random() < 0.5 else int(rng.integers(1, max_n))
        out.append((b, hkv * g, hkv, nq, nkv, d, bool(rng.integers(0, 2)), 5000 + i))
    return out


FWD = _shapes(11, 24, [64, 128, 192, 256, 320, 384, 448, 512, 640, 768, 896, 1024], 1600)
MASKED = _shapes(12, 12, [64, 128, 256, 512, 1024], 900)
BWD = _shapes(13, 10, [64, 128], 700)
FP8 = _shapes(14, 10, [128], 1600)


@pytest.mark.parametrize("case", FWD, ids=[str(c) for c in FWD])
def test_random_forward(case):
    b, hq, hkv, nq, nkv, d, causal, seed = case
    check_case(b, hq, hkv, nq, nkv, d, causal, seed, nrows=min(nq, 64))


@pytest.mark.parametrize("case", MASKED, ids=[str(c) for c in MASKED])
def test_random_masked(case):
    b, hq, hkv, nq, nkv, d, causal, seed = case
    # the stored mask broadcasts over batch and / or heads, or is full
    shape = [(1, 1, nq, nkv), (b, 1, nq, nkv), (1, hq, nq, nkv), (b, hq, nq, nkv)][seed % 4]
    run_mask_case(b, hq, hkv, nq, nkv, d, causal, shape, seed, nrows=min(nq, 64))


@pytest.mark.parametrize("case", BWD, ids=[str(c) for c in BWD])
def test_random_backward(case):
    b, hq, hkv, nq, nkv, d, causal, seed = case
    check_bwd(b, hq, hkv, nq, nkv, d, causal, seed)


@pytest.mark.parametrize("case", FP8, ids=[str(c) for c in FP8])
def test_random_fp8(case):
    b, hq, hkv, nq, nkv, _, causal, seed = case
    run_fp8(b, hq, hkv, nq, nkv, causal, seed, nrows=min(nq, 64))
