"""Seeded synthetic inputs for exact attention forward.

This module is the only code shared between the float64 CPU oracle (under
``oracle/``) and the CUDA path.  It draws random numbers and nothing else: it
holds none of the attention arithmetic.

Recipe (the same for every workload): ``torch.Generator().manual_seed(seed)``,
then ``torch.randn`` in float32 in the order Q, K, V, an optional float32
multiply by ``amp`` (0.5 for the large-head-dim workloads), then a cast to
bfloat16 on the CPU.  Layout is (B, H, N, D) with D contiguous, the layout the
FFPA page's usage example gives (page "ffpa-attn 0.2.3 METADATA", section
"Quick Start").  The pages time their kernels on captured model activations
that are not available here; iid Gaussian inputs of the same shapes stand in
for them.

Row sampling for parity checks on large workloads: per (b, h) head,
``numpy.random.default_rng(seed + 1000)`` draws distinct query rows; row 0 and
row Nq-1 are always included.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    D: int
    causal: bool
    seed: int
    amp: float = 1.0
    sample_rows: int = 0  # 0 = every row is checked

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))

    def flops(self) -> float:
        """4*B*Hq*Nq*Nkv*D, halved when causal (the convention the
        throughput figures on these pages use)."""
        f = 4.0 * self.B * self.Hq * self.Nq * self.Nkv * self.D
        return f / 2.0 if self.causal else f

    def hbm_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V once (bf16), write O (bf16)
        and LSE (fp32) once.  The N x N score matrix never touches HBM."""
        q = self.B * self.Hq * self.Nq * self.D * 2
        kv = 2 * self.B * self.Hkv * self.Nkv * self.D * 2
        o = self.B * self.Hq * self.Nq * self.D * 2
        lse = self.B * self.Hq * self.Nq * 4
        return q + kv + o + lse

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "Hq": self.Hq, "Hkv": self.Hkv,
                "Nq": self.Nq, "Nkv": self.Nkv, "D": self.D, "causal": self.causal,
                "seed": self.seed, "amp": self.amp, "scale": self.scale}


# The five workloads: a small self-attention case the oracle checks in full,
# two causal D=128 cases (plain and GQA), and two large-head-dim cases.
WORKLOADS = {
    "selfattn_b1_h1_n128_d64": Workload("selfattn_b1_h1_n128_d64", 1, 1, 1, 128, 128, 64, False, 0),
    "causal_b4_h16_n2048_d128": Workload("causal_b4_h16_n2048_d128", 4, 16, 16, 2048, 2048, 128, True, 1),
    "gqa_causal_b2_hq32_hkv8_n8192_d128": Workload("gqa_causal_b2_hq32_hkv8_n8192_d128", 2, 32, 8, 8192, 8192, 128, True, 2,
                                                   sample_rows=256),
    "splitd_b1_h8_n4096_d512": Workload("splitd_b1_h8_n4096_d512", 1, 8, 8, 4096, 4096, 512, False, 3, amp=0.5,
                                        sample_rows=256),
    "cross_splitd_b1_h4_nq1024_nkv8192_d1024": Workload("cross_splitd_b1_h4_nq1024_nkv8192_d1024", 1, 4, 4, 1024, 8192,
                                                        1024, False, 4, amp=0.5, sample_rows=256),
}
WORKLOAD_ORDER = list(WORKLOADS)
# The bench's default: the largest workload (GQA causal N8192, 1.1 TFLOP per call)
BENCH_WORKLOAD = "gqa_causal_b2_hq32_hkv8_n8192_d128"


def make_qkv(B: int, Hq: int, Hkv: int, Nq: int, Nkv: int, D: int, seed: int, amp: float = 1.0):
    """Return bf16 CPU tensors q [B,Hq,Nq,D], k and v [B,Hkv,Nkv,D]."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Hq, Nq, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, Hkv, Nkv, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, Hkv, Nkv, D), generator=g, dtype=torch.float32)
    if amp != 1.0:
        q.mul_(amp)
        k.mul_(amp)
        v.mul_(amp)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def make_workload_inputs(w: Workload):
    return make_qkv(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D, w.seed, w.amp)


def sample_rows(Nq: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct query-row indices; always holds 0 and Nq-1."""
    if count <= 0 or count >= Nq:
        return np.arange(Nq)
    rng = np.random.default_rng(seed + 1000)
    inner = rng.choice(np.arange(1, Nq - 1), size=count - 2, replace=False)
    return np.sort(np.concatenate([[0, Nq - 1], inner]).astype(np.int64))


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact upcast of a bf16 (or any float) tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
