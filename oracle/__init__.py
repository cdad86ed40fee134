"""Float64 CPU oracle for exact attention: forward, additive mask, backward, FP8 inputs (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path never does.
"""
from .attention import (attention, attention_backward, attention_backward_head,  # noqa: F401
                        attention_backward_sampled,
                        attention_bruteforce, attention_head,
                        attention_online_head, causal_visible, kv_head_of, lse_merge,
                        probs_head, scores_head)
from . import fp8  # noqa: F401,E402
