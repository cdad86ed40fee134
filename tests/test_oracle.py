"""Pins for the float64 oracle: checks against things other than itself.

Each ``check_*`` helper takes an attention function with the oracle's
signature ``fn(q, k, v, scale, causal) -> (O, LSE)`` and returns the largest
deviation from what the mathematics fixes.  The tests run every helper on the
real oracle (all must pass) and on deliberately broken copies of it (each
broken copy must be caught by at least one helper), so that a plausible slip
in the oracle -- a dropped scale, a transposed operand, a wrong GQA head, a
sign error in the rescale, a wrong causal offset -- cannot go unnoticed.

Sources for what is fixed (by page title and section):
* "FlashAttention v1/v2/v3/v4" (lo0.es), "El truco que hizo posible todo:
  online softmax": softmax definition; online form exact.
* "FlashAttention: Fast and Memory-Efficient Exact Attention with IO-Awareness":
  exact attention, no approximation.
* "ffpa-attn 0.2.3" README feature table: GQA/MQA, cross, causal.
* "ZYFA: FP8 FlashAttention Kernels for AMD MI355X", "The details that make it
  production-grade": results over different key ranges merge via the LSE.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import importlib
oracle_mod = importlib.import_module("oracle.attention")

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed, amp=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * amp


# ---------------------------------------------------------------------------
# check helpers: each returns the max deviation (0 is perfect)

def check_bruteforce(fn):
    worst = 0.0
    cases = [(1, 1, 1, 5, 5, 4), (2, 4, 2, 3, 7, 5), (1, 3, 1, 8, 3, 2), (1, 2, 2, 6, 6, 3)]
    for n, (B, Hq, Hkv, Nq, Nkv, D) in enumerate(cases):
        q = rnd((B, Hq, Nq, D), 10 + n)
        k = rnd((B, Hkv, Nkv, D), 20 + n)
        v = rnd((B, Hkv, Nkv, D), 30 + n)
        for causal in (False, True):
            O, L = fn(q, k, v, 0.7, causal)
            Ob, Lb = oracle.attention_bruteforce(q, k, v, 0.7, causal)
            fin = np.isfinite(Lb)
            if not np.array_equal(fin, np.isfinite(L)):
                return math.inf
            worst = max(worst, np.abs(O - Ob).max(), np.abs(L[fin] - Lb[fin]).max(initial=0.0))
    return worst


def _sdpa(q, k, v, scale, causal):
    """torch float64 SDPA with an explicit bottom-right causal mask, plus the
    log-sum-exp of the masked scaled scores from torch.logsumexp."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    Hq, Hkv = tq.shape[1], tk.shape[1]
    tk_r = tk.repeat_interleave(Hq // Hkv, dim=1)
    tv_r = tv.repeat_interleave(Hq // Hkv, dim=1)
    Nq, Nkv = tq.shape[2], tk.shape[2]
    mask = None
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nkv)[None, :]
        mask = j <= i + (Nkv - Nq)
    O = torch.nn.functional.scaled_dot_product_attention(tq, tk_r, tv_r, attn_mask=mask, scale=scale)
    s = torch.matmul(tq, tk_r.transpose(-1, -2)) * scale
    if mask is not None:
        s = s.masked_fill(~mask, -math.inf)
    return O.numpy(), torch.logsumexp(s, dim=-1).numpy()


def check_torch_sdpa(fn):
    worst = 0.0
    cases = [(2, 4, 4, 33, 33, 16, False), (2, 4, 4, 33, 33, 16, True), (1, 8, 2, 17, 17, 8, True),
             (1, 8, 1, 9, 21, 8, False), (1, 2, 2, 10, 40, 8, False), (1, 2, 2, 10, 40, 8, True),
             (1, 1, 1, 70, 70, 64, True)]
    for n, (B, Hq, Hkv, Nq, Nkv, D, causal) in enumerate(cases):
        q = rnd((B, Hq, Nq, D), 40 + n)
        k = rnd((B, Hkv, Nkv, D), 50 + n)
        v = rnd((B, Hkv, Nkv, D), 60 + n)
        scale = 1.0 / math.sqrt(D)
        O, L = fn(q, k, v, scale, causal)
        Ot, Lt = _sdpa(q, k, v, scale, causal)
        worst = max(worst, np.abs(O - Ot).max(), np.abs(L - Lt).max())
    # the stock is_causal flag (top-left) agrees with bottom-right when Nq == Nkv
    q, k, v = rnd((1, 2, 12, 8), 1), rnd((1, 2, 12, 8), 2), rnd((1, 2, 12, 8), 3)
    Ot = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=True, scale=0.3).numpy()
    worst = max(worst, np.abs(fn(q, k, v, 0.3, True)[0] - Ot).max())
    return worst


def check_identical_keys(fn):
    """All keys equal to one vector kappa: every visible score of row i equals
    s_i = scale * q_i . kappa, so O_i is the plain mean of V and
    LSE_i = s_i + ln Nkv."""
    B, Hq, Hkv, Nq, Nkv, D = 1, 4, 2, 6, 11, 8
    q = rnd((B, Hq, Nq, D), 70)
    kappa = rnd((D,), 71)
    k = np.broadcast_to(kappa, (B, Hkv, Nkv, D)).copy()
    v = rnd((B, Hkv, Nkv, D), 72)
    scale = 0.37
    O, L = fn(q, k, v, scale, False)
    worst = 0.0
    for h in range(Hq):
        kvh = h // (Hq // Hkv)
        worst = max(worst, np.abs(O[0, h] - v[0, kvh].mean(axis=0)[None, :]).max())
        worst = max(worst, np.abs(L[0, h] - (scale * q[0, h] @ kappa + math.log(Nkv))).max())
    return worst


def check_one_hot(fn):
    """Keys are unit basis vectors e_j; query i is 60 * e_{pi(i)}: score 60 on
    key pi(i) and 0 elsewhere, so O_i = V_{pi(i)} up to 7*e^-60 and
    LSE_i = 60 + ln(1 + 7 e^-60)."""
    Nkv = D = 8
    k = np.eye(Nkv)[None, None]
    v = rnd((1, 1, Nkv, 5), 80)
    perm = np.array([3, 0, 7, 5, 1, 6, 2, 4])
    q = (60.0 * np.eye(D)[perm])[None, None]
    O, L = fn(q, k, v, 1.0, False)
    want_L = 60.0 + math.log1p(7 * math.exp(-60.0))
    return max(np.abs(O[0, 0] - v[0, 0, perm]).max(), np.abs(L[0, 0] - want_L).max())


def check_causal_row0(fn):
    """Causal, Nq == Nkv: row 0 sees key 0 only: O_0 = V_0, LSE_0 = scale q0.k0."""
    q, k, v = rnd((2, 3, 9, 6), 90), rnd((2, 3, 9, 6), 91), rnd((2, 3, 9, 6), 92)
    O, L = fn(q, k, v, 0.5, True)
    want = 0.5 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    return max(np.abs(O[:, :, 0] - v[:, :, 0]).max(), np.abs(L[:, :, 0] - want).max())


def check_constant_shift(fn):
    """Append one feature: q'_i[D] = c_i / scale, k'_j[D] = 1, so every score
    of row i grows by c_i.  O is unchanged and LSE grows by c_i."""
    B, Hq, Nq, Nkv, D = 1, 2, 7, 13, 6
    q, k, v = rnd((B, Hq, Nq, D), 100), rnd((B, Hq, Nkv, D), 101), rnd((B, Hq, Nkv, D), 102)
    c = rnd((B, Hq, Nq), 103, amp=5.0)
    scale = 0.8
    q2 = np.concatenate([q, (c / scale)[..., None]], axis=-1)
    k2 = np.concatenate([k, np.ones((B, Hq, Nkv, 1))], axis=-1)
    worst = 0.0
    for causal in (False, True):
        O1, L1 = fn(q, k, v, scale, causal)
        O2, L2 = fn(q2, k2, v, scale, causal)
        worst = max(worst, np.abs(O1 - O2).max(), np.abs(L2 - L1 - c).max())
    return worst


def check_scale_zero(fn):
    """scale = 0: every visible weight is equal.  Non-causal: O = mean of V,
    LSE = ln Nkv.  Causal (Nq == Nkv): O_i = mean of V[0..i], LSE_i = ln(i+1)."""
    q, k, v = rnd((1, 2, 10, 4), 110), rnd((1, 2, 10, 4), 111), rnd((1, 2, 10, 4), 112)
    O, L = fn(q, k, v, 0.0, False)
    worst = max(np.abs(O - v.mean(axis=2, keepdims=True)).max(), np.abs(L - math.log(10)).max())
    O, L = fn(q, k, v, 0.0, True)
    cum = np.cumsum(v, axis=2) / np.arange(1, 11)[None, None, :, None]
    worst = max(worst, np.abs(O - cum).max(), np.abs(L - np.log(np.arange(1, 11))[None, None]).max())
    return worst


def check_key_permutation(fn):
    q, k, v = rnd((1, 2, 5, 4), 120), rnd((1, 2, 9, 4), 121), rnd((1, 2, 9, 3), 122)
    perm = np.random.default_rng(123).permutation(9)
    O1, L1 = fn(q, k, v, 0.6, False)
    O2, L2 = fn(q, k[:, :, perm], v[:, :, perm], 0.6, False)
    return max(np.abs(O1 - O2).max(), np.abs(L1 - L2).max())


def check_gqa_repeat(fn):
    """GQA equals MHA on repeat-interleaved K/V (consecutive groups)."""
    q, k, v = rnd((2, 8, 6, 4), 130), rnd((2, 2, 6, 4), 131), rnd((2, 2, 6, 4), 132)
    worst = 0.0
    for causal in (False, True):
        O1, L1 = fn(q, k, v, 0.5, causal)
        O2, L2 = fn(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), 0.5, causal)
        worst = max(worst, np.abs(O1 - O2).max(), np.abs(L1 - L2).max())
    return worst


def check_causal_future(fn):
    """Causal row i depends on no key or value j > i (Nq == Nkv)."""
    q, k, v = rnd((1, 1, 8, 4), 140), rnd((1, 1, 8, 4), 141), rnd((1, 1, 8, 4), 142)
    O1, L1 = fn(q, k, v, 0.9, True)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 5:] += 7.0
    v2[:, :, 5:] -= 3.0
    O2, L2 = fn(q, k2, v2, 0.9, True)
    return max(np.abs(O1[:, :, :5] - O2[:, :, :5]).max(), np.abs(L1[:, :, :5] - L2[:, :, :5]).max())


def check_hand_examples(fn):
    with open(os.path.join(HERE, "golden", "hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    worst = 0.0
    for c in cases:
        q = np.array(c["q"], dtype=np.float64)[None, None]
        k = np.array(c["k"], dtype=np.float64)[None, None]
        v = np.array(c["v"], dtype=np.float64)[None, None]
        O, L = fn(q, k, v, c["scale"], c["causal"])
        want_O = np.array(c["O"], dtype=np.float64)
        want_L = np.array([float(x) for x in c["LSE"]])
        worst = max(worst, np.abs(O[0, 0] - want_O).max())
        fin = np.isfinite(want_L)
        if not np.array_equal(fin, np.isfinite(L[0, 0])):
            return math.inf
        worst = max(worst, np.abs(L[0, 0][fin] - want_L[fin]).max(initial=0.0))
    return worst


CHECKS = [check_bruteforce, check_torch_sdpa, check_identical_keys, check_one_hot, check_causal_row0,
          check_constant_shift, check_scale_zero, check_key_permutation, check_gqa_repeat,
          check_causal_future, check_hand_examples]


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_oracle_pin(check):
    assert check(oracle.attention) < 1e-10


# ---------------------------------------------------------------------------
# further invariants of the oracle's own helpers

def test_rows_sum_to_one():
    q, k = rnd((40, 16), 1), rnd((50, 16), 2)
    for causal in (False, True):
        P = oracle.probs_head(q, k, 0.25, causal)
        assert np.abs(P.sum(axis=1) - 1.0).max() < 1e-13
        assert (P >= 0).all()
    # causal with Nq > Nkv: the first Nq - Nkv rows see nothing
    P = oracle.probs_head(rnd((9, 4), 3), rnd((5, 4), 4), 1.0, True)
    assert np.all(P[:4] == 0) and np.abs(P[4:].sum(axis=1) - 1).max() < 1e-13


def test_fully_masked_rows():
    q, k, v = rnd((1, 2, 9, 4), 5), rnd((1, 2, 5, 4), 6), rnd((1, 2, 5, 4), 7)
    O, L = oracle.attention(q, k, v, 0.5, True)
    assert np.all(O[:, :, :4] == 0) and np.all(np.isneginf(L[:, :, :4]))
    assert np.all(np.isfinite(L[:, :, 4:]))
    # the first visible row (i = Nq - Nkv) sees key 0 only
    assert np.abs(O[:, :, 4] - v[:, :, 0]).max() < 1e-15


@pytest.mark.parametrize("block", [1, 3, 16, 64, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_online_equals_two_pass(block, causal):
    q, k, v = rnd((37, 16), 8), rnd((100, 16), 9, amp=2.0), rnd((100, 12), 10)
    if causal:
        k, v = k[:60], v[:60]
    O1, L1 = oracle.attention_head(q, k, v, 0.5, causal)
    O2, L2 = oracle.attention_online_head(q, k, v, 0.5, causal, block)
    fin = np.isfinite(L1)
    assert np.array_equal(fin, np.isfinite(L2))
    assert np.abs(O1 - O2).max() < 1e-13
    assert np.abs(L1[fin] - L2[fin]).max() < 1e-13


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("cuts", [(40,), (7, 64), (1, 2, 90)])
def test_lse_merge_of_key_ranges(causal, cuts):
    """Attention over all keys equals the LSE merge of attention over disjoint
    key ranges.  The causal case uses Nq == Nkv and masks each range with the
    global positions."""
    N, D = 100, 8
    q, k, v = rnd((N, D), 11), rnd((N, D), 12), rnd((N, D), 13)
    O, L = oracle.attention_head(q, k, v, 0.4, causal)
    edges = [0, *cuts, N]
    parts = []
    for a, b in zip(edges[:-1], edges[1:]):
        S = 0.4 * (q @ k[a:b].T)
        if causal:
            S = np.where(np.arange(a, b)[None, :] <= np.arange(N)[:, None], S, -np.inf)
        m = S.max(axis=1)
        live = np.isfinite(m)
        m0 = np.where(live, m, 0)
        E = np.exp(S - m0[:, None])
        l = E.sum(axis=1)
        l1 = np.where(live, l, 1)
        parts.append((np.where(live[:, None], E @ v[a:b] / l1[:, None], 0),
                      np.where(live, m0 + np.log(l1), -np.inf)))
    O2, L2 = oracle.lse_merge(parts)
    assert np.abs(O - O2).max() < 1e-13
    assert np.abs(L - L2).max() < 1e-13


def test_kv_head_mapping():
    assert [oracle.kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.kv_head_of(h, 4, 1) for h in range(4)] == [0, 0, 0, 0]
    with pytest.raises(ValueError):
        oracle.kv_head_of(0, 6, 4)


# ---------------------------------------------------------------------------
# planted mistakes: each broken copy must fail at least one pin

def _mutant(kind):
    def fn(q, k, v, scale, causal):
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        if kind == "no_scale":
            return oracle.attention(q, k, v, 1.0, causal)
        if kind == "scale_squared":
            return oracle.attention(q, k, v, scale * scale, causal)
        if kind == "gqa_modulo":
            Hq, Hkv = q.shape[1], k.shape[1]
            idx = [h % Hkv for h in range(Hq)]
            return oracle.attention(q, k[:, idx], v[:, idx], scale, causal)
        if kind == "causal_topleft":
            O, L = oracle.attention(q, k, v, scale, False)
            if not causal:
                return O, L
            Nq, Nkv = q.shape[2], k.shape[2]
            O2, L2 = np.empty_like(O), np.empty_like(L)
            for b in range(q.shape[0]):
                for h in range(q.shape[1]):
                    kv = h // (q.shape[1] // k.shape[1])
                    S = scale * q[b, h] @ k[b, kv].T
                    S = np.where(np.arange(Nkv)[None] <= np.arange(Nq)[:, None], S, -np.inf)
                    m = S.max(1)
                    E = np.exp(S - m[:, None])
                    O2[b, h] = E @ v[b, kv] / E.sum(1)[:, None]
                    L2[b, h] = m + np.log(E.sum(1))
            return O2, L2
        if kind == "lse_no_max":
            O, L = oracle.attention(q, k, v, scale, causal)
            r = oracle.attention(q, k, v, scale, causal)
            # LSE without the max term added back
            Sm = np.zeros_like(L)
            for b in range(q.shape[0]):
                for h in range(q.shape[1]):
                    kv = h // (q.shape[1] // k.shape[1])
                    Sm[b, h] = oracle.scores_head(q[b, h], k[b, kv], scale, causal).max(1)
            return r[0], np.where(np.isfinite(L), L - Sm, L)
        if kind == "unnormalised":
            O, L = oracle.attention(q, k, v, scale, causal)
            return O * 1.01, L
        if kind == "transposed_pv":
            # weights applied to the transposed V block (only meaningful when shapes allow)
            O, L = oracle.attention(q, k, v, scale, causal)
            if v.shape[2] == v.shape[3]:
                vt = np.swapaxes(v, 2, 3)
                return oracle.attention(q, k, vt, scale, causal)[0], L
            return O[..., ::-1], L
        if kind == "online_sign":
            # rescale factor with the wrong sign in the online recurrence
            orig = np.exp
            B, Hq, Nq, _ = q.shape
            Hkv = k.shape[1]
            O = np.zeros((B, Hq, Nq, v.shape[3]))
            L = np.zeros((B, Hq, Nq))
            for b in range(B):
                for h in range(Hq):
                    kv = h // (Hq // Hkv)
                    qq, kk, vv = q[b, h], k[b, kv], v[b, kv]
                    m = np.full(Nq, -np.inf)
                    l = np.zeros(Nq)
                    acc = np.zeros((Nq, vv.shape[1]))
                    rows = np.arange(Nq)
                    for c0 in range(0, kk.shape[0], 2):
                        x = scale * qq @ kk[c0:c0 + 2].T
                        if causal:
                            vis = np.arange(c0, min(c0 + 2, kk.shape[0]))[None] <= rows[:, None] + (kk.shape[0] - Nq)
                            x = np.where(vis, x, -np.inf)
                        mn = np.maximum(m, x.max(1))
                        mn0 = np.where(np.isfinite(mn), mn, 0)
                        alpha = np.where(np.isfinite(m), orig(mn0 - m), 0)   # wrong sign
                        p = orig(x - mn0[:, None])
                        l = alpha * l + p.sum(1)
                        acc = alpha[:, None] * acc + p @ vv[c0:c0 + 2]
                        m = mn
                    live = np.isfinite(m)
                    l1 = np.where(live, l, 1)
                    O[b, h] = np.where(live[:, None], acc / l1[:, None], 0)
                    L[b, h] = np.where(live, np.where(live, m, 0) + np.log(l1), -np.inf)
            return O, L
        if kind in ("causal_strict", "causal_shift_sign", "lse_log2", "lse_unscaled", "pv_uses_k", "gqa_div_hkv"):
            return _variant(kind, q, k, v, scale, causal)
        raise ValueError(kind)
    return fn


def _variant(kind, q, k, v, scale, causal):
    """The definition written out once more with one deliberate slip."""
    B, Hq, Nq, _ = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    O = np.zeros((B, Hq, Nq, v.shape[3]))
    L = np.zeros((B, Hq, Nq))
    i = np.arange(Nq)[:, None]
    j = np.arange(Nkv)[None]
    for b in range(B):
        for h in range(Hq):
            kv = min(h // Hkv, Hkv - 1) if kind == "gqa_div_hkv" else h // (Hq // Hkv)
            raw = q[b, h] @ k[b, kv].T
            S = scale * raw
            if causal:
                if kind == "causal_strict":
                    vis = j < i + (Nkv - Nq)            # the diagonal masked too
                elif kind == "causal_shift_sign":
                    vis = j <= i - (Nkv - Nq)           # offset with the wrong sign
                else:
                    vis = j <= i + (Nkv - Nq)
                S = np.where(vis, S, -np.inf)
                raw = np.where(vis, raw, -np.inf)
            m = S.max(1) if Nkv else np.full(Nq, -np.inf)
            live = np.isfinite(m)
            m0 = np.where(live, m, 0.0)
            E = np.exp(S - m0[:, None])
            l1 = np.where(live, E.sum(1), 1.0)
            src = k[b, kv] if kind == "pv_uses_k" else v[b, kv]
            O[b, h] = np.where(live[:, None], E @ src / l1[:, None], 0.0)
            if kind == "lse_log2":
                L[b, h] = np.where(live, (m0 + np.log(l1)) / math.log(2.0), -np.inf)
            elif kind == "lse_unscaled":
                mr = np.where(live, raw.max(1), 0.0)
                L[b, h] = np.where(live, mr + np.log(np.exp(raw - mr[:, None]).sum(1)), -np.inf)
            else:
                L[b, h] = np.where(live, m0 + np.log(l1), -np.inf)
    return O, L


MUTANTS = ["no_scale", "scale_squared", "gqa_modulo", "causal_topleft", "lse_no_max", "unnormalised",
           "transposed_pv", "online_sign", "causal_strict", "causal_shift_sign", "lse_log2", "lse_unscaled",
           "pv_uses_k", "gqa_div_hkv"]


def test_variant_without_slip_matches_oracle():
    # the helper that plants the slips is itself the definition when no slip is chosen
    rng = np.random.default_rng(7)
    q = rng.standard_normal((2, 4, 9, 8))
    k = rng.standard_normal((2, 2, 13, 8))
    v = rng.standard_normal((2, 2, 13, 8))
    for causal in (False, True):
        O, L = _variant("none", q, k, v, 0.3, causal)
        O_ref, L_ref = oracle.attention(q, k, v, 0.3, causal)
        assert np.allclose(O, O_ref, atol=1e-12) and np.allclose(L, L_ref, atol=1e-12)


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistake(kind):
    fn = _mutant(kind)
    with np.errstate(all="ignore"):
        errs = []
        for c in CHECKS:
            try:
                errs.append(c(fn))
            except Exception:  # a crash is a detection too
                errs.append(math.inf)
    assert max(errs) > 1e-6, f"mutant {kind} passed every pin"


def test_oracle_module_has_no_product_imports():
    import ast
    for path in (oracle_mod.__file__, os.path.join(os.path.dirname(oracle_mod.__file__), "__init__.py"),
                 os.path.join(os.path.dirname(oracle_mod.__file__), "fp8.py")):
        tree = ast.parse(open(path).read())
        names = set()
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                names.update(a.name.split(".")[0] for a in node.names)
            elif isinstance(node, ast.ImportFrom) and node.level == 0:
                names.add(node.module.split(".")[0])
        assert names <= {"__future__", "math", "numpy"}, names
