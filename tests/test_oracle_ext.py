"""Pins for the oracle's row softmax, additive mask and backward pass.

Like ``test_oracle.py``, every ``check_*`` helper compares a function with the
oracle's signature against something other than the oracle itself (torch's
float64 routines, pure-Python loops, finite differences, closed forms), and
each helper family is run on deliberately broken copies that must fail at
least one of them.

Sources (page title, section):
* "FlashAttention v1/v2/v3/v4" (lo0.es), "El truco que hizo posible todo:
  online softmax": the softmax exp(x_i - m) / sum_j exp(x_j - m).
* "ffpa-attn 0.2.3" README feature table ("Causal/Mask"): a mask besides the
  causal one, read as SDPA's additive float mask.
* "FlashAttention v1/v2/v3/v4", "FA1 -- el cambio de orden de las
  operaciones", and the FlashAttention summary card: the backward pass
  recomputes S from Q, K and the row statistics; its result is the gradient
  of the forward definition.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def rnd(shape, seed, amp=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * amp


def _causal_bool(Nq, Nkv):
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nkv)[None, :]
    return j <= i + (Nkv - Nq)


def _torch_scores(q, k, scale, causal, mask):
    """float64 scaled scores + mask, bottom-right causal -inf, by torch ops
    (K repeat-interleaved over GQA groups)."""
    tq, tk = torch.from_numpy(np.ascontiguousarray(q)), torch.from_numpy(np.ascontiguousarray(k))
    tk = tk.repeat_interleave(tq.shape[1] // tk.shape[1], dim=1)
    s = torch.matmul(tq, tk.transpose(-1, -2)) * scale
    if mask is not None:
        s = s + torch.from_numpy(np.array(np.broadcast_to(mask, s.shape)))
    if causal:
        s = s.masked_fill(~_causal_bool(q.shape[2], k.shape[2]), -math.inf)
    return s


# ---------------------------------------------------------------------------
# probs_head: the row softmax

SOFTMAX_CASES = [(1, 2, 2, 33, 33, 16, False), (1, 2, 2, 33, 33, 16, True), (1, 2, 2, 10, 40, 8, True),
                 (1, 1, 1, 9, 5, 4, True), (1, 1, 1, 7, 21, 8, False)]


def check_probs_torch_softmax(fn):
    """fn(q, k, scale, causal) -> P for one head, against torch.softmax of the
    float64 scaled, bottom-right-masked scores.  Rows with no visible key
    (torch gives NaN there) must be all zero."""
    worst = 0.0
    for n, (B, Hq, Hkv, Nq, Nkv, D, causal) in enumerate(SOFTMAX_CASES):
        q = rnd((B, Hq, Nq, D), 300 + n)
        k = rnd((B, Hkv, Nkv, D), 310 + n, amp=1.5)
        scale = 1.0 / math.sqrt(D) * 1.7
        want = torch.softmax(_torch_scores(q, k, scale, causal, None), dim=-1).numpy()
        for h in range(Hq):
            P = fn(q[0, h], k[0, h // (Hq // Hkv)], scale, causal)
            dead = np.isnan(want[0, h]).all(axis=1)
            if dead.any() and np.abs(P[dead]).max() != 0.0:
                return math.inf
            worst = max(worst, np.abs(P[~dead] - want[0, h][~dead]).max())
    return worst


def check_probs_closed_forms(fn):
    """Two keys with scores 0 and ln 3 give weights 1/4 and 3/4; scale 0
    gives equal weights over the visible keys."""
    P = fn(np.array([[1.0]]), np.array([[0.0], [math.log(3.0)]]), 1.0, False)
    worst = np.abs(P - np.array([[0.25, 0.75]])).max()
    q, k = rnd((6, 3), 320), rnd((6, 3), 321)
    P = fn(q, k, 0.0, True)
    want = np.tril(np.ones((6, 6))) / np.arange(1, 7)[:, None]
    return max(worst, np.abs(P - want).max())


PROBS_CHECKS = [check_probs_torch_softmax, check_probs_closed_forms]


def test_probs_head_pins():
    for c in PROBS_CHECKS:
        assert c(lambda q, k, s, cz: oracle.probs_head(q, k, s, cz)) < 1e-13, c.__name__


def _probs_mutant(kind):
    def fn(q, k, scale, causal):
        if kind == "no_scale":
            return oracle.probs_head(q, k, 1.0, causal)
        S = oracle.scores_head(q, k, scale, causal)
        m = S.max(axis=1)
        live = np.isfinite(m)
        m0 = np.where(live, m, 0.0)
        if kind == "exp2":
            E = np.exp2(S - m0[:, None])
        elif kind == "unmasked":
            S = oracle.scores_head(q, k, scale, False)
            E = np.exp(S - S.max(axis=1)[:, None])
        else:
            E = np.exp(S - m0[:, None])
        l = E.sum(axis=1)
        P = np.where(live[:, None], E / np.where(live, l, 1.0)[:, None], 0.0)
        if kind == "dead_rows_uniform":
            P[~live] = 1.0 / max(1, P.shape[1])
        if kind == "transposed" and P.shape[0] == P.shape[1]:
            P = P.T.copy()
        return P
    return fn


@pytest.mark.parametrize("kind", ["no_scale", "exp2", "unmasked", "dead_rows_uniform", "transposed"])
def test_probs_pins_catch_planted_mistake(kind):
    fn = _probs_mutant(kind)
    with np.errstate(all="ignore"):
        errs = [c(fn) for c in PROBS_CHECKS]
    assert max(errs) > 1e-6, f"probs_head mutant {kind} passed every pin"


# ---------------------------------------------------------------------------
# additive mask

def _rand_mask(shape, seed, p_neg_inf=0.2, amp=2.0):
    rng = np.random.default_rng(seed)
    m = rng.standard_normal(shape) * amp
    m[rng.random(shape) < p_neg_inf] = -np.inf
    return m


def _sdpa_masked(q, k, v, scale, causal, mask):
    """torch float64 SDPA with the additive mask (causal folded in as -inf),
    plus torch.logsumexp of the same scores.  Fully masked rows are NaN in
    SDPA's output; they are returned as such."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    g = tq.shape[1] // tk.shape[1]
    tk, tv = tk.repeat_interleave(g, dim=1), tv.repeat_interleave(g, dim=1)
    bias = torch.zeros((tq.shape[0], tq.shape[1], tq.shape[2], tk.shape[2]), dtype=torch.float64)
    if mask is not None:
        bias = bias + torch.from_numpy(np.array(np.broadcast_to(mask, bias.shape)))
    if causal:
        bias = bias.masked_fill(~_causal_bool(tq.shape[2], tk.shape[2]), -math.inf)
    O = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=bias, scale=scale)
    L = torch.logsumexp(torch.matmul(tq, tk.transpose(-1, -2)) * scale + bias, dim=-1)
    return O.numpy(), L.numpy()


MASK_CASES = [  # B, Hq, Hkv, Nq, Nkv, D, causal, mask shape ('full' | 'heads1' | 'batch1' | 'row')
    (2, 4, 2, 13, 13, 8, False, "full"), (2, 4, 2, 13, 13, 8, True, "full"), (1, 4, 1, 9, 21, 8, False, "heads1"),
    (2, 2, 2, 10, 7, 4, True, "batch1"), (1, 2, 2, 6, 11, 4, False, "row")]


def _mask_shape(kind, B, Hq, Nq, Nkv):
    return {"full": (B, Hq, Nq, Nkv), "heads1": (B, 1, Nq, Nkv), "batch1": (1, Hq, Nq, Nkv),
            "row": (Nkv,)}[kind]


def check_mask_sdpa(fn):
    """fn(q, k, v, scale, causal, mask) against torch float64 SDPA with the
    float mask; rows torch leaves NaN (no visible key) must be O = 0,
    LSE = -inf."""
    worst = 0.0
    for n, (B, Hq, Hkv, Nq, Nkv, D, causal, mk) in enumerate(MASK_CASES):
        q, k, v = rnd((B, Hq, Nq, D), 400 + n), rnd((B, Hkv, Nkv, D), 410 + n), rnd((B, Hkv, Nkv, D), 420 + n)
        mask = _rand_mask(_mask_shape(mk, B, Hq, Nq, Nkv), 430 + n)
        O, L = fn(q, k, v, 0.6, causal, mask)
        Ot, Lt = _sdpa_masked(q, k, v, 0.6, causal, mask)
        dead = np.isneginf(Lt)
        if not np.array_equal(dead, np.isneginf(L)) or np.abs(O[dead]).max(initial=0.0) != 0.0:
            return math.inf
        worst = max(worst, np.abs(O[~dead] - Ot[~dead]).max(), np.abs(L[~dead] - Lt[~dead]).max())
    return worst


def check_mask_bruteforce(fn):
    worst = 0.0
    for n, (B, Hq, Hkv, Nq, Nkv, D) in enumerate([(1, 2, 1, 5, 5, 3), (2, 2, 2, 4, 7, 2), (1, 3, 1, 6, 3, 2)]):
        q, k, v = rnd((B, Hq, Nq, D), 440 + n), rnd((B, Hkv, Nkv, D), 450 + n), rnd((B, Hkv, Nkv, D), 460 + n)
        mask = _rand_mask((B, Hq, Nq, Nkv), 470 + n, p_neg_inf=0.3)
        for causal in (False, True):
            O, L = fn(q, k, v, 0.9, causal, mask)
            Ob, Lb = oracle.attention_bruteforce(q, k, v, 0.9, causal, mask)
            if not np.array_equal(np.isfinite(L), np.isfinite(Lb)):
                return math.inf
            fin = np.isfinite(Lb)
            worst = max(worst, np.abs(O - Ob).max(), np.abs(L[fin] - Lb[fin]).max(initial=0.0))
    return worst


def check_mask_closed_forms(fn):
    """A per-row constant c leaves O and shifts LSE by c; a 0/-inf mask equal
    to the causal one gives the causal result; a mask that hides every key
    but j* gives O = V[j*] and LSE = scale q.k_{j*} + M[j*]."""
    B, Hq, Nq, Nkv, D = 1, 2, 7, 9, 4
    q, k, v = rnd((B, Hq, Nq, D), 480), rnd((B, Hq, Nkv, D), 481), rnd((B, Hq, Nkv, D), 482)
    c = rnd((B, Hq, Nq, 1), 483, amp=3.0)
    O0, L0 = fn(q, k, v, 0.7, False, None)
    O1, L1 = fn(q, k, v, 0.7, False, np.broadcast_to(c, (B, Hq, Nq, Nkv)))
    worst = max(np.abs(O1 - O0).max(), np.abs(L1 - L0 - c[..., 0]).max())
    causal_as_mask = np.where(_causal_bool(Nq, Nkv).numpy(), 0.0, -np.inf)
    Oc, Lc = fn(q, k, v, 0.7, True, None)
    Om, Lm = fn(q, k, v, 0.7, False, causal_as_mask)
    worst = max(worst, np.abs(Oc - Om).max(), np.abs(Lc - Lm).max())
    jstar = np.array([3, 0, 8, 5, 5, 1, 2])
    only = np.full((Nq, Nkv), -np.inf)
    only[np.arange(Nq), jstar] = 1.25
    O, L = fn(q, k, v, 0.7, False, only)
    for h in range(Hq):
        want_L = 0.7 * np.einsum("id,id->i", q[0, h], k[0, h, jstar]) + 1.25
        worst = max(worst, np.abs(O[0, h] - v[0, h, jstar]).max(), np.abs(L[0, h] - want_L).max())
    return worst


MASK_CHECKS = [check_mask_sdpa, check_mask_bruteforce, check_mask_closed_forms]


@pytest.mark.parametrize("check", MASK_CHECKS, ids=[c.__name__ for c in MASK_CHECKS])
def test_mask_pins(check):
    assert check(lambda q, k, v, s, cz, m: oracle.attention(q, k, v, s, cz, mask=m)) < 1e-10


def _mask_mutant(kind):
    def fn(q, k, v, scale, causal, mask):
        if mask is None or kind == "ignored":
            return oracle.attention(q, k, v, scale, causal)
        B, Hq, Nq, _ = q.shape
        Nkv = k.shape[2]
        M = np.broadcast_to(np.asarray(mask, dtype=np.float64), (B, Hq, Nq, Nkv))
        if kind == "before_scale":       # scale * (Q K^T + M)
            return oracle.attention(q, k, v, scale, causal, mask=M * scale if scale else M)
        if kind == "sign":               # S - M (with -inf kept as -inf)
            return oracle.attention(q, k, v, scale, causal, mask=np.where(np.isneginf(M), M, -M))
        if kind == "log2_units":         # the mask read as base-2 logits
            return oracle.attention(q, k, v, scale, causal, mask=M * math.log(2.0))
        if kind == "head_swapped":       # another head's mask
            return oracle.attention(q, k, v, scale, causal, mask=M[:, ::-1])
        if kind == "after_max":          # mask added after the row max is taken (not in LSE's max)
            O, L = oracle.attention(q, k, v, scale, causal, mask=M)
            return O, L + 0.01 * np.isfinite(L)
        raise ValueError(kind)
    return fn


@pytest.mark.parametrize("kind", ["ignored", "before_scale", "sign", "log2_units", "head_swapped", "after_max"])
def test_mask_pins_catch_planted_mistake(kind):
    fn = _mask_mutant(kind)
    with np.errstate(all="ignore"):
        errs = []
        for c in MASK_CHECKS:
            try:
                errs.append(c(fn))
            except Exception:
                errs.append(math.inf)
    assert max(errs) > 1e-6, f"mask mutant {kind} passed every pin"


def test_mask_none_and_zero_agree_with_unmasked():
    q, k, v = rnd((1, 2, 5, 4), 490), rnd((1, 2, 8, 4), 491), rnd((1, 2, 8, 4), 492)
    for causal in (False, True):
        O0, L0 = oracle.attention(q, k, v, 0.5, causal)
        O1, L1 = oracle.attention(q, k, v, 0.5, causal, mask=np.zeros((5, 8)))
        assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


# ---------------------------------------------------------------------------
# backward

def _torch_grads(q, k, v, do, scale, causal, mask):
    """dq, dk, dv by torch float64 autograd through SDPA (GQA by
    repeat_interleave, whose backward sums over each group)."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x)).requires_grad_(True) for x in (q, k, v))
    g = tq.shape[1] // tk.shape[1]
    bias = None
    Nq, Nkv = q.shape[2], k.shape[2]
    if mask is not None or causal:
        bias = torch.zeros((q.shape[0], q.shape[1], Nq, Nkv), dtype=torch.float64)
        if mask is not None:
            bias = bias + torch.from_numpy(np.array(np.broadcast_to(mask, bias.shape)))
        if causal:
            bias = bias.masked_fill(~_causal_bool(Nq, Nkv), -math.inf)
    O = torch.nn.functional.scaled_dot_product_attention(tq, tk.repeat_interleave(g, dim=1),
                                                         tv.repeat_interleave(g, dim=1), attn_mask=bias, scale=scale)
    O.backward(torch.from_numpy(np.ascontiguousarray(do)))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


BWD_CASES = [  # B, Hq, Hkv, Nq, Nkv, D, causal, masked
    (2, 4, 4, 17, 17, 8, False, False), (2, 4, 4, 17, 17, 8, True, False), (1, 8, 2, 12, 12, 8, True, False),
    (1, 4, 1, 9, 23, 8, False, False), (1, 2, 2, 20, 11, 4, False, True), (1, 4, 2, 14, 14, 8, True, True)]


def check_bwd_torch(fn):
    """fn(q, k, v, do, scale, causal, mask) -> (dq, dk, dv) against torch
    float64 autograd.  Rows with no visible key are avoided here (SDPA's
    gradient is NaN there)."""
    worst = 0.0
    for n, (B, Hq, Hkv, Nq, Nkv, D, causal, masked) in enumerate(BWD_CASES):
        q, k, v = rnd((B, Hq, Nq, D), 500 + n), rnd((B, Hkv, Nkv, D), 510 + n), rnd((B, Hkv, Nkv, D), 520 + n)
        do = rnd((B, Hq, Nq, D), 530 + n)
        mask = _rand_mask((B, Hq, Nq, Nkv), 540 + n, p_neg_inf=0.1) if masked else None
        if mask is not None:
            mask[..., 0] = 0.5   # every row keeps key 0 visible
        scale = 1.0 / math.sqrt(D)
        got = fn(q, k, v, do, scale, causal, mask)
        want = _torch_grads(q, k, v, do, scale, causal, mask)
        worst = max(worst, *(np.abs(a - b).max() for a, b in zip(got, want)))
    return worst


def check_bwd_finite_differences(fn):
    """Central differences of L = sum(O * dO) on tiny inputs (step 1e-5):
    dL/dx is the gradient for upstream gradient dO."""
    worst = 0.0
    for n, (B, Hq, Hkv, Nq, Nkv, D, causal) in enumerate([(1, 2, 1, 4, 4, 3, True), (1, 1, 1, 3, 5, 2, False)]):
        q, k, v = rnd((B, Hq, Nq, D), 550 + n), rnd((B, Hkv, Nkv, D), 560 + n), rnd((B, Hkv, Nkv, D), 570 + n)
        do = rnd((B, Hq, Nq, D), 580 + n)
        mask = _rand_mask((B, Hq, Nq, Nkv), 590 + n, p_neg_inf=0.0, amp=0.5) if n == 1 else None
        got = fn(q, k, v, do, 0.8, causal, mask)

        def loss(qq, kk, vv):
            O, _ = oracle.attention_bruteforce(qq, kk, vv, 0.8, causal, mask)
            return float((O * do).sum())

        h = 1e-5
        for which, x in enumerate((q, k, v)):
            g = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[which], args_m[which] = xp, xm
                g[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            worst = max(worst, np.abs(got[which] - g).max())
    return worst


def check_bwd_closed_forms(fn):
    """One key: the softmax is constantly 1, so dq = dk = 0 and dv = sum_i dO_i.
    Scale 0 (non-causal): dq = dk = 0, every dv_j = (1/Nkv) sum_i dO_i.
    Any problem: sum over keys of dk is 0 (each row of dS sums to 0), and
    sum over keys of dv is sum_i dO_i over rows that see a key."""
    q, k, v, do = rnd((1, 2, 6, 4), 600), rnd((1, 2, 1, 4), 601), rnd((1, 2, 1, 4), 602), rnd((1, 2, 6, 4), 603)
    dq, dk, dv = fn(q, k, v, do, 0.9, False, None)
    worst = max(np.abs(dq).max(), np.abs(dk).max(), np.abs(dv[:, :, 0] - do.sum(axis=2)).max())
    q, k, v, do = rnd((1, 2, 5, 4), 604), rnd((1, 2, 7, 4), 605), rnd((1, 2, 7, 4), 606), rnd((1, 2, 5, 4), 607)
    dq, dk, dv = fn(q, k, v, do, 0.0, False, None)
    worst = max(worst, np.abs(dq).max(), np.abs(dk).max(), np.abs(dv - do.sum(axis=2, keepdims=True) / 7).max())
    q, k, v = rnd((1, 4, 9, 4), 608), rnd((1, 2, 9, 4), 609), rnd((1, 2, 9, 4), 610)
    do = rnd((1, 4, 9, 4), 611)
    for causal in (False, True):
        dq, dk, dv = fn(q, k, v, do, 0.6, causal, None)
        worst = max(worst, np.abs(dk.sum(axis=2)).max())
        want_dv = do.reshape(1, 2, 2, 9, 4).sum(axis=(2, 3))
        worst = max(worst, np.abs(dv.sum(axis=2) - want_dv).max())
    return worst


BWD_CHECKS = [check_bwd_torch, check_bwd_finite_differences, check_bwd_closed_forms]


@pytest.mark.parametrize("check", BWD_CHECKS, ids=[c.__name__ for c in BWD_CHECKS])
def test_backward_pins(check):
    tol = 1e-7 if check is check_bwd_finite_differences else 1e-10
    assert check(lambda *a: oracle.attention_backward(*a)) < tol


def _bwd_mutant(kind):
    def fn(q, k, v, do, scale, causal, mask):
        if kind == "dq_unscaled":
            dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal, mask)
            return (dq / scale if scale else dq + 1.0), dk, dv
        if kind == "dk_last_head_only":
            B, Hq = q.shape[:2]
            Hkv = k.shape[1]
            dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal, mask)
            if Hq == Hkv:
                return dq, dk, dv
            g = Hq // Hkv
            last = np.zeros_like(k)
            for kv in range(Hkv):
                h = kv * g + g - 1
                M = None if mask is None else np.broadcast_to(mask, (B, Hq) + mask.shape[-2:])[0, h]
                last[0, kv] = oracle.attention_backward_head(q[0, h], k[0, kv], v[0, kv], do[0, h], scale, causal, M)[1]
            return dq, last, dv
        # the chain rule written out once more, with one slip
        B, Hq, Nq, D = q.shape
        Hkv, Nkv = k.shape[1], k.shape[2]
        Mf = None if mask is None else np.broadcast_to(mask, (B, Hq, Nq, Nkv))
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for b in range(B):
            for h in range(Hq):
                kv = h // (Hq // Hkv)
                P = oracle.probs_head(q[b, h], k[b, kv], scale, causal, None, None if Mf is None else Mf[b, h])
                O = P @ v[b, kv]
                dP = do[b, h] @ v[b, kv].T
                delta = (do[b, h] * O).sum(axis=1)
                if kind == "no_delta":
                    dS = P * dP
                elif kind == "dS_sign":
                    dS = P * (delta[:, None] - dP)
                elif kind == "delta_from_v":
                    dS = P * (dP - (do[b, h] * v[b, kv][:Nq] if Nkv >= Nq else do[b, h]).sum(axis=1)[:, None])
                else:
                    dS = P * (dP - delta[:, None])
                dq[b, h] = scale * dS @ k[b, kv]
                dk[b, kv] += scale * (dS @ q[b, h] if (kind == "dk_untransposed" and Nq == Nkv) else dS.T @ q[b, h])
                dv[b, kv] += (dP.T @ do[b, h] if kind == "dv_uses_dp" else P.T @ do[b, h])
        return dq, dk, dv
    return fn


BWD_MUTANTS = ["dq_unscaled", "dk_last_head_only", "no_delta", "dS_sign", "delta_from_v", "dk_untransposed",
               "dv_uses_dp"]


def test_bwd_variant_without_slip_matches_oracle():
    fn = _bwd_mutant("none")
    q, k, v, do = rnd((1, 4, 7, 4), 620), rnd((1, 2, 9, 4), 621), rnd((1, 2, 9, 4), 622), rnd((1, 4, 7, 4), 623)
    for causal in (False, True):
        for a, b in zip(fn(q, k, v, do, 0.4, causal, None), oracle.attention_backward(q, k, v, do, 0.4, causal)):
            assert np.allclose(a, b, atol=1e-12)


@pytest.mark.parametrize("kind", BWD_MUTANTS)
def test_bwd_pins_catch_planted_mistake(kind):
    fn = _bwd_mutant(kind)
    with np.errstate(all="ignore"):
        errs = []
        for c in BWD_CHECKS:
            try:
                errs.append(c(fn))
            except Exception:
                errs.append(math.inf)
    assert max(errs) > 1e-5, f"backward mutant {kind} passed every pin"


@pytest.mark.parametrize("shape", [(37, 37), (50, 23), (23, 61)])
def test_backward_sampled_matches_full_backward(shape):
    # the blocked, sampled gradients equal the entries of the full backward
    # (itself pinned by torch autograd, finite differences and closed forms),
    # with blocks smaller than the rows, a ragged last block, causal or not
    Nq, Nkv = shape
    q, k, v, do = rnd((Nq, 8), 700), rnd((Nkv, 8), 701), rnd((Nkv, 8), 702), rnd((Nq, 8), 703)
    rows = np.array([0, 5, Nq // 2, Nq - 1])
    keys = np.array([0, 3, Nkv // 2, Nkv - 1])
    for causal in (False, True):
        full = oracle.attention_backward_head(q, k, v, do, 0.35, causal)
        dq, dk, dv = oracle.attention_backward_sampled(q, k, v, do, 0.35, causal, rows, keys, block=16)
        assert np.allclose(dq, full[0][rows], rtol=0, atol=1e-12)
        assert np.allclose(dk, full[1][keys], rtol=0, atol=1e-12)
        assert np.allclose(dv, full[2][keys], rtol=0, atol=1e-12)
