"""Float64 CPU oracle for exact scaled-dot-product attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg (and its ``--impl reference`` arm) may use it.  It shares no
code with the CUDA path; the two meet only through the seeded inputs of
``exact_attention_attn_gb300.workloads``, which hold no attention arithmetic.

What is computed (the plain definition; sources by page title and section):

* "FlashAttention: Fast and Memory-Efficient Exact Attention with IO-Awareness"
  (paper summary card, problem statement): standard attention forms the full
  N x N score matrix S = Q K^T, takes a row softmax and multiplies by V.  The
  IO-aware method reaches the same result exactly ("Exact - no approximation").
* "FlashAttention v1/v2/v3/v4: el bibliotecario que nunca despeja la mesa"
  (lo0.es), section "El truco que hizo posible todo: online softmax": the
  softmax is exp(x_i - m) / sum_j exp(x_j - m) with m the row maximum; the
  online form keeps a running max m and running sum l, rescales l and the
  partial output by exp(m_old - m_new) when a new block arrives, and divides
  by the final l; the section states that this equals the standard softmax.
* "ffpa-attn 0.2.3" METADATA (FFPA README), the feature table under the title
  and "Quick Start": layout (B, H, N, D); self-attention Nq = Nkv,
  cross-attention Nq != Nkv, GQA/MQA Hq != Hkv, causal masking.
* "ZYFA: FP8 FlashAttention Kernels for AMD MI355X", section "The details that
  make it production-grade": log-sum-exp values let results computed over
  disjoint key ranges be merged.
* "ffpa-attn 0.2.3" README feature table ("Causal/Mask"): an attention mask
  besides the causal one.  Read here as SDPA's additive float mask: it is
  added to the scaled scores before the row maximum, and an entry of -inf
  hides that key from that query.
* "FlashAttention v1/v2/v3/v4", section "FA1 -- el cambio de orden de las
  operaciones", and the "FlashAttention: Fast and Memory-Efficient Exact
  Attention with IO-Awareness" summary card: the backward pass keeps only the
  row statistics and recomputes S from Q and K.  What it computes is the
  gradient of the forward definition; ``attention_backward`` writes that
  gradient out (chain rule through the row softmax, below).

Readings where the pages are silent (each is listed with the others in the
design notes):

1. LSE is the natural log of sum_j exp(scale * q.k_j) over unmasked keys.
2. Causal masking with Nq != Nkv is bottom-right aligned: query i may see key
   j iff j <= i + (Nkv - Nq).  With Nq == Nkv this is the usual lower
   triangle.
3. A row with no visible key (only possible when causal and Nq > Nkv) has
   O = 0 and LSE = -inf.
4. GQA groups are consecutive: query head hq reads key/value head
   hq // (Hq / Hkv).
5. scale is an explicit argument (the workloads use 1/sqrt(D)).
6. The additive mask M (any array that broadcasts to [B, Hq, Nq, Nkv]) enters
   as S = scale * Q K^T + M, then the causal mask; finite entries and -inf
   are allowed.  A row whose every entry ends up -inf is reading 3's row.

Parity status: pinned (see tests/test_oracle.py): brute force on tiny inputs,
torch's float64 scaled_dot_product_attention, closed forms and invariants.
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# index helpers (readings 2 and 4 above)

def kv_head_of(hq: int, Hq: int, Hkv: int) -> int:
    """Key/value head read by query head ``hq`` (consecutive GQA groups)."""
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return hq // (Hq // Hkv)


def causal_visible(rows: np.ndarray, Nq: int, Nkv: int) -> np.ndarray:
    """Boolean [len(rows), Nkv]: key j is visible to query row i iff
    j <= i + (Nkv - Nq) (bottom-right aligned causal mask)."""
    rows = np.asarray(rows, dtype=np.int64)
    return np.arange(Nkv, dtype=np.int64)[None, :] <= (rows[:, None] + (Nkv - Nq))


# ---------------------------------------------------------------------------
# the plain definition, one head at a time

def scores_head(q: np.ndarray, k: np.ndarray, scale: float, causal: bool,
                rows: np.ndarray | None = None, mask: np.ndarray | None = None) -> np.ndarray:
    """S = scale * Q K^T (+ mask) for the chosen query rows, masked entries -inf.
    ``mask`` is this head's additive mask, broadcastable to [Nq, Nkv] (all
    rows; the chosen ones are taken from it)."""
    Nq, Nkv = q.shape[0], k.shape[0]
    rows = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    S = scale * (q[rows] @ k.T)
    if mask is not None:
        S = S + np.broadcast_to(np.asarray(mask, dtype=np.float64), (Nq, Nkv))[rows]
    if causal:
        S = np.where(causal_visible(rows, Nq, Nkv), S, -np.inf)
    return S


def probs_head(q, k, scale, causal, rows=None, mask=None) -> np.ndarray:
    """Row softmax of the masked scores: P[i, j] = exp(S_ij - m_i) / l_i.
    Rows with no visible key are all zero."""
    S = scores_head(q, k, scale, causal, rows, mask)
    m = S.max(axis=1) if S.shape[1] else np.full(S.shape[0], -np.inf)
    live = np.isfinite(m)
    m0 = np.where(live, m, 0.0)
    E = np.exp(S - m0[:, None])               # exp(-inf) == 0 for masked keys
    l = E.sum(axis=1)
    return np.where(live[:, None], E / np.where(live, l, 1.0)[:, None], 0.0)


def attention_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                   causal: bool, rows: np.ndarray | None = None, mask: np.ndarray | None = None):
    """One head.  q [Nq, D], k and v [Nkv, D], float64.

    Returns (O [r, D], LSE [r]) for the r chosen query rows:
    m_i = max_j S_ij, l_i = sum_j exp(S_ij - m_i), O_i = sum_j exp(S_ij - m_i) v_j / l_i,
    LSE_i = m_i + ln l_i.
    """
    S = scores_head(q, k, scale, causal, rows, mask)
    r = S.shape[0]
    if S.shape[1] == 0:
        return np.zeros((r, v.shape[1])), np.full(r, -np.inf)
    m = S.max(axis=1)
    live = np.isfinite(m)
    m0 = np.where(live, m, 0.0)
    E = np.exp(S - m0[:, None])
    l = E.sum(axis=1)
    l1 = np.where(live, l, 1.0)
    O = np.where(live[:, None], (E @ v) / l1[:, None], 0.0)
    LSE = np.where(live, m0 + np.log(l1), -np.inf)
    return O, LSE


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool,
              rows: np.ndarray | None = None, mask: np.ndarray | None = None):
    """Batched oracle.  q [B, Hq, Nq, D], k and v [B, Hkv, Nkv, D] (float64);
    mask (optional) broadcastable to [B, Hq, Nq, Nkv].

    Returns O [B, Hq, r, D] and LSE [B, Hq, r] (r = Nq, or len(rows) when a
    row subset is given; the same rows are used for every head).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, Nq, D = q.shape
    Bk, Hkv, Nkv, Dk = k.shape
    if Bk != B or Dk != D or v.shape[:3] != k.shape[:3]:
        raise ValueError("shape mismatch")
    r = Nq if rows is None else len(rows)
    M = None if mask is None else np.broadcast_to(np.asarray(mask, dtype=np.float64), (B, Hq, Nq, Nkv))
    O = np.zeros((B, Hq, r, v.shape[3]))
    LSE = np.zeros((B, Hq, r))
    for b in range(B):
        for h in range(Hq):
            kv = kv_head_of(h, Hq, Hkv)
            O[b, h], LSE[b, h] = attention_head(q[b, h], k[b, kv], v[b, kv], scale, causal, rows,
                                                None if M is None else M[b, h])
    return O, LSE


# ---------------------------------------------------------------------------
# brute force, pure-Python loops (tiny inputs only)

def attention_bruteforce(q, k, v, scale, causal, mask=None):
    """Same definition with explicit loops and math.exp; for N, D <= ~16.
    ``mask`` (optional) broadcasts to [B, Hq, Nq, Nkv] and is added to each
    scaled score; a -inf entry drops the key."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    M = None if mask is None else np.broadcast_to(np.asarray(mask, dtype=np.float64), (B, Hq, Nq, Nkv))
    group = Hq // Hkv
    O = np.zeros((B, Hq, Nq, v.shape[3]))
    LSE = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            kh = h // group
            for i in range(Nq):
                s = []
                for j in range(Nkv):
                    if causal and j > i + (Nkv - Nq):
                        continue
                    dot = 0.0
                    for d in range(D):
                        dot += float(q[b, h, i, d]) * float(k[b, kh, j, d])
                    x = scale * dot
                    if M is not None:
                        if M[b, h, i, j] == -math.inf:
                            continue
                        x += float(M[b, h, i, j])
                    s.append((j, x))
                if not s:
                    LSE[b, h, i] = -math.inf
                    continue
                mx = max(x for _, x in s)
                tot = sum(math.exp(x - mx) for _, x in s)
                for d in range(v.shape[3]):
                    acc = 0.0
                    for j, x in s:
                        acc += math.exp(x - mx) * float(v[b, kh, j, d])
                    O[b, h, i, d] = acc / tot
                LSE[b, h, i] = mx + math.log(tot)
    return O, LSE


# ---------------------------------------------------------------------------
# the online (blockwise) softmax, in the order the blog's online-softmax
# section gives it

def attention_online_head(q, k, v, scale, causal, block: int):
    """Walk the keys in blocks of ``block``; keep running max m and running
    sum l per row; when a block arrives with local maximum m_blk:
        m_next = max(m, m_blk)
        l_next = exp(m - m_next) * l + sum_j exp(x_j - m_next)
        acc    = exp(m - m_next) * acc + sum_j exp(x_j - m_next) v_j
    and finally O = acc / l, LSE = m + ln l.
    """
    Nq, Nkv = q.shape[0], k.shape[0]
    Dv = v.shape[1]
    m = np.full(Nq, -np.inf)
    l = np.zeros(Nq)
    acc = np.zeros((Nq, Dv))
    rows = np.arange(Nq)
    for c0 in range(0, Nkv, block):
        c1 = min(Nkv, c0 + block)
        x = scale * (q @ k[c0:c1].T)
        if causal:
            vis = np.arange(c0, c1)[None, :] <= (rows[:, None] + (Nkv - Nq))
            x = np.where(vis, x, -np.inf)
        m_blk = x.max(axis=1)
        m_next = np.maximum(m, m_blk)
        live = np.isfinite(m_next)
        mn0 = np.where(live, m_next, 0.0)
        alpha = np.where(np.isfinite(m), np.exp(m - mn0), 0.0)
        p = np.exp(x - mn0[:, None])
        l = alpha * l + p.sum(axis=1)
        acc = alpha[:, None] * acc + p @ v[c0:c1]
        m = m_next
    live = np.isfinite(m)
    l1 = np.where(live, l, 1.0)
    O = np.where(live[:, None], acc / l1[:, None], 0.0)
    LSE = np.where(live, np.where(live, m, 0.0) + np.log(l1), -np.inf)
    return O, LSE


# ---------------------------------------------------------------------------
# merging partial results over disjoint key ranges (split-KV combine)

def lse_merge(parts):
    """Merge partial (O_s, LSE_s) pairs computed over disjoint key ranges of
    the same query rows: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
    Parts whose LSE is -inf (no visible key in that range) contribute nothing."""
    lses = np.stack([np.asarray(p[1], dtype=np.float64) for p in parts])   # [S, r]
    Os = np.stack([np.asarray(p[0], dtype=np.float64) for p in parts])     # [S, r, D]
    mx = lses.max(axis=0)
    live = np.isfinite(mx)
    mx0 = np.where(live, mx, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - mx0[None, :]), 0.0)
    tot = w.sum(axis=0)
    tot1 = np.where(live, tot, 1.0)
    LSE = np.where(live, mx0 + np.log(tot1), -np.inf)
    O = np.where(live[:, None], (w[:, :, None] * Os).sum(axis=0) / tot1[:, None], 0.0)
    return O, LSE


# ---------------------------------------------------------------------------
# backward: the gradient of the forward definition

def attention_backward_head(q, k, v, do, scale, causal, mask=None):
    """Gradients of one head's O with respect to q, k and v, given the
    upstream gradient dO [Nq, Dv] of the output.

    With P the row softmax of S = scale * Q K^T (+ mask, causal -inf) and
    O = P V, the chain rule through the row softmax gives
        dV = P^T dO
        dP = dO V^T
        Delta_i = sum_j P_ij dP_ij  (= sum_d dO_id O_id)
        dS = P * (dP - Delta)        (elementwise, Delta broadcast over j)
        dQ = scale * dS K,   dK = scale * dS^T Q.
    Masked entries have P = 0 and receive no gradient; rows with no visible
    key contribute nothing.  Returns (dq [Nq, D], dk [Nkv, D], dv [Nkv, Dv]).
    """
    P = probs_head(q, k, scale, causal, None, mask)
    O = P @ v
    dV = P.T @ do
    dP = do @ v.T
    delta = (do * O).sum(axis=1)
    dS = P * (dP - delta[:, None])
    return scale * (dS @ k), scale * (dS.T @ q), dV


def attention_backward(q, k, v, do, scale, causal, mask=None):
    """Batched gradients: q and do [B, Hq, Nq, D], k and v [B, Hkv, Nkv, D],
    mask (optional) broadcastable to [B, Hq, Nq, Nkv].  A key/value head
    shared by a GQA group of query heads receives the sum of their gradients.
    Returns (dq, dk, dv) in float64 with the shapes of q, k and v."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    M = None if mask is None else np.broadcast_to(np.asarray(mask, dtype=np.float64), (B, Hq, Nq, Nkv))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            kv = kv_head_of(h, Hq, Hkv)
            gq, gk, gv = attention_backward_head(q[b, h], k[b, kv], v[b, kv], do[b, h], scale, causal,
                                                 None if M is None else M[b, h])
            dq[b, h] = gq
            dk[b, kv] += gk
            dv[b, kv] += gv
    return dq, dk, dv


def attention_backward_sampled(q, k, v, do, scale, causal, rows, keys, block: int = 1024):
    """Chosen entries of one head's gradients, for heads too long to form
    N x N matrices: dq at query rows `rows` and the head's contribution to
    dk, dv at keys `keys`, by the formulas of attention_backward_head (the
    chain rule through the row softmax).  P is formed `block` query rows at
    a time (probs_head on those rows), so memory stays at block x Nkv; each
    row block adds its terms of dV[keys] = sum_i P_i,keys dO_i and
    dK[keys] = scale sum_i dS_i,keys Q_i, with Delta_i = dO_i . O_i and
    O_i = sum_j P_ij V_j of its own rows.
    Returns (dq [len(rows), D], dk [len(keys), D], dv [len(keys), Dv])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    keys = np.asarray(keys, dtype=np.int64)
    Nq = q.shape[0]
    dq = np.zeros((len(rows), q.shape[1]))
    dk = np.zeros((len(keys), k.shape[1]))
    dv = np.zeros((len(keys), v.shape[1]))
    for r0 in range(0, Nq, block):
        idx = np.arange(r0, min(Nq, r0 + block))
        P = probs_head(q, k, scale, causal, idx)          # [b, Nkv]
        delta = (do[idx] * (P @ v)).sum(axis=1)            # Delta_i = dO_i . O_i
        Pk = P[:, keys]
        dSk = Pk * (do[idx] @ v[keys].T - delta[:, None])  # dS at the chosen keys
        dv += Pk.T @ do[idx]
        dk += scale * (dSk.T @ q[idx])
        sel = np.nonzero((rows >= idx[0]) & (rows <= idx[-1]))[0]
        for s in sel:                                       # dQ rows of this block
            i = rows[s] - r0
            dS_row = P[i] * (do[rows[s]] @ v.T - delta[i])
            dq[s] = scale * (dS_row @ k)
    return dq, dk, dv
