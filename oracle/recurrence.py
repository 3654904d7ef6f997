"""Online-softmax recurrences in FP64 -- TEST INFRASTRUCTURE (cross-checks only).

These functions restate, from the pages' equations, the streaming forms of the
method. They exist to check the direct definition in ``attn_oracle.c`` against
an independently written algorithm that the pages prove equal to it; the CUDA
path never uses them and they never use the CUDA path.

Citations (pages and sections):
  P1 "Derive online softmax, prove it is exact, ..." -- "A strong answer",
     block recurrence for (m, l, a) and the final o = a / l.
  P2 "Implement online softmax for a whole tile of queries ..." -- "A strong
     answer", the query-tile equations for S_j, m', P_j, l', A', alpha, the
     m_ref guard paragraph, and the single diag(l)^-1 at the end.
  P3 "Online softmax" (interview.clozo.ai) -- "Step 2" (element update of the
     pair (m, d); written l here), "Step 3" (second pass), "Step 4" (merge),
     "Worked example".
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = float("-inf")


# ---------------------------------------------------------------- scalar pair
def pair_start():
    """P3 Step 2: the pair starts at (m, l) = (-inf, 0)."""
    return (NEG_INF, 0.0)


def pair_update(pair, x):
    """P3 Step 2: read one element x. The new max is max(m, x); the old sum,
    referenced to the old max, is multiplied by exp(m_old - m_new); the new
    term exp(x - m_new) is added."""
    m_old, l_old = pair
    m_new = max(m_old, x)
    shrink = math.exp(m_old - m_new) if m_old != NEG_INF else 0.0
    return (m_new, l_old * shrink + math.exp(x - m_new))


def pair_merge(a, b):
    """P3 Step 4: merge two pairs. The merged max is the larger one; each sum
    is rescaled to it before adding."""
    (m1, l1), (m2, l2) = a, b
    m = max(m1, m2)
    if m == NEG_INF:
        return (NEG_INF, 0.0)
    t1 = l1 * math.exp(m1 - m) if m1 != NEG_INF else 0.0
    t2 = l2 * math.exp(m2 - m) if m2 != NEG_INF else 0.0
    return (m, t1 + t2)


def online_normalizer(xs):
    """P3 Step 2 over a whole vector; returns the list of pairs after each
    element (the rows of the P3 worked-example table)."""
    pair = pair_start()
    out = []
    for x in xs:
        pair = pair_update(pair, float(x))
        out.append(pair)
    return out


def second_pass(xs, pair):
    """P3 Step 3: outputs exp(x_i - m) / l from the final pair."""
    m, l = pair
    return [math.exp(float(x) - m) / l for x in xs]


# --------------------------------------------------------- one query, blocks
def single_query_blocks(q, K, V, scale, block):
    """P1 "A strong answer": one query, keys in blocks of `block`. Hold the max
    m, the normalizer l and the unnormalised output a; when a block raises the
    max, rescale l and a by exp(m_old - m_new); finish with a / l.
    Returns (o, lse)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    m, l = NEG_INF, 0.0
    a = np.zeros(V.shape[1])
    for start in range(0, K.shape[0], block):
        s = scale * (K[start:start + block] @ q)
        m_new = max(m, float(s.max()))
        r = math.exp(m - m_new) if m != NEG_INF else 0.0
        w = np.exp(s - m_new)
        l = r * l + float(w.sum())
        a = r * a + w @ V[start:start + block]
        m = m_new
    return a / l, m + math.log(l)


# ----------------------------------------------------------- query-tile form
def tile_blocks(Q, K, V, scale, q0=0, Bc=64, causal=False, window=None,
                Lk=None):
    """P2 "A strong answer": a tile of Br queries starting at absolute position
    q0, keys streamed in blocks of Bc. State m, l in R^Br and A in R^{Br x d}.
    Per block: S_j = scale Q K_j^T (masked keys get -inf), m' = max(m,
    rowmax S_j), the guard m_ref = 0 where m' = -inf (P2's paragraph on the
    m_ref guard), alpha = exp(m - m_ref), P_j = exp(S_j - m_ref),
    l' = alpha l + P_j 1, A' = diag(alpha) A + P_j V_j. After the last block,
    O = diag(l)^-1 A. Rows that never saw a key return o = 0, lse = -inf
    (the empty-row reading used throughout).

    Masks follow the oracle's readings: causal j <= i; window i - W < j <= i;
    padding j < Lk. Returns (O [Br,d], lse [Br])."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Br = Q.shape[0]
    N = K.shape[0] if Lk is None else min(int(Lk), K.shape[0])
    m = np.full(Br, NEG_INF)
    l = np.zeros(Br)
    A = np.zeros((Br, V.shape[1]))
    qpos = q0 + np.arange(Br)
    with np.errstate(invalid="ignore"):
        for s0 in range(0, K.shape[0], Bc):
            kpos = np.arange(s0, min(s0 + Bc, K.shape[0]))
            S = scale * (Q @ K[kpos].T)
            vis = kpos[None, :] < N
            if causal or window is not None:
                vis = vis & (kpos[None, :] <= qpos[:, None])
            if window is not None:
                vis = vis & (kpos[None, :] > qpos[:, None] - window)
            S = np.where(vis, S, NEG_INF)
            m_new = np.maximum(m, S.max(axis=1))
            m_ref = np.where(np.isneginf(m_new), 0.0, m_new)
            alpha = np.exp(m - m_ref)
            P = np.exp(S - m_ref[:, None])
            l = alpha * l + P.sum(axis=1)
            A = alpha[:, None] * A + P @ V[kpos]
            m = m_new
    empty = l == 0.0
    O = np.where(empty[:, None], 0.0, A / np.where(empty, 1.0, l)[:, None])
    lse = np.where(empty, NEG_INF,
                   np.where(np.isneginf(m), 0.0, m) + np.log(np.where(empty, 1.0, l)))
    return O, lse


# --------------------------------------------- merge of (o, lse) partials
def merge_partials(o_parts, lse_parts):
    """Merge per-chunk results (o_s normalised, lse_s) into the full-row
    result with the P3 Step 4 rule, as the Flash-Decoding reduction described
    under P3 "Trade-offs and edge cases" does: with m* = max lse_s,
    w_s = exp(lse_s - m*), o = sum w_s o_s / sum w_s, lse = m* + log sum w_s.
    Empty chunks carry lse = -inf and weight 0."""
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    o_parts = np.asarray(o_parts, dtype=np.float64)
    m = lse_parts.max()
    if m == NEG_INF:
        return np.zeros(o_parts.shape[1]), NEG_INF
    w = np.exp(lse_parts - m)
    tot = w.sum()
    return (w[:, None] * o_parts).sum(axis=0) / tot, m + math.log(tot)
