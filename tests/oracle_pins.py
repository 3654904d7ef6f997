"""Pins for the FP64 oracle: facts fixed by the pages or by mathematics,
each independent of the oracle's own code.

Every pin is a function ``pin_*(orc)`` that raises AssertionError when the
oracle `orc` (an ``oracle.Oracle``) disagrees. ``test_oracle_pins.py`` runs
them on the real oracle, and runs them again on planted mutants of the C
source, each of which must fail at least one pin.

Pages cited:
  P1 "Derive online softmax, prove it is exact, and explain why it makes
     FlashAttention fast without reducing FLOPs" (inferenceinterviews.com)
  P2 "Implement online softmax for a whole tile of queries, not one query,
     and write the rescaling step in matrix form" (inferenceinterviews.com)
  P3 "Online softmax" (interview.clozo.ai/blog/online-softmax.html)
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import torch

from oracle import MASK_CAUSAL, MASK_PADDING, MASK_WINDOW
from oracle import recurrence as rec

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        return json.load(f)


def _softmax_by_attention(orc, xs_list):
    """Softmax of several vectors through the attention oracle: one batch
    entry per vector, query e_0, key j = x_j e_0, values = identity rows,
    scale 1, keys past each vector's length removed by the padding mask.
    Then o = softmax(x) and lse = log sum exp(x)."""
    n = max(len(x) for x in xs_list)
    B = len(xs_list)
    q = np.zeros((B, 1, 1, n), np.float32)
    q[:, 0, 0, 0] = 1.0
    k = np.zeros((B, 1, n, n), np.float32)
    v = np.zeros((B, 1, n, n), np.float32)
    for b, xs in enumerate(xs_list):
        k[b, 0, :len(xs), 0] = xs
        v[b, 0] = np.eye(n, dtype=np.float32)
    lens = np.array([len(x) for x in xs_list], np.int32)
    o, lse = orc.attention(q, k, v, 1.0, MASK_PADDING, 0, lens)
    return o[:, 0, 0, :], lse[:, 0, 0]


# ------------------------------------------------------------------ P3 example
def pin_worked_example_attention(orc):
    """P3 "Worked example": softmax([2, 1, 3, 0.5]) = .2321 .0854 .6308 .0518
    (4 decimals, sum 1); the normalizer referenced to the max 3 is 1.5853."""
    g = golden("worked_example.json")
    tol = 0.5 * 10.0 ** (-g["decimals"])
    o, lse = _softmax_by_attention(orc, [g["vector"]])
    assert np.all(np.abs(o[0, :4] - np.array(g["outputs"])) <= tol), o[0]
    assert abs(o[0].sum() - g["outputs_sum"]) <= 1e-15
    m, l = g["pairs_after_each_element"][-1]
    assert abs(math.exp(lse[0] - m) - l) <= tol, lse


def pin_worked_example_recurrence(orc):
    """P3 "Worked example" table and merge paragraph, against recurrence.py
    (does not use `orc`: pins the streaming cross-check itself)."""
    g = golden("worked_example.json")
    tol = 0.5 * 10.0 ** (-g["decimals"])
    pairs = rec.online_normalizer(g["vector"])
    for (m, l), (gm, gl) in zip(pairs, g["pairs_after_each_element"]):
        assert m == gm and abs(l - gl) <= tol, (m, l, gm, gl)
    outs = rec.second_pass(g["vector"], pairs[-1])
    assert all(abs(a - b) <= tol for a, b in zip(outs, g["outputs"]))
    mg = g["merge"]
    left = rec.online_normalizer(mg["left_block"])[-1]
    right = rec.online_normalizer(mg["right_block"])[-1]
    assert abs(left[1] - mg["left_pair"][1]) <= tol and left[0] == mg["left_pair"][0]
    assert abs(right[1] - mg["right_pair"][1]) <= tol and right[0] == mg["right_pair"][0]
    merged = rec.pair_merge(left, right)
    assert merged[0] == mg["merged_pair"][0]
    assert abs(merged[1] - mg["merged_pair"][1]) <= tol


# ---------------------------------------------------------- 50-digit brute force
def _visible_bruteforce(i, j, Lk, mask_kind, window):
    ok = j < Lk
    if mask_kind & (MASK_CAUSAL | MASK_WINDOW):
        ok = ok and j <= i
    if mask_kind & MASK_WINDOW:
        ok = ok and j > i - window
    return ok


def _exact_attention_decimal(q, k, v, scale, mask_kind, window, seqlens):
    getcontext().prec = 50
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    sc = Decimal(repr(scale))
    for b in range(B):
        Lk = Nk if seqlens is None else int(seqlens[b])
        for h in range(H):
            for i in range(Nq):
                js = [j for j in range(Nk)
                      if _visible_bruteforce(i, j, Lk, mask_kind, window)]
                if not js:
                    lse[b, h, i] = -math.inf
                    continue
                s = {j: sc * sum(Decimal(int(q[b, h, i, t])) * Decimal(int(k[b, h, j, t]))
                                 for t in range(d)) for j in js}
                m = max(s.values())
                e = {j: (s[j] - m).exp() for j in js}
                l = sum(e.values())
                for t in range(d):
                    o[b, h, i, t] = float(sum(e[j] * Decimal(int(v[b, h, j, t]))
                                              for j in js) / l)
                lse[b, h, i] = float(m + l.ln())
    return o, lse


def pin_bruteforce_50_digits(orc):
    """Tiny integer inputs evaluated in 50-digit decimal arithmetic, every
    mask combination including rows with no visible key."""
    rng = np.random.default_rng(1234)
    cases = [
        (0, 0, None), (MASK_CAUSAL, 0, None), (MASK_WINDOW, 2, None),
        (MASK_PADDING, 0, [3, 1]), (MASK_WINDOW | MASK_PADDING, 1, [4, 2]),
        (MASK_PADDING, 0, [0, 2]), (MASK_CAUSAL | MASK_PADDING, 0, [2, 4]),
    ]
    for mask_kind, window, seqlens in cases:
        q = rng.integers(-3, 4, size=(2, 2, 3, 3)).astype(np.float32)
        k = rng.integers(-3, 4, size=(2, 2, 4, 3)).astype(np.float32)
        v = rng.integers(-3, 4, size=(2, 2, 4, 3)).astype(np.float32)
        sl = None if seqlens is None else np.array(seqlens, np.int32)
        o, lse = orc.attention(q, k, v, 0.5, mask_kind, window, sl)
        eo, else_ = _exact_attention_decimal(q, k, v, 0.5, mask_kind, window, sl)
        assert np.all(np.abs(o - eo) <= 1e-15 * np.maximum(1, np.abs(eo))), (mask_kind, o, eo)
        fin = np.isfinite(else_)
        assert np.array_equal(fin, np.isfinite(lse)), (mask_kind, lse, else_)
        assert np.all(np.abs(lse[fin] - else_[fin]) <= 1e-14 * np.maximum(1, np.abs(else_[fin])))
        assert np.all(lse[~fin] == -np.inf)


# ------------------------------------------------------- library special case
def _bool_mask(Nq, Nk, mask_kind, window, Lk):
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    m = j < Lk
    if mask_kind & (MASK_CAUSAL | MASK_WINDOW):
        m = m & (j <= i)
    if mask_kind & MASK_WINDOW:
        m = m & (j > i - window)
    return np.broadcast_to(m, (Nq, Nk))


def pin_library_sdpa(orc):
    """torch's scaled_dot_product_attention on the CPU in float64, and
    torch.logsumexp of the masked scores, agree with the oracle to 1e-12
    (rows with no visible key excluded: conventions differ there)."""
    rng = np.random.default_rng(7)
    for (B, H, Nq, Nk, d, mask_kind, window, seqlens) in [
        (2, 3, 17, 29, 16, 0, 0, None),
        (1, 2, 40, 40, 32, MASK_CAUSAL, 0, None),
        (2, 2, 33, 33, 8, MASK_WINDOW, 5, None),
        (3, 1, 20, 26, 24, MASK_PADDING, 0, [26, 7, 13]),
        (2, 2, 30, 30, 16, MASK_WINDOW | MASK_PADDING, 9, [30, 21]),
    ]:
        q = rng.standard_normal((B, H, Nq, d)).astype(np.float32)
        k = rng.standard_normal((B, H, Nk, d)).astype(np.float32)
        v = rng.standard_normal((B, H, Nk, d)).astype(np.float32)
        scale = 1.0 / math.sqrt(d)
        sl = None if seqlens is None else np.array(seqlens, np.int32)
        o, lse = orc.attention(q, k, v, scale, mask_kind, window, sl)
        for b in range(B):
            Lk = Nk if sl is None else int(sl[b])
            mask = torch.from_numpy(np.array(_bool_mask(Nq, Nk, mask_kind, window, Lk)))
            rows = mask.any(dim=1)
            tq = torch.from_numpy(q[b]).double()
            tk = torch.from_numpy(k[b]).double()
            tv = torch.from_numpy(v[b]).double()
            ref = torch.nn.functional.scaled_dot_product_attention(
                tq, tk, tv, attn_mask=mask, scale=scale)
            scores = (tq @ tk.transpose(-1, -2)) * scale
            scores = scores.masked_fill(~mask, float("-inf"))
            ref_lse = torch.logsumexp(scores, dim=-1)
            got = torch.from_numpy(o[b])
            assert torch.all((got[:, rows] - ref[:, rows]).abs() <= 1e-12), (mask_kind, b)
            got_lse = torch.from_numpy(lse[b])
            assert torch.all((got_lse[:, rows] - ref_lse[:, rows]).abs() <= 1e-12), (mask_kind, b)


# ------------------------------------------------------------- closed forms
def pin_uniform_scores(orc):
    """q = 0 makes every visible score 0: o is the mean of the visible value
    rows and lse = log(number of visible keys)."""
    rng = np.random.default_rng(11)
    B, H, N, d = 2, 2, 23, 8
    q = np.zeros((B, H, N, d), np.float32)
    k = rng.standard_normal((B, H, N, d)).astype(np.float32)
    v = rng.standard_normal((B, H, N, d)).astype(np.float32)
    sl = np.array([23, 10], np.int32)
    for mask_kind, window in [(0, 0), (MASK_CAUSAL, 0), (MASK_WINDOW, 5),
                              (MASK_PADDING, 0), (MASK_WINDOW | MASK_PADDING, 4)]:
        o, lse = orc.attention(q, k, v, 0.3, mask_kind, window, sl)
        for b in range(B):
            Lk = int(sl[b]) if mask_kind & MASK_PADDING else N
            vis = _bool_mask(N, N, mask_kind, window, Lk)
            for i in range(N):
                js = np.nonzero(vis[i])[0]
                if len(js) == 0:
                    continue
                want = v[b][:, js, :].astype(np.float64).mean(axis=1)
                assert np.max(np.abs(o[b, :, i] - want)) <= 1e-15, (mask_kind, b, i)
                assert np.max(np.abs(lse[b, :, i] - math.log(len(js)))) <= 1e-15


def pin_single_visible_key(orc):
    """A row that sees exactly one key returns that key's value row, and its
    lse is that one score."""
    rng = np.random.default_rng(12)
    B, H, N, d = 2, 3, 9, 16
    q = rng.standard_normal((B, H, N, d)).astype(np.float32)
    k = rng.standard_normal((B, H, N, d)).astype(np.float32)
    v = rng.standard_normal((B, H, N, d)).astype(np.float32)
    scale = 0.25
    # causal: row 0 sees key 0 only
    o, lse = orc.attention(q, k, v, scale, MASK_CAUSAL)
    s00 = scale * np.einsum("bhd,bhd->bh", q[:, :, 0].astype(np.float64), k[:, :, 0].astype(np.float64))
    assert np.max(np.abs(o[:, :, 0] - v[:, :, 0])) <= 1e-15
    assert np.max(np.abs(lse[:, :, 0] - s00)) <= 1e-14
    # padding with one key: every row sees key 0
    o, lse = orc.attention(q, k, v, scale, MASK_PADDING, 0, np.array([1, 1], np.int32))
    assert np.max(np.abs(o - v[:, :, :1])) <= 1e-15
    # window of one key: row i sees key i
    o, lse = orc.attention(q, k, v, scale, MASK_WINDOW, 1)
    sii = scale * np.einsum("bhid,bhid->bhi", q.astype(np.float64), k.astype(np.float64))
    assert np.max(np.abs(o - v)) <= 1e-15
    assert np.max(np.abs(lse - sii)) <= 1e-14


def pin_fully_masked_rows(orc):
    """Rows with no visible key: o = 0, lse = -inf, and no NaN anywhere (the
    empty-row reading; P2's m_ref guard paragraph gives the per-block case)."""
    rng = np.random.default_rng(13)
    B, H, N, d = 2, 2, 12, 8
    q = rng.standard_normal((B, H, N, d)).astype(np.float32)
    k = rng.standard_normal((B, H, N, d)).astype(np.float32)
    v = rng.standard_normal((B, H, N, d)).astype(np.float32)
    o, lse = orc.attention(q, k, v, 0.3, MASK_PADDING, 0, np.array([0, 5], np.int32))
    assert np.all(o[0] == 0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(o[1])) and np.all(np.isfinite(lse[1]))
    # window 3 over 5 keys: rows i >= 5 + 3 - 1 = 7 see nothing
    o, lse = orc.attention(q, k, v, 0.3, MASK_WINDOW | MASK_PADDING, 3,
                           np.array([5, 5], np.int32))
    assert not np.any(np.isnan(o)) and not np.any(np.isnan(lse))
    assert np.all(o[:, :, 7:] == 0) and np.all(lse[:, :, 7:] == -np.inf)
    assert np.all(np.isfinite(lse[:, :, :7]))


# ------------------------------------------------ P1 and P2 exactness claims
def pin_single_query_blocks(orc):
    """P1 "A strong answer" test paragraph: one query, 1,000 keys in blocks of
    128 (partial last block) equals the direct softmax to ~1e-16; at score
    magnitudes ~1e4 both stay finite and agree exactly, while a softmax
    without the max subtraction returns NaN."""
    claim = golden("page_error_claims.json")["single_query_blocks"]
    rng = np.random.default_rng(0)
    N, d = claim["n_keys"], 64
    q = rng.standard_normal(d).astype(np.float32)
    K = rng.standard_normal((N, d)).astype(np.float32)
    V = rng.standard_normal((N, d)).astype(np.float32)
    scale = 1.0 / math.sqrt(d)
    o, lse = orc.attention(q[None, None, None], K[None, None], V[None, None], scale)
    ob, lseb = rec.single_query_blocks(q, K, V, scale, claim["block"])
    # a few ulps of the output magnitude: the page prints 1e-16
    assert np.max(np.abs(o[0, 0, 0] - ob)) <= 8 * claim["max_abs_error_ordinary_scores"]
    assert abs(lse[0, 0, 0] - lseb) <= 1e-14
    for sign in (1.0, -1.0):
        # scores of magnitude ~1e4 (both signs: all-negative rows too)
        qb = (q * 0 + 1.0).astype(np.float32)
        Kb = (sign * (1e4 * math.sqrt(d) / d) + rng.standard_normal((N, d)) * 2.0).astype(np.float32)
        o2, lse2 = orc.attention(qb[None, None, None], Kb[None, None], V[None, None], scale)
        ob2, lseb2 = rec.single_query_blocks(qb, Kb, V, scale, claim["block"])
        assert np.all(np.isfinite(o2)) and np.isfinite(lse2).all()
        assert np.max(np.abs(o2[0, 0, 0] - ob2)) <= max(claim["max_abs_error_scores_1e4"], 1e-15)
        s = scale * (Kb.astype(np.float64) @ qb.astype(np.float64))
        assert abs(abs(s).mean() - 1e4) < 200
        with np.errstate(over="ignore", invalid="ignore", under="ignore"):
            naive = np.exp(s) / np.exp(s).sum()
        assert not np.all(np.isfinite(naive))


def pin_query_tile(orc):
    """P2 "A strong answer" test paragraph: query tile Br=128, d=64, key
    blocks Bc=64 over N=1,000 keys equals the direct softmax, non-causal,
    causal at tile offsets 0, 300, 872, and with the largest scores planted
    in the last five keys; the page reports max error < 5.2e-15."""
    claim = golden("page_error_claims.json")["query_tile"]
    rng = np.random.default_rng(1)
    N, Br, d, Bc = claim["n_keys"], claim["Br"], claim["d"], claim["Bc"]
    scale = 1.0 / math.sqrt(d)
    K = rng.standard_normal((N, d)).astype(np.float32)
    V = rng.standard_normal((N, d)).astype(np.float32)
    Qt = rng.standard_normal((Br, d)).astype(np.float32)
    Kp = K.copy()
    Kp[N - 5:, d - 1] += 10.0 / scale
    Qp = Qt.copy()
    Qp[:, d - 1] = 1.0
    worst = 0.0
    for (Q, Kx, q0, causal) in [(Qt, K, 0, False), (Qt, K, 0, True), (Qt, K, 300, True),
                                (Qt, K, 872, True), (Qp, Kp, 0, False), (Qp, Kp, 872, True)]:
        Qfull = np.zeros((q0 + Br, d), np.float32)
        Qfull[q0:] = Q
        o, lse = orc.attention(Qfull[None, None], Kx[None, None], V[None, None], scale,
                               MASK_CAUSAL if causal else 0)
        ot, lset = rec.tile_blocks(Q, Kx, V, scale, q0=q0, Bc=Bc, causal=causal)
        worst = max(worst, float(np.max(np.abs(o[0, 0, q0:] - ot))))
        assert np.max(np.abs(lse[0, 0, q0:] - lset)) <= 1e-13
    assert worst < claim["max_abs_error"], worst


def pin_online_vs_safe_vectors(orc):
    """P3 "Worked example": across 1,000 seeded random vectors the online
    pair and the two-pass safe softmax differ by less than 1e-12."""
    claim = golden("page_error_claims.json")["online_vs_safe_random_vectors"]
    rng = np.random.default_rng(2018)
    xs_list = []
    for _ in range(claim["n_vectors"]):
        n = int(rng.integers(1, 48))
        xs_list.append((rng.standard_normal(n) * rng.uniform(0.1, 30)).astype(np.float32))
    o, lse = _softmax_by_attention(orc, xs_list)
    worst = 0.0
    for b, xs in enumerate(xs_list):
        pair = rec.online_normalizer(xs)[-1]
        outs = np.array(rec.second_pass(xs, pair))
        worst = max(worst, float(np.max(np.abs(o[b, :len(xs)] - outs))))
        worst = max(worst, abs(lse[b] - (pair[0] + math.log(pair[1]))) / max(1.0, abs(lse[b])))
    assert worst < claim["max_abs_difference"], worst


# ------------------------------------------------------------- invariants
def pin_invariants(orc):
    """P3 "Step 2": after n elements the normalizer referenced to the max lies
    in [1, n], so max s <= lse <= max s + log n; and the weights of a row sum
    to one (values all ones give o = 1)."""
    rng = np.random.default_rng(14)
    B, H, N, d = 2, 2, 37, 16
    q = (rng.standard_normal((B, H, N, d)) * 3).astype(np.float32)
    k = rng.standard_normal((B, H, N, d)).astype(np.float32)
    ones = np.ones((B, H, N, d), np.float32)
    scale = 0.25
    sl = np.array([37, 19], np.int32)
    for mask_kind, window in [(0, 0), (MASK_CAUSAL, 0), (MASK_WINDOW | MASK_PADDING, 6)]:
        o, lse = orc.attention(q, k, ones, scale, mask_kind, window, sl)
        s = scale * np.einsum("bhid,bhjd->bhij", q.astype(np.float64), k.astype(np.float64))
        for b in range(B):
            Lk = int(sl[b]) if mask_kind & MASK_PADDING else N
            vis = _bool_mask(N, N, mask_kind, window, Lk)
            for i in range(N):
                n = int(vis[i].sum())
                if n == 0:
                    assert np.all(o[b, :, i] == 0)
                    continue
                mx = s[b, :, i][:, vis[i]].max(axis=-1)
                assert np.all(lse[b, :, i] >= mx - 1e-12)
                assert np.all(lse[b, :, i] <= mx + math.log(n) + 1e-12)
                assert np.max(np.abs(o[b, :, i] - 1.0)) <= 1e-14


def pin_merge_of_chunks(orc):
    """P3 "Step 4" and the Flash-Decoding reduction under P3 "Trade-offs and
    edge cases": per-chunk (o_s, lse_s) from the oracle, merged in random
    groupings and split counts, equal the whole-row oracle result."""
    rng = np.random.default_rng(15)
    B, H, N, d = 1, 2, 300, 32
    q = rng.standard_normal((B, H, 1, d)).astype(np.float32)
    k = rng.standard_normal((B, H, N, d)).astype(np.float32)
    v = rng.standard_normal((B, H, N, d)).astype(np.float32)
    scale = 1.0 / math.sqrt(d)
    o_full, lse_full = orc.attention(q, k, v, scale)
    for trial in range(6):
        nsplit = int(rng.integers(1, 12))
        cuts = np.sort(rng.choice(np.arange(1, N), size=nsplit - 1, replace=False)) if nsplit > 1 else []
        bounds = [0, *[int(c) for c in cuts], N]
        parts_o, parts_l = [], []
        for a, b in zip(bounds[:-1], bounds[1:]):
            o_s, l_s = orc.attention(q, k[:, :, a:b], v[:, :, a:b], scale)
            parts_o.append(o_s[0, :, 0])
            parts_l.append(l_s[0, :, 0])
        parts_o = np.stack(parts_o, 1)   # [H, S, d]
        parts_l = np.stack(parts_l, 1)   # [H, S]
        for h in range(H):
            # random binary tree of merges
            items = [(parts_o[h, s], parts_l[h, s]) for s in range(len(bounds) - 1)]
            while len(items) > 1:
                t = int(rng.integers(0, len(items) - 1))
                (oa, la), (ob, lb) = items[t], items[t + 1]
                om, lm = rec.merge_partials(np.stack([oa, ob]), [la, lb])
                items[t:t + 2] = [(om, lm)]
            om, lm = items[0]
            assert np.max(np.abs(om - o_full[0, h, 0])) <= 1e-14
            assert abs(lm - lse_full[0, h, 0]) <= 1e-13


ALL_PINS = [
    pin_worked_example_attention,
    pin_worked_example_recurrence,
    pin_bruteforce_50_digits,
    pin_library_sdpa,
    pin_uniform_scores,
    pin_single_visible_key,
    pin_fully_masked_rows,
    pin_single_query_blocks,
    pin_query_tile,
    pin_online_vs_safe_vectors,
    pin_invariants,
    pin_merge_of_chunks,
]
