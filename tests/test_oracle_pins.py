"""The FP64 oracle against what the pages and mathematics fix (CPU only).

1. Every pin in ``oracle_pins.ALL_PINS`` passes on the oracle.
2. Mistakes the pages name, planted in copies of the streaming recurrence,
   are caught (rescaling l but not the accumulator; m started at 0; no m_ref
   guard under a window).
3. Planted mutants of the C oracle (dropped term, wrong sign, wrong index,
   transposed operand, off-by-one masks) each fail at least one pin.
"""
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import recurrence as rec
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


# ------------------------------------------------- named mistakes, planted
def _blocks_rescale_l_only(q, K, V, scale, block):
    """Copy of the single-query recurrence with the mistake P1 "Common
    mistakes" names: l is rescaled but the accumulator is not."""
    m, l = -math.inf, 0.0
    a = np.zeros(V.shape[1])
    for s0 in range(0, K.shape[0], block):
        s = scale * (K[s0:s0 + block] @ q)
        m_new = max(m, float(s.max()))
        r = math.exp(m - m_new) if m != -math.inf else 0.0
        w = np.exp(s - m_new)
        l = r * l + w.sum()
        a = a + w @ V[s0:s0 + block]          # planted: no rescale of a
        m = m_new
    return a / l


def _blocks_m0_zero(q, K, V, scale, block):
    """Copy with m started at 0 instead of -inf (P1 "Common mistakes"): the
    first block's weights are referenced to max(0, block max)."""
    m, l = 0.0, 0.0
    a = np.zeros(V.shape[1])
    for s0 in range(0, K.shape[0], block):
        s = scale * (K[s0:s0 + block] @ q)
        m_new = max(m, float(s.max()))
        r = math.exp(m - m_new)
        w = np.exp(s - m_new)
        l = r * l + w.sum()
        a = r * a + w @ V[s0:s0 + block]
        m = m_new
    return a / l


def test_planted_rescale_l_only_is_caught(orc):
    """Late maxima (largest scores in the last keys) expose it (P1, P2)."""
    rng = np.random.default_rng(3)
    N, d = 1000, 64
    scale = 1 / 8
    q = rng.standard_normal(d).astype(np.float32)
    K = rng.standard_normal((N, d)).astype(np.float32)
    V = rng.standard_normal((N, d)).astype(np.float32)
    q[-1] = 1.0
    K[N - 5:, -1] += 10 / scale
    o, _ = orc.attention(q[None, None, None], K[None, None], V[None, None], scale)
    good = rec.single_query_blocks(q, K, V, scale, 128)[0]
    bad = _blocks_rescale_l_only(q, K, V, scale, 128)
    assert np.max(np.abs(good - o[0, 0, 0])) < 1e-13
    assert np.max(np.abs(bad - o[0, 0, 0])) > 1e-2


def test_planted_m0_zero_is_caught(orc):
    """All-negative scores far below zero (P1 "Common mistakes")."""
    rng = np.random.default_rng(4)
    N, d = 300, 16
    scale = 0.25
    q = np.ones(d, np.float32)
    K = (-(200.0 + rng.standard_normal((N, d)))).astype(np.float32)   # scores about -800
    V = rng.standard_normal((N, d)).astype(np.float32)
    o, _ = orc.attention(q[None, None, None], K[None, None], V[None, None], scale)
    assert np.all(np.isfinite(o))
    with np.errstate(invalid="ignore", divide="ignore", under="ignore"):
        bad = _blocks_m0_zero(q, K, V, scale, 64)
    assert not np.all(np.isfinite(bad)) or np.max(np.abs(bad - o[0, 0, 0])) > 1e-2


def test_planted_missing_guard_is_caught(orc):
    """Under a window a row can see no key in a block while its max is still
    -inf; without the m_ref guard NaN reaches the accumulator (P2)."""
    rng = np.random.default_rng(5)
    N, d, W, Bc = 256, 16, 8, 32
    Q = rng.standard_normal((N, d)).astype(np.float32)
    K = rng.standard_normal((N, d)).astype(np.float32)
    V = rng.standard_normal((N, d)).astype(np.float32)
    o, _ = orc.attention(Q[None, None], K[None, None], V[None, None], 0.25, oracle.MASK_WINDOW, W)
    ot, _ = rec.tile_blocks(Q, K, V, 0.25, Bc=Bc, window=W)
    assert np.max(np.abs(ot - o[0, 0])) < 1e-13
    # planted: reference the weights to m_new itself (no guard)
    m = np.full(N, -np.inf)
    l = np.zeros(N)
    A = np.zeros((N, d))
    qpos = np.arange(N)
    with np.errstate(invalid="ignore"):
        for s0 in range(0, N, Bc):
            kp = np.arange(s0, s0 + Bc)
            S = 0.25 * Q @ K[kp].T
            vis = (kp[None] <= qpos[:, None]) & (kp[None] > qpos[:, None] - W)
            S = np.where(vis, S, -np.inf)
            m_new = np.maximum(m, S.max(1))
            alpha = np.exp(m - m_new)
            P_ = np.exp(S - m_new[:, None])
            l = alpha * l + P_.sum(1)
            A = alpha[:, None] * A + P_ @ V[kp]
            m = m_new
        bad = A / l[:, None]
    assert np.any(np.isnan(bad))


# ------------------------------------------------------- C-source mutants
MUTANTS = [
    ("dropped scale", "s[j] = scale * dot;", "s[j] = dot;"),
    ("max started at 0", "double m = -INFINITY;", "double m = 0.0;"),
    ("wrong sign in normalizer", "if (vis[j]) l += exp(s[j] - m);",
     "if (vis[j]) l += exp(s[j] + m);"),
    ("dropped normalization", "double p = exp(s[j] - m) / l;", "double p = exp(s[j] - m);"),
    ("lse without log", "*lse_out = m + log(l);", "*lse_out = m + l;"),
    ("lse without max", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("transposed key operand",
     "dot += (double)q_row[t] * (double)k_row[t];",
     "dot += (double)q_row[t] * (double)k_head[(long long)t * Nk + j];"),
    ("value row index reversed", "const float* v_row = v_head + j * (long long)d;",
     "const float* v_row = v_head + (Nk - 1 - j) * (long long)d;"),
    ("value column fixed", "o_row[t] += p * (double)v_row[t];",
     "o_row[t] += p * (double)v_row[0];"),
    ("causal off by one", "&& j > i)", "&& j >= i)"),
    ("window off by one", "j <= i - window)", "j < i - window)"),
    ("padding off by one", "if (j >= Lk) return 0;", "if (j > Lk) return 0;"),
    ("batch index from head", "long long b = bh / H;", "long long b = bh % H;"),
    ("key head offset uses Nq", "k + bh * (long long)Nk * d,", "k + bh * (long long)Nq * d,"),
]


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_fails_a_pin(mutant_dir, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, "mutation site not unique: %r" % old
    path = os.path.join(mutant_dir, "m_%d.c" % (abs(hash(name)) % 10 ** 8))
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_oracle(path, path[:-2] + ".so", force=True)
    mut = oracle.Oracle(lib)
    failed = []
    for pin in P.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mut)
        except Exception:   # noqa: BLE001 -- any failure counts as caught
            failed.append(pin.__name__)
    assert failed, "mutant %r passed every pin" % name
