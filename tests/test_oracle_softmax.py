"""The FP64 row-softmax oracle against what the pages and mathematics fix.

P3 "Worked example" (outputs, normalizer), torch.softmax / logsumexp in
float64, rows summing to one, the online pair of P3 "Step 2" on 1,000
seeded random vectors (< 1e-12, the page's figure), scores of magnitude 1e4
(finite; the naive form overflows), and planted mutants of the C source.
"""
import math
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
from oracle import recurrence as rec
import oracle_pins as P


def pin_sm_worked_example(orc):
    g = P.golden("worked_example.json")
    tol = 0.5 * 10.0 ** (-g["decimals"])
    y, lse = orc.softmax_rows(np.array([g["vector"]], np.float32))
    assert np.all(np.abs(y[0] - np.array(g["outputs"])) <= tol)
    m, l = g["pairs_after_each_element"][-1]
    assert abs(math.exp(lse[0] - m) - l) <= tol


def pin_sm_library(orc):
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((37, 513)) * rng.uniform(0.1, 20, size=(37, 1))).astype(np.float32)
    y, lse = orc.softmax_rows(x)
    t = torch.from_numpy(x).double()
    assert np.abs(torch.softmax(t, dim=1).numpy() - y).max() <= 8e-15   # a few ulps of 1
    assert np.abs(torch.logsumexp(t, dim=1).numpy() - lse).max() <= 1e-12
    assert np.abs(y.sum(axis=1) - 1).max() <= 1e-13


def pin_sm_online_pairs(orc):
    claim = P.golden("page_error_claims.json")["online_vs_safe_random_vectors"]
    rng = np.random.default_rng(2018)
    worst = 0.0
    for _ in range(claim["n_vectors"] // 50):
        n = int(rng.integers(1, 300))
        xs = (rng.standard_normal((50, n)) * rng.uniform(0.1, 30)).astype(np.float32)
        y, lse = orc.softmax_rows(xs)
        for r in range(50):
            pair = rec.online_normalizer(xs[r])[-1]
            worst = max(worst, float(np.abs(np.array(rec.second_pass(xs[r], pair)) - y[r]).max()))
            worst = max(worst, abs(pair[0] + math.log(pair[1]) - lse[r]) / max(1.0, abs(lse[r])))
    assert worst < claim["max_abs_difference"]


def pin_sm_large_scores(orc):
    rng = np.random.default_rng(22)
    for sign in (1.0, -1.0):
        x = (sign * 1e4 + rng.standard_normal((4, 1000)) * 3).astype(np.float32)
        y, lse = orc.softmax_rows(x)
        assert np.all(np.isfinite(y)) and np.all(np.isfinite(lse))
        assert np.abs(y.sum(axis=1) - 1).max() <= 1e-13
        with np.errstate(over="ignore", invalid="ignore", under="ignore"):
            naive = np.exp(x.astype(np.float64)) / np.exp(x.astype(np.float64)).sum(1, keepdims=True)
        assert not np.all(np.isfinite(naive))


def pin_sm_masked_entries(orc):
    """-inf entries get weight 0 (torch agrees); an all -inf row gives 0 and
    lse = -inf, no NaN."""
    rng = np.random.default_rng(23)
    x = rng.standard_normal((3, 40)).astype(np.float32)
    x[0, ::3] = -np.inf
    x[2, :] = -np.inf
    y, lse = orc.softmax_rows(x)
    t = torch.from_numpy(x[:2]).double()
    assert np.abs(torch.softmax(t, dim=1).numpy() - y[:2]).max() <= 8e-15
    assert np.all(y[0, ::3] == 0)
    assert np.all(y[2] == 0) and lse[2] == -np.inf and not np.isnan(y).any()


SM_PINS = [pin_sm_worked_example, pin_sm_library, pin_sm_online_pairs, pin_sm_large_scores,
           pin_sm_masked_entries]


@pytest.mark.parametrize("pin", SM_PINS, ids=lambda f: f.__name__)
def test_softmax_pin(orc, pin):
    pin(orc)


SM_MUTANTS = [
    ("max not taken", "if ((double)xr[i] > mx) mx = (double)xr[i];",
     "if ((double)xr[i] > mx) mx = 0.0;"),
    ("normalizer sign", "for (long long i = 0; i < n; ++i) sum += exp((double)xr[i] - mx);",
     "for (long long i = 0; i < n; ++i) sum += exp(mx - (double)xr[i]);"),
    ("output not normalized", "yr[i] = exp((double)xr[i] - mx) / sum;",
     "yr[i] = exp((double)xr[i] - mx);"),
    ("lse without max", "lse[r] = mx + log(sum);", "lse[r] = log(sum);"),
    ("row stride", "const float* xr = x + r * n;", "const float* xr = x + r;"),
]


@pytest.mark.parametrize("name,old,new", SM_MUTANTS, ids=[m[0] for m in SM_MUTANTS])
def test_softmax_mutant_fails_a_pin(name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, old
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "m.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        mut = oracle.Oracle(oracle.compile_oracle(path, path[:-2] + ".so", force=True))
        failed = []
        for pin in SM_PINS:
            try:
                with np.errstate(all="ignore"):
                    pin(mut)
            except Exception:   # noqa: BLE001
                failed.append(pin.__name__)
        assert failed, "mutant %r passed every pin" % name
