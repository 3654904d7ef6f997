"""The FP64 backward oracle against independent facts (CPU only).

1. Central finite differences of the FP64 blockwise forward in
   ``oracle/recurrence.py`` (pinned by the forward pins) for L = sum(dO * O).
2. torch autograd through scaled_dot_product_attention in float64.
3. Shift invariances of softmax: sum_j dK_j = 0 and sum_j dV_j = sum of dO
   over rows that see a key; a closed form (one visible key per row: dQ =
   dK = 0, dV = dO); rows with no visible key give zero gradients.
4. Planted mutants of the backward source each fail at least one pin.
"""
import math
import types

import numpy as np
import pytest
import torch

import oracle.backward as OB
from oracle import recurrence as rec


def _inputs(seed, B, H, Nq, Nk, d, scale_q=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, Nq, d)) * scale_q
    k = rng.standard_normal((B, H, Nk, d))
    v = rng.standard_normal((B, H, Nk, d))
    do = rng.standard_normal((B, H, Nq, d))
    return q, k, v, do


def _loss(q, k, v, do, scale, mask_kind, window, Lk):
    causal = bool(mask_kind & (OB.MASK_CAUSAL | OB.MASK_WINDOW))
    win = window if mask_kind & OB.MASK_WINDOW else None
    O, _ = rec.tile_blocks(q, k, v, scale, q0=0, Bc=3, causal=causal, window=win, Lk=Lk)
    return float((do * O).sum())


# ------------------------------------------------------------------- pins
def pin_finite_differences(bwd):
    eps = 1e-6
    for (mask_kind, window, L, seed) in [(0, 0, None, 1), (OB.MASK_CAUSAL, 0, None, 2),
                                         (OB.MASK_WINDOW | OB.MASK_PADDING, 3, 6, 3)]:
        q, k, v, do = _inputs(seed, 1, 1, 6, 7, 4)
        Lk = 7 if L is None else L
        sl = None if L is None else np.array([L])
        dq, dk, dv = bwd(q, k, v, do, 0.5, mask_kind, window, sl)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for idx in np.ndindex(x.shape[2:]):
                xp, xm = x.copy(), x.copy()
                xp[(0, 0) + idx] += eps
                xm[(0, 0) + idx] -= eps
                args_p = {"q": q, "k": k, "v": v}
                args_m = dict(args_p)
                args_p[name], args_m[name] = xp, xm
                fp = _loss(args_p["q"][0, 0], args_p["k"][0, 0], args_p["v"][0, 0], do[0, 0], 0.5,
                           mask_kind, window, Lk)
                fm = _loss(args_m["q"][0, 0], args_m["k"][0, 0], args_m["v"][0, 0], do[0, 0], 0.5,
                           mask_kind, window, Lk)
                fd = (fp - fm) / (2 * eps)
                assert abs(fd - g[(0, 0) + idx]) <= 1e-7, (name, idx, fd, g[(0, 0) + idx])


def pin_torch_autograd(bwd):
    for (mask_kind, window, seqlens, seed) in [(0, 0, None, 4), (OB.MASK_CAUSAL, 0, None, 5),
                                               (OB.MASK_WINDOW, 4, None, 6),
                                               (OB.MASK_PADDING, 0, [9, 20], 7)]:
        B, H, Nq, Nk, d = 2, 2, 17, 20, 8
        q, k, v, do = _inputs(seed, B, H, Nq, Nk, d)
        scale = 1 / math.sqrt(d)
        dq, dk, dv = bwd(q, k, v, do, scale, mask_kind, window, seqlens)
        for b in range(B):
            Lk = Nk if seqlens is None else seqlens[b]
            mask = torch.from_numpy(np.array(OB.visible_mask(Nq, Nk, mask_kind, window, Lk)))
            tq, tk, tv = (torch.tensor(x[b], requires_grad=True) for x in (q, k, v))
            out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                                                   scale=scale)
            out.backward(torch.from_numpy(do[b]))
            assert np.abs(tq.grad.numpy() - dq[b]).max() <= 1e-12
            assert np.abs(tk.grad.numpy() - dk[b]).max() <= 1e-12
            assert np.abs(tv.grad.numpy() - dv[b]).max() <= 1e-12


def pin_invariants(bwd):
    q, k, v, do = _inputs(8, 2, 3, 19, 23, 8, scale_q=2.0)
    sl = np.array([23, 11])
    for mask_kind, window in [(0, 0), (OB.MASK_CAUSAL, 0), (OB.MASK_WINDOW | OB.MASK_PADDING, 5)]:
        dq, dk, dv = bwd(q, k, v, do, 0.3, mask_kind, window, sl)
        for b in range(2):
            Lk = int(sl[b]) if mask_kind & OB.MASK_PADDING else 23
            rows = OB.visible_mask(19, 23, mask_kind, window, Lk).any(axis=1)
            for h in range(3):
                assert np.abs(dk[b, h].sum(axis=0)).max() <= 1e-12
                assert np.abs(dv[b, h].sum(axis=0) - do[b, h][rows].sum(axis=0)).max() <= 1e-12


def pin_closed_forms(bwd):
    q, k, v, do = _inputs(9, 1, 2, 9, 9, 4)
    dq, dk, dv = bwd(q, k, v, do, 0.5, OB.MASK_WINDOW, 1, None)   # one key per row
    assert np.abs(dq).max() <= 1e-14 and np.abs(dk).max() <= 1e-14
    assert np.abs(dv - do).max() <= 1e-14
    dq, dk, dv = bwd(q, k, v, do, 0.5, OB.MASK_PADDING, 0, np.array([0]))  # no visible key
    assert np.all(dq == 0) and np.all(dk == 0) and np.all(dv == 0)


PINS = [pin_finite_differences, pin_torch_autograd, pin_invariants, pin_closed_forms]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin):
    pin(OB.attention_backward)


MUTANTS = [
    ("dropped softmax-jacobian term", "dS = P * (dP - rs)", "dS = P * dP"),
    ("wrong sign", "dS = P * (dP - rs)", "dS = P * (dP + rs)"),
    ("missing scale in dq", "dq[b, h] = scale * (dS @ k[b, h])", "dq[b, h] = dS @ k[b, h]"),
    ("dk from dO instead of Q", "dk[b, h] = scale * (dS.T @ q[b, h])",
     "dk[b, h] = scale * (dS.T @ do[b, h])"),
    ("dv from dP", "dV = P.T @ do[b, h]", "dV = dP.T @ do[b, h]"),
    ("dP with k", "dP = do[b, h] @ v[b, h].T", "dP = do[b, h] @ k[b, h].T"),
    ("row sum over columns", "rs = (P * dP).sum(axis=1, keepdims=True)",
     "rs = (P * dP).sum(axis=0, keepdims=True)"),
    ("causal off by one", "vis = vis & (j <= i)", "vis = vis & (j < i)"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_backward_mutant_fails_a_pin(name, old, new):
    src = open(OB.__file__).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_backward_mutant")
    exec(compile(src.replace(old, new), "mutant", "exec"), mod.__dict__)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod.attention_backward)
        except Exception:   # noqa: BLE001
            failed.append(pin.__name__)
    assert failed, "mutant %r passed every pin" % name
