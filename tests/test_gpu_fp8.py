"""E4M3 forward (attn_fwd_fp8) against the FP64 oracle (GPU only).

Both sides see the same real inputs: E4M3 values times power-of-two factors,
exact in FP32. The kernel rounds the attention weights to E4M3 for the P V
product, which is the dominant difference from the exact result; the
tolerance is derived from that rounding.

Derivation. A weight p in [2^-6, 2^8] (the kernel's P is at most 2^8) rounds
to nearest with relative error at most 2^-4 (three mantissa bits); below
2^-6 (subnormal) the absolute error is at most 2^-10. The kernel's P is the
row's weight relative to a reference at or below the final row maximum, so
in units where the maximum weight is 1 every error is at most
delta_j = max(2^-4 p_j, 2^-10). Rounding errors of different keys are
independent and uniform on [-delta_j, delta_j], so the error of output
element t is a sum with standard deviation
    sigma_t = sqrt(sum_j delta_j^2 v_jt^2 / 3) / l,   l = sum_j p_j.
The test allows 6 sigma_t + 2^-8 |o_t| (BF16 output rounding) + 1e-5 (FP32
arithmetic). When a few keys dominate, 6 sigma_t exceeds the worst case
sum_j delta_j |v_jt| / l, so the bound also holds there. The LSE does not
involve the rounded weights: |lse - lse_ref| <= 1e-3, as for BF16.
"""
import math

import numpy as np
import pytest
import torch

from oracle import backward as OB
from online_softmax_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_LSE = 1e-3


def _fp8_inputs(B, H, Nq, Nk, d=128, seed=0, seqlen_range=None, scale_q=1.0):
    x = W.random_inputs(B, H, Nq, Nk, d, dtype=torch.float32, seed=seed,
                        seqlen_range=seqlen_range, scale_q=scale_q)
    out = {"seqlens_k": x["seqlens_k"]}
    for n in ("q", "k", "v"):
        out[n], out["descale_" + n] = W.quantize_e4m3(x[n])
    return out


def _real(x, n):
    """The real input the E4M3 tensor stands for (exact in FP32)."""
    return (x[n].float() * x["descale_" + n]).numpy()


def _run(attn, x, mask_kind=0, window=0):
    sl = x["seqlens_k"]
    o, lse = attn.attn_fwd_fp8(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["descale_q"],
                               x["descale_k"], x["descale_v"], mask_kind=mask_kind, window=window,
                               seqlens_k=None if sl is None else sl.cuda())
    attn.attn_check_device_error()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _bound(qr, kr, vr, scale, mask_kind, window, seqlens, rows):
    """6 sigma_t of the module docstring for the listed flat rows."""
    B, H, Nq, d = qr.shape
    Nk = kr.shape[2]
    out = np.zeros((len(rows), d))
    for n, flat in enumerate(rows):
        i, bh = flat % Nq, flat // Nq
        b, h = bh // H, bh % H
        Lk = Nk if seqlens is None else int(min(max(seqlens[b], 0), Nk))
        vis = OB.visible_mask(Nq, Nk, mask_kind, window, Lk)[i]
        if not vis.any():
            continue
        s = scale * (kr[b, h][vis].astype(np.float64) @ qr[b, h, i].astype(np.float64))
        p = np.exp(s - s.max())
        delta = np.maximum(2.0 ** -4 * p, 2.0 ** -10)
        v = vr[b, h][vis].astype(np.float64)
        out[n] = 6.0 * np.sqrt((delta[:, None] ** 2 * v ** 2).sum(0) / 3.0) / p.sum()
    return out


def _check(o, lse, ro, rl, bound, what=""):
    assert not np.isnan(o).any() and not np.isnan(lse).any(), what
    empty = np.isneginf(rl)
    assert np.array_equal(np.isneginf(lse), empty), (what, "lse -inf pattern differs")
    assert np.all(o[empty] == 0.0), what
    tol = bound + 2.0 ** -8 * np.abs(ro) + 1e-5
    excess = np.abs(o - ro) - tol
    assert excess.max() <= 0, (what, float(np.abs(o - ro).max()), float(tol.min()))
    if (~empty).any():
        assert np.abs(lse[~empty] - rl[~empty]).max() <= TOL_LSE, what


def _compare(attn, orc, x, mask_kind=0, window=0, rows=None, what=""):
    qr, kr, vr = _real(x, "q"), _real(x, "k"), _real(x, "v")
    B, H, Nq, d = qr.shape
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(attn, x, mask_kind, window)
    sl = x["seqlens_k"]
    if rows is None:
        rows = np.arange(B * H * Nq)
    ro, rl = orc.attention(qr, kr, vr, scale, mask_kind, window,
                           None if sl is None else sl.numpy(), rows=rows)
    bound = _bound(qr, kr, vr, scale, mask_kind, window, None if sl is None else sl.numpy(),
                   rows)
    _check(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], ro, rl, bound, what)
    return o, lse


SHAPES = [
    # (B, H, Nq, Nk, mask_kind, window, seqlen_range)
    (1, 2, 300, 1000, 0, 0, None),            # ragged query pair and key block
    (1, 1, 128, 128, 0, 0, None),             # one tile, one block
    (2, 2, 700, 700, W.MASK_CAUSAL, 0, None),
    (2, 3, 520, 900, W.MASK_WINDOW | W.MASK_PADDING, 200, (0, 900)),
    (1, 2, 77, 3000, W.MASK_PADDING, 0, (1, 3000)),
    # causal CTAs walk their key blocks from the diagonal down over many
    # blocks (up to 32 per CTA, past both rings' wrap-around)
    (1, 1, 4096, 4096, W.MASK_CAUSAL, 0, None),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_fwd_fp8_shapes(cuda_lib, orc, shape):
    B, H, Nq, Nk, mk, win, sr = shape
    x = _fp8_inputs(B, H, Nq, Nk, seed=B * 1000 + Nq, seqlen_range=sr)
    _compare(cuda_lib, orc, x, mk, win, what=str(shape))


def test_fwd_fp8_large_scores(cuda_lib, orc):
    """Scores of magnitude ~100 (Q drawn 8x wider): the lazy reference moves
    often and a few keys carry each row."""
    x = _fp8_inputs(1, 2, 256, 1000, seed=7, scale_q=8.0)
    _compare(cuda_lib, orc, x, what="large scores")


def test_fwd_fp8_matches_bf16_path_closely(cuda_lib):
    """Same real inputs through the BF16 kernel: the two agree within the
    E4M3 rounding of the weights (a layout or scale mistake in the 8-bit
    operands would give O(1) differences)."""
    x = _fp8_inputs(1, 4, 512, 2048, seed=3)
    o8, l8 = _run(cuda_lib, x)
    qb, kb, vb = (torch.from_numpy(_real(x, n)).to(torch.bfloat16).cuda() for n in "qkv")
    ob, lb = cuda_lib.attn_fwd(qb, kb, vb)
    ob, lb = ob.float().cpu().numpy(), lb.cpu().numpy()
    assert np.abs(l8 - lb).max() <= 1e-3
    assert np.abs(o8 - ob).max() <= 0.02
    assert np.sqrt(np.mean((o8 - ob) ** 2)) <= 2e-3


def test_fwd_fp8_full_size_prefill_sampled(cuda_lib, orc):
    """The prefill workload (B1 H64 8192^2 d128) stored as E4M3, in the
    benchmark's launch configuration: sampled rows against the oracle."""
    w = W.PREFILL
    x = W.generate_fp8(w)
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([
        np.array([0, 1, 127, 128, 255, 256, w.Nq - 1, w.H * w.Nq - 1]),
        rng.choice(w.B * w.H * w.Nq, 120, replace=False)]))
    o, lse = _compare(cuda_lib, orc, x, rows=rows, what=w.name)
    assert not np.isnan(o).any() and np.isfinite(lse).all()


def test_fwd_fp8_bad_arguments(cuda_lib):
    x = _fp8_inputs(1, 1, 128, 128, d=128, seed=1)
    q, k, v = (x[n].cuda() for n in "qkv")
    with pytest.raises(cuda_lib.AttnError) as e:
        cuda_lib.attn_fwd_fp8(q, k, v, 0.0, 1.0, 1.0)
    assert e.value.status == cuda_lib.ATTN_ERR_INVALID_ARG
    q64 = torch.zeros(1, 1, 128, 64, dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(cuda_lib.AttnError) as e:
        cuda_lib.attn_fwd_fp8(q64, q64, q64, 1.0, 1.0, 1.0)
    assert e.value.status == cuda_lib.ATTN_ERR_UNSUPPORTED
    with pytest.raises(TypeError):
        cuda_lib.attn_fwd_fp8(q.to(torch.bfloat16), k, v, 1.0, 1.0, 1.0)
