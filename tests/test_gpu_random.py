"""Seeded random cases through every entry point, each against the FP64
oracle element by element (GPU only).

Shapes, head dims, masks, window lengths, key lengths and scales are drawn
from a fixed seed per case, so a failure names a reproducible case. The
tolerances are the ones the dedicated parity tests derive (BF16 outputs
2e-2 max-abs, LSE 1e-3; backward 2e-2 normwise; row softmax 4e-6 of the
largest output; E4M3 the rounding bound of test_gpu_fp8.py).
"""
import math

import numpy as np
import pytest
import torch

from oracle import backward as OB
from online_softmax_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MASKS = [W.MASK_NONE, W.MASK_CAUSAL, W.MASK_WINDOW, W.MASK_PADDING,
         W.MASK_CAUSAL | W.MASK_PADDING, W.MASK_WINDOW | W.MASK_PADDING]


def _case(seed, max_nq=700, max_nk=1500, d_choices=(64, 128), b_max=3, h_max=4):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, b_max + 1))
    H = int(rng.integers(1, h_max + 1))
    Nq = int(rng.integers(1, max_nq + 1))
    Nk = int(rng.integers(1, max_nk + 1))
    d = int(rng.choice(d_choices))
    mask = int(MASKS[rng.integers(0, len(MASKS))])
    window = int(rng.integers(1, max(2, Nk + 1))) if mask & W.MASK_WINDOW else 0
    scale = float(rng.uniform(0.3, 2.0)) / math.sqrt(d)
    sr = (0, Nk) if mask & W.MASK_PADDING else None
    return dict(B=B, H=H, Nq=Nq, Nk=Nk, d=d, mask=mask, window=window, scale=scale, sr=sr,
                seed=seed)


def _close(o, lse, ro, rl, tol_o=2e-2, tol_l=1e-3, what=""):
    o = np.asarray(o, np.float64)
    lse = np.asarray(lse, np.float64)
    assert not np.isnan(o).any() and not np.isnan(lse).any(), what
    empty = np.isneginf(rl)
    assert np.array_equal(np.isneginf(lse), empty), (what, "empty-row pattern")
    assert np.all(o[empty] == 0), what
    assert np.abs(o - ro).max() <= tol_o, (what, float(np.abs(o - ro).max()))
    if (~empty).any():
        assert np.abs(lse[~empty] - rl[~empty]).max() <= tol_l, what


@pytest.mark.parametrize("seed", range(24))
def test_random_forward_bf16(cuda_lib, orc, seed):
    c = _case(seed)
    x = W.random_inputs(c["B"], c["H"], c["Nq"], c["Nk"], c["d"], seed=seed,
                        seqlen_range=c["sr"])
    dev = torch.device("cuda:0")
    sl = x["seqlens_k"]
    o, lse = cuda_lib.attn_fwd(*(x[n].to(dev) for n in "qkv"), scale=c["scale"],
                               mask_kind=c["mask"], window=c["window"],
                               seqlens_k=None if sl is None else sl.to(dev))
    cuda_lib.attn_check_device_error()
    ro, rl = orc.attention(x["q"].float().numpy(), x["k"].float().numpy(), x["v"].float().numpy(),
                           c["scale"], c["mask"], c["window"], None if sl is None else sl.numpy())
    _close(o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, what=str(c))


@pytest.mark.parametrize("seed", range(12))
def test_random_decode(cuda_lib, orc, seed):
    c = _case(100 + seed, max_nq=1, max_nk=20000)
    c["Nq"] = 1
    rng = np.random.default_rng(seed)
    splits = int(rng.integers(1, 129))
    x = W.random_inputs(c["B"], c["H"], 1, c["Nk"], c["d"], seed=seed,
                        seqlen_range=(0, c["Nk"]) if seed % 3 == 0 else None)
    dev = torch.device("cuda:0")
    sl = x["seqlens_k"]
    B, H, _, d = x["q"].shape
    ws = torch.empty(cuda_lib.attn_decode_workspace_bytes(B, H, d, splits), dtype=torch.uint8,
                     device=dev)
    o, lse = cuda_lib.attn_decode_splitkv(*(x[n].to(dev) for n in "qkv"), scale=c["scale"],
                                          seqlens_k=None if sl is None else sl.to(dev),
                                          num_splits=splits, workspace=ws)
    cuda_lib.attn_check_device_error()
    ro, rl = orc.attention(x["q"].float().numpy(), x["k"].float().numpy(), x["v"].float().numpy(),
                           c["scale"], W.MASK_PADDING if sl is not None else 0, 0,
                           None if sl is None else sl.numpy())
    _close(o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, what=str((c, splits)))


@pytest.mark.parametrize("seed", range(6))
def test_random_backward(cuda_lib, seed):
    c = _case(200 + seed, max_nq=400, max_nk=400, b_max=2, h_max=2)
    x = W.random_inputs(c["B"], c["H"], c["Nq"], c["Nk"], c["d"], seed=seed,
                        seqlen_range=c["sr"])
    g = torch.Generator("cpu").manual_seed(seed)
    do = torch.randn(x["q"].shape, generator=g).to(torch.bfloat16)
    dev = torch.device("cuda:0")
    sl = x["seqlens_k"]
    sld = None if sl is None else sl.to(dev)
    q, k, v, dod = (t.to(dev) for t in (x["q"], x["k"], x["v"], do))
    o, lse = cuda_lib.attn_fwd(q, k, v, scale=c["scale"], mask_kind=c["mask"], window=c["window"],
                               seqlens_k=sld)
    grads = cuda_lib.attn_bwd(q, k, v, o, dod, lse, scale=c["scale"], mask_kind=c["mask"],
                              window=c["window"], seqlens_k=sld)
    cuda_lib.attn_check_device_error()
    refs = OB.attention_backward(x["q"].float().numpy(), x["k"].float().numpy(),
                                 x["v"].float().numpy(), do.float().numpy(), c["scale"], c["mask"],
                                 c["window"], None if sl is None else sl.numpy())
    for got, ref, name in zip(grads, refs, ("dq", "dk", "dv")):
        got = got.float().cpu().numpy()
        assert not np.isnan(got).any(), (c, name)
        scale_ref = max(np.abs(ref).max(), 1e-6)
        assert np.abs(got - ref).max() <= 2e-2 * scale_ref, (c, name)


@pytest.mark.parametrize("seed", range(10))
def test_random_softmax_rows(cuda_lib, orc, seed):
    rng = np.random.default_rng(300 + seed)
    rows = int(rng.integers(1, 300))
    n = int(rng.integers(1, 70000)) if seed % 2 else int(rng.integers(1, 3000))
    bf16 = bool(seed % 3 == 0)
    x = W.softmax_inputs(rows, n, dtype=torch.bfloat16 if bf16 else torch.float32, seed=seed,
                         scale=float(rng.uniform(0.5, 8)))
    if seed % 4 == 1:
        x[:, rng.integers(0, n, size=max(1, n // 7))] = float("-inf")
    y, lse = cuda_lib.attn_softmax_rows(x.cuda())
    cuda_lib.attn_check_device_error()
    ry, rl = orc.softmax_rows(x.float().numpy())
    y = y.float().cpu().numpy()
    lse = lse.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lse), fin)
    if bf16:
        assert np.all(np.abs(y - ry) <= 2.0 ** -8 * np.abs(ry) + 1e-7), (rows, n)
    else:
        assert np.abs(y - ry).max() <= 4e-6 * max(np.abs(ry).max(), 1e-30), (rows, n)
    if fin.any():
        assert np.abs(lse[fin] - rl[fin]).max() <= 2e-5 * max(1.0, np.abs(rl[fin]).max())


@pytest.mark.parametrize("seed", range(6))
def test_random_forward_fp8(cuda_lib, orc, seed):
    import test_gpu_fp8 as F8
    c = _case(400 + seed, max_nq=600, max_nk=1200, d_choices=(128,), b_max=2, h_max=3)
    x = F8._fp8_inputs(c["B"], c["H"], c["Nq"], c["Nk"], seed=seed, seqlen_range=c["sr"])
    F8._compare(cuda_lib, orc, x, c["mask"], c["window"], what=str(c))
