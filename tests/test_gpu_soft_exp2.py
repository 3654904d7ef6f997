"""The fused forward with part of P's exponentials on the FMA pipe.

P1 ("What did FlashAttention-2 and -3 change?") credits FlashAttention-4 with
computing some of the softmax exponentials in software on the FMA units
instead of the special-function unit. The forward kernel can do this for a
compile-time number of every 16 exponential pairs (ATTN_SOFT_EXP2_PAIRS_BF16,
ATTN_SOFT_EXP2_PAIRS_E4M3; the default build, by measurement, keeps every
BF16 exponential on the special-function unit and computes 1 of every 16
E4M3 pairs in software, so test_gpu_fp8.py covers that split). This file builds
the library a second time with two of every 16 pairs in software for both
input types, and checks that build's forward against the FP64 oracle at the
same tolerances as the default build, through the same C interface.

The software exponential has relative error 1.02e-4 (pinned on the CPU in
test_exp2_poly.py), below the BF16 rounding of P (2^-9) and far below the
E4M3 rounding (2^-4), so the default tolerances apply unchanged; l gains at
most 1e-4 relative error, i.e. 1e-4 in the log-sum-exp.
"""
import math
import os

import numpy as np
import pytest
import torch

import test_gpu_fp8 as F8
from test_gpu_parity import TOL_LSE, TOL_O_BF16, assert_close, oracle_fwd
from online_softmax_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu

FLAGS = ("-DATTN_SOFT_EXP2_PAIRS_BF16=2", "-DATTN_SOFT_EXP2_PAIRS_E4M3=2")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def soft_lib(cuda_lib):
    from online_softmax_02_gb300 import build as B
    bdir = os.path.join(ROOT, "_build", "attn_soft_exp2")
    path = B.build(extra_flags=FLAGS, out=os.path.join(bdir, "libattn_soft_exp2.so"),
                   build_dir=bdir)
    return cuda_lib.open_build(path)


def _fwd(attn, lib, x, mask_kind=0, window=0):
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    sl = x.get("seqlens_k")
    o, lse = attn.attn_fwd(q, k, v, mask_kind=mask_kind, window=window,
                           seqlens_k=None if sl is None else sl.to(dev), lib=lib)
    attn.attn_check_device_error(lib=lib)
    return o.float().cpu().numpy(), lse.cpu().numpy()


SHAPES = [
    # B, H, Nq, Nk, d, mask, window, seqlen_range
    (1, 2, 300, 300, 128, 0, 0, None),
    (2, 3, 513, 700, 128, W.MASK_CAUSAL, 0, None),
    (1, 2, 1000, 1000, 64, W.MASK_CAUSAL, 0, None),
    (3, 2, 600, 600, 128, W.MASK_WINDOW | W.MASK_PADDING, 64, (0, 600)),
    (2, 2, 640, 640, 128, W.MASK_CAUSAL | W.MASK_PADDING, 0, (50, 640)),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_soft_exp2_bf16_against_oracle(cuda_lib, soft_lib, orc, shape):
    B, H, Nq, Nk, d, mk, win, sr = shape
    x = W.random_inputs(B, H, Nq, Nk, d, seed=hash(shape) % 1000, seqlen_range=sr)
    o, lse = _fwd(cuda_lib, soft_lib, x, mk, win)
    ro, rl = oracle_fwd(orc, x, mk, win)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what=str(shape))


def test_soft_exp2_bf16_late_max_and_large_scores(cuda_lib, soft_lib, orc):
    x = W.random_inputs(1, 2, 256, 1000, 128, seed=6)
    x["q"][..., -1] = 1.0
    x["k"][:, :, -5:, -1] += 10.0 * math.sqrt(128)
    o, lse = _fwd(cuda_lib, soft_lib, x)
    ro, rl = oracle_fwd(orc, x)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what="late max")
    x = W.random_inputs(1, 2, 400, 700, 128, seed=5, scale_q=30.0)
    o, lse = _fwd(cuda_lib, soft_lib, x, W.MASK_CAUSAL)
    ro, rl = oracle_fwd(orc, x, W.MASK_CAUSAL)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what="large scores")


def test_soft_exp2_build_differs_from_default(cuda_lib, soft_lib):
    """The second build really computes some weights another way: its output
    differs from the default build's in some elements (by about the BF16
    rounding of P), while the log-sum-exp agrees to the polynomial's error."""
    x = W.random_inputs(1, 4, 512, 2048, 128, seed=12)
    o1, l1 = _fwd(cuda_lib, soft_lib, x)
    o0, l0 = _fwd(cuda_lib, None, x)
    diff = np.abs(o1 - o0)
    assert diff.max() > 0
    assert diff.max() <= 2e-2
    assert np.abs(l1 - l0).max() <= 2e-4


@pytest.mark.parametrize("shape", F8.SHAPES[:4], ids=[str(s) for s in F8.SHAPES[:4]])
def test_soft_exp2_e4m3_against_oracle(cuda_lib, soft_lib, orc, shape):
    B, H, Nq, Nk, mk, win, sr = shape
    x = F8._fp8_inputs(B, H, Nq, Nk, seed=B * 1000 + Nq, seqlen_range=sr)
    qr, kr, vr = F8._real(x, "q"), F8._real(x, "k"), F8._real(x, "v")
    sl = x["seqlens_k"]
    dev = torch.device("cuda:0")
    o, lse = cuda_lib.attn_fwd_fp8(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev),
                                   x["descale_q"], x["descale_k"], x["descale_v"],
                                   mask_kind=mk, window=win,
                                   seqlens_k=None if sl is None else sl.to(dev), lib=soft_lib)
    cuda_lib.attn_check_device_error(lib=soft_lib)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    rows = np.arange(B * H * Nq)
    ro, rl = orc.attention(qr, kr, vr, 1.0 / math.sqrt(128), mk, win,
                           None if sl is None else sl.numpy(), rows=rows)
    bound = F8._bound(qr, kr, vr, 1.0 / math.sqrt(128), mk, win,
                      None if sl is None else sl.numpy(), rows)
    F8._check(o.reshape(-1, 128), lse.reshape(-1), ro, rl, bound, str(shape))
