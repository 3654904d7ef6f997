"""The software exponential of the forward kernels (attn_exp2_soft) against
float64 2^x and against CUDA's exp2f (torch.exp2), GPU only.

Bound: the degree-3 polynomial's relative error 1.013e-4 on [-1/2, 1/2]
(pinned on the CPU in test_exp2_poly.py) plus FP32 evaluation (a few ulps):
|y / 2^x - 1| <= 1.05e-4 for -126 <= x <= 127; exact powers of two at
integers (p(0) = 1); +0 for x <= -127 and x = -inf; between -127 and -126 a
denormal below 2^-126.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

REL = 1.05e-4


def _soft(attn, x):
    y = attn.attn_exp2_soft(torch.as_tensor(x, dtype=torch.float32).cuda())
    attn.attn_check_device_error()
    return y.cpu().numpy().astype(np.float64)


def test_exp2_soft_relative_error(cuda_lib):
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-126.0, 127.0, 1_000_001),
                        rng.uniform(-30, 9, 1_000_000)]).astype(np.float32)
    y = _soft(cuda_lib, x)
    ref = np.exp2(x.astype(np.float64))
    assert np.abs(y / ref - 1).max() <= REL
    yf = torch.exp2(torch.from_numpy(x).cuda()).cpu().numpy().astype(np.float64)   # exp2f
    assert np.abs(y / yf - 1).max() <= REL + 2e-7


def test_exp2_soft_special_values(cuda_lib):
    k = np.arange(-126, 128, dtype=np.float32)
    assert np.array_equal(_soft(cuda_lib, k), np.exp2(k.astype(np.float64)))
    lo = np.array([-np.inf, -1e30, -200.0, -127.5, -127.0], np.float32)
    assert np.all(_soft(cuda_lib, lo) == 0.0)
    edge = np.array([-126.99, -126.75, -126.51, -126.49, -126.3, -126.01], np.float32)
    y = _soft(cuda_lib, edge)
    assert np.all(y >= 0) and np.all(y < 2.0 ** -126)
    # odd length: the last element of the final pair
    x = np.linspace(-5, 5, 7).astype(np.float32)
    assert np.abs(_soft(cuda_lib, x) / np.exp2(x.astype(np.float64)) - 1).max() <= REL
