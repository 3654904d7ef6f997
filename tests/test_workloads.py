"""Host-side checks of the seeded input generators (no attention arithmetic
lives there): the E4M3 storage of a workload and the row-softmax inputs."""
import math

import numpy as np
import pytest
import torch

from online_softmax_02_gb300 import workloads as W


def test_quantize_e4m3_power_of_two_scale_and_range():
    g = torch.Generator("cpu").manual_seed(0)
    for scale in (1e-3, 0.7, 3.0, 250.0):
        t = torch.randn(64, 128, generator=g) * scale
        t8, d = W.quantize_e4m3(t)
        assert t8.dtype == torch.float8_e4m3fn and t8.shape == t.shape
        assert d > 0 and math.log2(d) == round(math.log2(d))
        assert float(t8.float().abs().max()) <= W.E4M3_MAX
        assert float(t.abs().max()) / d > W.E4M3_MAX / 2      # the smallest such power of two
        # dequantised values are exact in FP32 and within E4M3 rounding of t
        real = t8.float() * d
        assert torch.equal(real, (t8.float().double() * d).float())
        big = t.abs() / d >= 2.0 ** -6                        # normal range of E4M3
        rel = ((real - t).abs() / t.abs())[big]
        assert float(rel.max()) <= 2.0 ** -4 + 1e-7


def test_quantize_e4m3_zero_tensor():
    t8, d = W.quantize_e4m3(torch.zeros(4, 8))
    assert d == 1.0 and float(t8.float().abs().max()) == 0.0


def test_generate_fp8_uses_the_same_draws():
    w = W.Workload("t", 1, 2, 40, 50, 128, torch.bfloat16, seed=9)
    x32 = W.generate(W.Workload("t", 1, 2, 40, 50, 128, torch.float32, seed=9))
    x8 = W.generate_fp8(w)
    for n in "qkv":
        real = x8[n].float() * x8["descale_" + n]
        assert real.shape == x32[n].shape
        assert float((real - x32[n]).abs().max()) <= 2.0 ** -4 * float(x32[n].abs().max())


def test_softmax_inputs_seeded_and_typed():
    a = W.softmax_inputs(3, 100, seed=4)
    b = W.softmax_inputs(3, 100, seed=4)
    assert torch.equal(a, b) and a.dtype == torch.float32 and a.is_contiguous()
    c = W.softmax_inputs(3, 100, dtype=torch.bfloat16, seed=4, scale=2.0)
    assert c.dtype == torch.bfloat16
    assert torch.equal(c, (a * 2.0).to(torch.bfloat16))
