"""attn_softmax_rows (GPU) against the FP64 row-softmax oracle.

Tolerances from the arithmetic: FP32 path (ex2.approx, FP32 sums):
max|y - y_ref| <= 4e-6 * max|y_ref| per row block and |lse - lse_ref| <= 2e-5;
BF16 outputs are rounded once: |y - y_ref| <= 2^-8 |y_ref| + 1e-7 per entry.
"""
import numpy as np
import pytest
import torch

from online_softmax_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(attn, x):
    y, lse = attn.attn_softmax_rows(x.cuda())
    attn.attn_check_device_error()
    return y.float().cpu().numpy(), lse.cpu().numpy()


def _check(y, lse, ry, rl, bf16):
    assert not np.isnan(y).any() and not np.isnan(lse).any()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(lse[~fin] == -np.inf) and np.all(y[~fin] == 0)
    if bf16:
        assert np.all(np.abs(y - ry) <= 2.0 ** -8 * np.abs(ry) + 1e-7)
    else:
        assert np.abs(y - ry).max() <= 4e-6 * max(np.abs(ry).max(), 1e-30)
    if fin.any():
        assert np.abs(lse[fin] - rl[fin]).max() <= 2e-5 * max(1.0, np.abs(rl[fin]).max())


# Row lengths chosen to reach every launch shape (16-byte vectors: 4 FP32 or
# 8 BF16 values): warp mode with 1, 2, 4, 8 and 16 vectors per lane and a
# partial CTA of rows; CTA mode with 4 and 8 vectors per thread; one streamed
# CTA per row; clusters of 2, 4, 5, 7 and 8 streamed CTAs (ragged last slices,
# slices longer than the split size at 8); the scalar kernel for lengths that
# are not a vector multiple.
SHAPES = [(1, 4), (37, 200), (9, 480), (64, 1024), (6, 2048), (8, 4096), (5, 6144), (5, 12288),
          (16, 32768),
          (3, 32776), (4, 100000), (2, 200000), (2, 300000), (37, 513), (3, 7)]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_softmax_rows_shapes(cuda_lib, orc, shape, dtype):
    rows, n = shape
    x = W.softmax_inputs(rows, n, dtype=dtype, seed=rows + n, scale=3.0)
    y, lse = _run(cuda_lib, x)
    ry, rl = orc.softmax_rows(x.float().numpy())
    _check(y, lse, ry, rl, dtype == torch.bfloat16)


def test_softmax_rows_masked_and_large(cuda_lib, orc):
    x = W.softmax_inputs(6, 2048, seed=5, scale=2.0)
    x[0, ::5] = float("-inf")        # masked entries
    x[1, :] = float("-inf")          # fully masked row
    x[2] += 1e4                      # large scores
    x[3] -= 1e4
    x[4, -1] = 60.0                  # late maximum
    y, lse = _run(cuda_lib, x)
    ry, rl = orc.softmax_rows(x.numpy())
    _check(y, lse, ry, rl, False)


def test_softmax_rows_workload_sampled(cuda_lib, orc):
    """The benchmarked shape ([4096, 32768] FP32): 64 sampled rows against the
    oracle, every row sums to one."""
    x = W.softmax_inputs()
    y, lse = _run(cuda_lib, x)
    assert np.abs(y.sum(axis=1, dtype=np.float64) - 1.0).max() <= 1e-4
    idx = np.random.default_rng(0).choice(x.shape[0], 64, replace=False)
    ry, rl = orc.softmax_rows(x[idx].numpy())
    _check(y[idx], lse[idx], ry, rl, False)


def test_softmax_rows_misaligned_base(cuda_lib, orc):
    """A base address 4 bytes past a 16-byte boundary takes the scalar kernel."""
    flat = W.softmax_inputs(1, 17 * 1024 + 1, seed=9).reshape(-1)
    x = flat[1:].reshape(17, 1024)
    xd = torch.empty(17 * 1024 + 1, dtype=torch.float32, device="cuda")[1:].view(17, 1024)
    xd.copy_(x)
    yd = torch.empty(17 * 1024 + 1, dtype=torch.float32, device="cuda")[1:].view(17, 1024)
    y, lse = cuda_lib.attn_softmax_rows(xd, y=yd)
    cuda_lib.attn_check_device_error()
    ry, rl = orc.softmax_rows(x.numpy())
    _check(y.cpu().numpy(), lse.cpu().numpy(), ry, rl, False)


@pytest.mark.parametrize("n", [200, 4096, 6144, 32768, 100000, 513])
def test_softmax_rows_in_place(cuda_lib, orc, n):
    """y == x: warp, CTA, streamed, cluster and scalar shapes."""
    x = W.softmax_inputs(5, n, seed=n, scale=2.0)
    xd = x.cuda()
    y, lse = cuda_lib.attn_softmax_rows(xd, y=xd)
    cuda_lib.attn_check_device_error()
    assert y.data_ptr() == xd.data_ptr()
    ry, rl = orc.softmax_rows(x.numpy())
    _check(y.cpu().numpy(), lse.cpu().numpy(), ry, rl, False)
