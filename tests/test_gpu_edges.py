"""Long, large and degenerate cases against the FP64 oracle (GPU only):
131072 keys through the forward kernel, a 32K-token causal head on sampled
rows, many small heads, decode with one key per split and the split limit,
one-element softmax rows, one-key / one-query E4M3 problems, and query
tiles that see no key beside tiles that do."""
import math

import numpy as np
import pytest
import torch

from online_softmax_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 2e-2, 1e-3


def _check(o, lse, ro, rl, tol_o=TOL_O):
    o = np.asarray(o, np.float64)
    lse = np.asarray(lse, np.float64)
    assert not np.isnan(o).any() and not np.isnan(lse).any()
    empty = np.isneginf(rl)
    assert np.array_equal(np.isneginf(lse), empty)
    assert np.abs(o - ro).max() <= tol_o
    if (~empty).any():
        assert np.abs(lse[~empty] - rl[~empty]).max() <= TOL_LSE


def _fwd(attn, x, mask=0, window=0):
    dev = torch.device("cuda:0")
    o, lse = attn.attn_fwd(*(x[n].to(dev) for n in "qkv"), mask_kind=mask, window=window)
    attn.attn_check_device_error()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def test_forward_131072_keys(cuda_lib, orc):
    x = W.random_inputs(1, 1, 200, 131072, 128, seed=31)
    o, lse = _fwd(cuda_lib, x)
    ro, rl = orc.attention(*(x[n].float().numpy() for n in "qkv"), 1 / math.sqrt(128))
    _check(o, lse, ro, rl)


def test_forward_causal_32k_sampled_rows(cuda_lib, orc):
    x = W.random_inputs(1, 1, 32768, 32768, 128, seed=32)
    o, lse = _fwd(cuda_lib, x, W.MASK_CAUSAL)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, 16383, 32766, 32767],
                                     np.random.default_rng(3).choice(32768, 40, replace=False)]))
    ro, rl = orc.attention(*(x[n].float().numpy() for n in "qkv"), 1 / math.sqrt(128),
                           W.MASK_CAUSAL, rows=rows)
    _check(o.reshape(-1, 128)[rows], lse.reshape(-1)[rows], ro, rl)


def test_forward_many_small_heads(cuda_lib, orc):
    x = W.random_inputs(64, 64, 3, 70, 64, seed=33)
    o, lse = _fwd(cuda_lib, x, W.MASK_CAUSAL)
    ro, rl = orc.attention(*(x[n].float().numpy() for n in "qkv"), 1 / math.sqrt(64),
                           W.MASK_CAUSAL)
    _check(o, lse, ro, rl)


@pytest.mark.parametrize("nk,splits", [(1000, 1000), (1024, 1024), (5, 64), (1, 1)])
def test_decode_split_extremes(cuda_lib, orc, nk, splits):
    x = W.random_inputs(2, 3, 1, nk, 128, seed=nk)
    dev = torch.device("cuda:0")
    ws = torch.empty(cuda_lib.attn_decode_workspace_bytes(2, 3, 128, splits), dtype=torch.uint8,
                     device=dev)
    o, lse = cuda_lib.attn_decode_splitkv(*(x[n].to(dev) for n in "qkv"), num_splits=splits,
                                          workspace=ws)
    cuda_lib.attn_check_device_error()
    ro, rl = orc.attention(*(x[n].float().numpy() for n in "qkv"), 1 / math.sqrt(128))
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl)


def test_softmax_one_element_rows(cuda_lib):
    x = W.softmax_inputs(1000, 1, seed=34, scale=50.0)
    x[7, 0] = float("-inf")
    y, lse = cuda_lib.attn_softmax_rows(x.cuda())
    cuda_lib.attn_check_device_error()
    y, lse = y.cpu().numpy(), lse.cpu().numpy()
    keep = np.ones(1000, bool)
    keep[7] = False
    assert np.abs(y[keep] - 1.0).max() <= 1e-6
    assert y[7, 0] == 0.0 and lse[7] == -np.inf
    assert np.abs(lse[keep] - x.numpy()[keep, 0]).max() <= 2e-5 * 50 * 5


@pytest.mark.parametrize("nq,nk", [(1, 1), (300, 1), (1, 700)])
def test_fp8_degenerate_shapes(cuda_lib, orc, nq, nk):
    import test_gpu_fp8 as F8
    x = F8._fp8_inputs(1, 2, nq, nk, seed=nq * 1000 + nk)
    F8._compare(cuda_lib, orc, x, what=str((nq, nk)))


@pytest.mark.parametrize("d", [64, 128])
def test_forward_empty_second_tile(cuda_lib, orc, d):
    """A window of one key with short key lengths: in each 256-row pair of
    query tiles the first tile has visible keys and the second has none, so
    the second tile's output buffer is written while the first tile still
    computes. Rows without a key must come out exactly 0 with lse = -inf."""
    x = W.random_inputs(2, 3, 256, 256, d, seed=35 + d)
    x["seqlens_k"] = torch.tensor([100, 60], dtype=torch.int32)
    dev = torch.device("cuda:0")
    o, lse = cuda_lib.attn_fwd(*(x[n].to(dev) for n in "qkv"), mask_kind=W.MASK_WINDOW | W.MASK_PADDING,
                               window=1, seqlens_k=x["seqlens_k"].to(dev))
    cuda_lib.attn_check_device_error()
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    ro, rl = orc.attention(*(x[n].float().numpy() for n in "qkv"), 1 / math.sqrt(d),
                           W.MASK_WINDOW | W.MASK_PADDING, 1, x["seqlens_k"].numpy())
    empty = np.isneginf(rl)
    assert empty[:, :, 128:].all() and (~empty[:, :, :60]).all()
    assert np.all(o[empty] == 0.0)
    _check(o, lse, ro, rl)
