"""attn_decode_splitkv_noalloc: split-KV decode for callers that cannot
allocate device memory on their call path (a serving process whose device
memory is all reserved for its own pool, or one that must not call
cudaMalloc/cudaFree there because those calls can synchronise the device).

Its partials live in a fixed 4 MiB array inside libattn.so instead of a
caller workspace. This file is named so that pytest collects it last.
"""
import pytest
import torch

from online_softmax_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 2e-2, 1e-3   # the tolerances the other decode tests use


def _decode_both(attn, x, num_splits):
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    sl = x["seqlens_k"].to(dev) if x.get("seqlens_k") is not None else None
    B, H, _, d = q.shape
    o_ref, lse_ref = attn.attn_decode_splitkv(q, k, v, seqlens_k=sl, num_splits=num_splits)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, 1), float("nan"), dtype=torch.float32, device=dev)
    attn.attn_decode_splitkv_noalloc(q, k, v, o, lse, seqlens_k=sl, num_splits=num_splits)
    attn.attn_check_device_error()
    return o, lse, o_ref, lse_ref


def _assert_same(o, lse, o_ref, lse_ref):
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O
    fin = torch.isfinite(lse_ref)
    assert torch.equal(torch.isfinite(lse), fin)
    if fin.any():
        assert (lse[fin] - lse_ref[fin]).abs().max().item() <= TOL_LSE


def test_noalloc_matches_workspace_entry_point_twice(cuda_lib):
    # first call: a large problem (fills much of the fixed array)
    x1 = W.random_inputs(1, 32, 1, 20000, 128, seed=31)
    _assert_same(*_decode_both(cuda_lib, x1, 64))
    # second call in a row: smaller, padded, with empty sequences -- the
    # array still holds the first call's partials
    x2 = W.random_inputs(3, 4, 1, 3000, 64, seed=32, seqlen_range=(0, 3000))
    x2["seqlens_k"][0] = 0
    _assert_same(*_decode_both(cuda_lib, x2, 16))


def test_noalloc_rejects_problems_beyond_the_fixed_scratch(cuda_lib):
    dev = torch.device("cuda:0")
    B, H, d, S = 2, 64, 128, 128     # 16384 slots * 129 floats > 4 MiB
    assert cuda_lib.attn_decode_workspace_bytes(B, H, d, S) > 4 * 1024 * 1024
    q = torch.zeros(B, H, 1, d, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(B, H, 256, d, dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    with pytest.raises(cuda_lib.AttnError) as ei:
        cuda_lib.attn_decode_splitkv_noalloc(q, k, k, o, num_splits=S)
    assert ei.value.status == cuda_lib.ATTN_ERR_INVALID_ARG
