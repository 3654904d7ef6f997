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
    # The same two kernels run on the same inputs; only where the partials
    # are kept differs, so the results agree bit for bit.
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)


def test_noalloc_matches_workspace_entry_point_twice(cuda_lib):
    # First call: the partials fill the fixed array to within 256 bytes of
    # its end (64 heads x 127 splits x 129 FP32 values, 4194048 of 4194304
    # bytes), so the log-sum-exp region at the top of the array is used.
    assert cuda_lib.attn_decode_workspace_bytes(1, 64, 128, 127) == 4194048
    x1 = W.random_inputs(1, 64, 1, 20000, 128, seed=31)
    _assert_same(*_decode_both(cuda_lib, x1, 127))
    # Second call in a row: smaller, padded, with an empty sequence -- the
    # array still holds the first call's partials.
    x2 = W.random_inputs(3, 4, 1, 3000, 64, seed=32, seqlen_range=(0, 3000))
    x2["seqlens_k"][0] = 0
    _assert_same(*_decode_both(cuda_lib, x2, 16))


def test_noalloc_rejects_problems_beyond_the_fixed_scratch(cuda_lib):
    dev = torch.device("cuda:0")
    # one split more than the largest accepted problem above
    assert cuda_lib.attn_decode_workspace_bytes(1, 64, 128, 128) > 4 * 1024 * 1024
    B, H, d, S = 1, 64, 128, 128
    q = torch.zeros(B, H, 1, d, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(B, H, 256, d, dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    with pytest.raises(cuda_lib.AttnError) as ei:
        cuda_lib.attn_decode_splitkv_noalloc(q, k, k, o, num_splits=S)
    assert ei.value.status == cuda_lib.ATTN_ERR_INVALID_ARG
