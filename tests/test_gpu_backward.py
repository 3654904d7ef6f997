"""attn_bwd (GPU) against the FP64 backward oracle, through the C interface.

The backward consumes the forward's own BF16 O and FP32 LSE, as a caller
would. Tolerance, from the arithmetic: P and dS are rounded to BF16 (relative
2^-9) for the tensor-core products, O enters D = <dO, O> in BF16, and the
results are stored in BF16 (relative 2^-9 of the largest entry); the
accumulation is FP32. Normwise: max|g - g_ref| <= 2e-2 * max|g_ref| for each
of dQ, dK, dV; no NaN; exact zeros for queries that see no key and for keys
that no query sees (measured normwise errors are 3e-3 to 7e-3).
"""
import math

import numpy as np
import pytest
import torch

import oracle.backward as OB
from online_softmax_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _run(attn, x, mk, win, seed):
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    sl = x["seqlens_k"].to(dev) if x.get("seqlens_k") is not None else None
    g = torch.Generator("cpu").manual_seed(seed)
    do = torch.randn(q.shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    o, lse = attn.attn_fwd(q, k, v, mask_kind=mk, window=win, seqlens_k=sl)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, do.to(dev), lse, mask_kind=mk, window=win,
                               seqlens_k=sl)
    attn.attn_check_device_error()
    return do, dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy()


def _check(name, got, ref):
    assert not np.isnan(got).any(), name
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    assert err <= TOL * max(scale, 1e-6), (name, err, scale)
    return err / max(scale, 1e-30)


BWD_SHAPES = [
    # B, H, Nq, Nk, d, mask, window, seqlen_range
    (1, 2, 256, 256, 128, 0, 0, None),
    (2, 2, 300, 300, 128, W.MASK_CAUSAL, 0, None),
    (1, 2, 513, 700, 64, 0, 0, None),
    (1, 2, 700, 513, 128, W.MASK_CAUSAL, 0, None),
    (2, 3, 400, 400, 128, W.MASK_WINDOW | W.MASK_PADDING, 100, (0, 400)),
    (2, 2, 333, 333, 64, W.MASK_PADDING, 0, (1, 333)),
    (1, 1, 5, 3, 128, 0, 0, None),
    (1, 2, 1024, 1024, 128, W.MASK_CAUSAL, 0, None),
]


@pytest.mark.parametrize("shape", BWD_SHAPES, ids=[str(s) for s in BWD_SHAPES])
def test_bwd_matches_oracle(cuda_lib, shape):
    B, H, Nq, Nk, d, mk, win, sr = shape
    x = W.random_inputs(B, H, Nq, Nk, d, seed=sum(shape[:5]), seqlen_range=sr)
    do, dq, dk, dv = _run(cuda_lib, x, mk, win, seed=3)
    sl = None if x["seqlens_k"] is None else x["seqlens_k"].numpy()
    rq, rk, rv = OB.attention_backward(x["q"].float().numpy(), x["k"].float().numpy(),
                                       x["v"].float().numpy(), do.float().numpy(),
                                       1 / math.sqrt(d), mk, win, sl)
    errs = [_check(n, g, r) for n, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv))]
    # queries that see no key, and keys no query sees, get exactly zero
    for b in range(B):
        Lk = Nk if sl is None else int(sl[b])
        vis = OB.visible_mask(Nq, Nk, mk, win, Lk)
        assert np.all(dq[b][:, ~vis.any(axis=1)] == 0)
        assert np.all(dk[b][:, ~vis.any(axis=0)] == 0)
        assert np.all(dv[b][:, ~vis.any(axis=0)] == 0)
    print("normwise errors dq %.2e dk %.2e dv %.2e" % tuple(errs))


def test_bwd_short_workspace_raises(cuda_lib):
    dev = torch.device("cuda:0")
    q = torch.zeros(1, 1, 130, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(1, 1, 130, dtype=torch.float32, device=dev)
    ws = torch.empty(16, dtype=torch.uint8, device=dev)
    with pytest.raises(cuda_lib.AttnError) as ei:
        cuda_lib.attn_bwd(q, q, q, q, q, lse, workspace=ws)
    assert ei.value.status == cuda_lib.ATTN_ERR_INVALID_ARG


def test_bwd_full_size_sampled_heads(cuda_lib):
    """The benchmarked backward shape (B1 H64 8192^2 d128), in the bench's
    launch configuration: every head computed on the GPU, heads 0 and 63
    compared with the FP64 oracle (about 90 GFLOP of FP64 each)."""
    w = W.PREFILL
    x = W.generate(w)
    do, dq, dk, dv = _run(cuda_lib, x, w.mask_kind, w.window, seed=w.seed + 1)
    assert not (np.isnan(dq).any() or np.isnan(dk).any() or np.isnan(dv).any())
    for h in (0, w.H - 1):
        sl = slice(h, h + 1)
        rq, rk, rv = OB.attention_backward(
            x["q"][:, sl].float().numpy(), x["k"][:, sl].float().numpy(),
            x["v"][:, sl].float().numpy(), do[:, sl].float().numpy(), w.scale)
        for n, g, r in (("dq", dq[:, sl], rq), ("dk", dk[:, sl], rk), ("dv", dv[:, sl], rv)):
            _check(n, g, r)


def test_bwd_three_kernel_build_d128(cuda_lib):
    """The backward built with dQ in its own queries-outer kernel (S and dP
    recomputed there, ATTN_BWD_FUSED_DQ=0; the form d = 64 always uses)
    against the oracle at d = 128."""
    import os
    from online_softmax_02_gb300 import build as B
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    bdir = os.path.join(root, "_build", "attn_bwd3")
    lib = cuda_lib.open_build(B.build(extra_flags=("-DATTN_BWD_FUSED_DQ=0",),
                                      out=os.path.join(bdir, "libattn_bwd3.so"),
                                      build_dir=os.path.join(bdir, "_objs")))
    for (Bn, H, Nq, Nk, d, mk, win, sr) in [(2, 2, 300, 300, 128, W.MASK_CAUSAL, 0, None),
                                            (2, 3, 400, 400, 128, W.MASK_WINDOW | W.MASK_PADDING,
                                             100, (0, 400))]:
        x = W.random_inputs(Bn, H, Nq, Nk, d, seed=Nq + Nk, seqlen_range=sr)
        dev = torch.device("cuda:0")
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
        sl = x["seqlens_k"].to(dev) if x.get("seqlens_k") is not None else None
        g = torch.Generator("cpu").manual_seed(7)
        do = torch.randn(q.shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
        o, lse = cuda_lib.attn_fwd(q, k, v, mask_kind=mk, window=win, seqlens_k=sl)
        dq, dk, dv = cuda_lib.attn_bwd(q, k, v, o, do.to(dev), lse, mask_kind=mk, window=win,
                                       seqlens_k=sl, lib=lib)
        cuda_lib.attn_check_device_error(lib=lib)
        refs = OB.attention_backward(x["q"].float().numpy(), x["k"].float().numpy(),
                                     x["v"].float().numpy(), do.float().numpy(),
                                     1.0 / math.sqrt(d), mk, win,
                                     None if sl is None else x["seqlens_k"].numpy())
        for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
            _check(name, got.float().cpu().numpy(), ref)
