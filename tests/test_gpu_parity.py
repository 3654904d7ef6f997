"""CUDA path against the FP64 oracle, element by element, through the C
interface (GPU only).

Tolerances (from the accuracy targets of this library):
  BF16 forward / decode: max |o - o_ref| <= 2e-2, max |lse - lse_ref| <= 1e-3.
  FP32 forward: max |o - o_ref| / max |o_ref| <= 1e-5 (normwise relative),
                max |lse - lse_ref| <= 1e-5.
  Always: no NaN; lse is -inf exactly where the oracle's is (rows with no
  visible key), and o is exactly 0 there.
"""
import math

import numpy as np
import pytest
import torch

from online_softmax_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_O_BF16, TOL_LSE = 2e-2, 1e-3
TOL_O_F32_REL, TOL_LSE_F32 = 1e-5, 1e-5


def _np(t):
    return t.detach().float().cpu().numpy()


def assert_close(o, lse, ro, rl, tol_o, tol_l, rel=False, what=""):
    o = np.asarray(o, np.float64)
    lse = np.asarray(lse, np.float64)
    assert not np.isnan(o).any(), (what, "NaN in o")
    assert not np.isnan(lse).any(), (what, "NaN in lse")
    empty = np.isneginf(rl)
    assert np.array_equal(np.isneginf(lse), empty), (what, "lse -inf pattern differs")
    assert np.isfinite(lse[~empty]).all(), (what, "inf in lse")
    if empty.any():
        assert np.all(o[empty] == 0.0), (what, "empty rows must be 0")
    err_o = np.abs(o - ro).max() if o.size else 0.0
    if rel:
        err_o = err_o / max(np.abs(ro).max(), 1e-30)
    err_l = np.abs(lse[~empty] - rl[~empty]).max() if (~empty).any() else 0.0
    assert err_o <= tol_o, (what, "o error", err_o)
    assert err_l <= tol_l, (what, "lse error", err_l)
    return err_o, err_l


def run_fwd(attn, x, mask_kind=0, window=0, scale=None, dtype=torch.bfloat16):
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    sl = x.get("seqlens_k")
    sl = sl.to(dev) if sl is not None else None
    fn = attn.attn_fwd if dtype == torch.bfloat16 else attn.attn_fwd_f32
    o, lse = fn(q, k, v, scale=scale, mask_kind=mask_kind, window=window, seqlens_k=sl)
    attn.attn_check_device_error()
    return _np(o), _np(lse)


def oracle_fwd(orc, x, mask_kind=0, window=0, scale=None, rows=None):
    d = x["q"].shape[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    sl = x.get("seqlens_k")
    return orc.attention(_np(x["q"]), _np(x["k"]), _np(x["v"]), scale, mask_kind, window,
                         None if sl is None else sl.numpy(), rows=rows)


# --------------------------------------------------------------- FP32 path
@pytest.mark.parametrize("q0", [0, 300, 872])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("planted", [False, True])
def test_tile_test_fp32(cuda_lib, orc, q0, causal, planted):
    """P2's test: 128 query rows at tile offset q0 over 1,000 keys, d = 64."""
    w = W.tile_test(q0, causal, planted)
    x = W.generate(w)
    o, lse = run_fwd(cuda_lib, x, w.mask_kind, dtype=torch.float32)
    ro, rl = oracle_fwd(orc, x, w.mask_kind)
    assert_close(o, lse, ro, rl, TOL_O_F32_REL, TOL_LSE_F32, rel=True, what=w.name)


@pytest.mark.parametrize("shape", [
    (1, 2, 300, 300, 128, 0, 0), (2, 1, 257, 1000, 64, W.MASK_CAUSAL, 0),
    (1, 3, 100, 100, 128, W.MASK_WINDOW, 7), (2, 2, 65, 129, 64, W.MASK_PADDING, 0),
])
def test_fwd_f32_shapes(cuda_lib, orc, shape):
    B, H, Nq, Nk, d, mk, win = shape
    x = W.random_inputs(B, H, Nq, Nk, d, dtype=torch.float32, seed=11,
                        seqlen_range=(0, Nk) if mk & W.MASK_PADDING else None)
    o, lse = run_fwd(cuda_lib, x, mk, win, dtype=torch.float32)
    ro, rl = oracle_fwd(orc, x, mk, win)
    assert_close(o, lse, ro, rl, TOL_O_F32_REL, TOL_LSE_F32, rel=True, what=str(shape))


# ------------------------------------------------------ BF16 tensor-core path
FWD_SHAPES = [
    # B, H, Nq, Nk, d, mask, window, seqlen_range
    (1, 2, 256, 256, 128, 0, 0, None),            # one CTA, exact tiles
    (1, 2, 300, 300, 128, 0, 0, None),            # ragged query and key tails
    (2, 3, 513, 700, 128, W.MASK_CAUSAL, 0, None),
    (1, 2, 1000, 1000, 64, 0, 0, None),
    (1, 2, 1000, 1000, 64, W.MASK_CAUSAL, 0, None),
    (1, 1, 5, 3, 128, 0, 0, None),                # smaller than a tile
    (1, 1, 1, 1, 128, W.MASK_CAUSAL, 0, None),
    (1, 2, 100, 1000, 128, W.MASK_CAUSAL, 0, None),   # Nq < Nk, top-left causal
    (1, 2, 1000, 100, 128, W.MASK_CAUSAL, 0, None),   # Nq > Nk
    (2, 2, 777, 777, 128, W.MASK_WINDOW, 200, None),
    (3, 2, 600, 600, 128, W.MASK_WINDOW | W.MASK_PADDING, 64, (0, 600)),
    (4, 1, 515, 515, 64, W.MASK_PADDING, 0, (0, 515)),
    (2, 2, 300, 300, 128, W.MASK_WINDOW | W.MASK_PADDING, 1, (1, 300)),
    (2, 2, 640, 640, 128, W.MASK_CAUSAL | W.MASK_PADDING, 0, (50, 640)),
]


@pytest.mark.parametrize("shape", FWD_SHAPES, ids=[str(s) for s in FWD_SHAPES])
def test_fwd_bf16_shapes(cuda_lib, orc, shape):
    B, H, Nq, Nk, d, mk, win, sr = shape
    x = W.random_inputs(B, H, Nq, Nk, d, seed=hash(shape) % 1000, seqlen_range=sr)
    o, lse = run_fwd(cuda_lib, x, mk, win)
    ro, rl = oracle_fwd(orc, x, mk, win)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what=str(shape))


@pytest.mark.parametrize("scale_q", [30.0, 60.0])
def test_fwd_bf16_large_scores(cuda_lib, orc, scale_q):
    """Scores of magnitude 100-300 (|lse| up to about 140 and 290): the
    running max must keep exp in range, and the log-sum-exp holds the same
    1e-3 absolute bound as everywhere else (measured: 3e-5 and 6e-5, the
    size of FP32 rounding of scores that large)."""
    x = W.random_inputs(1, 2, 400, 700, 128, seed=5, scale_q=scale_q)
    o, lse = run_fwd(cuda_lib, x, W.MASK_CAUSAL)
    ro, rl = oracle_fwd(orc, x, W.MASK_CAUSAL)
    assert np.abs(rl[np.isfinite(rl)]).max() > 100
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what="large scores")


def test_fwd_bf16_late_max(cuda_lib, orc):
    """Largest scores planted in the last five keys (the max arrives late)."""
    x = W.random_inputs(1, 2, 256, 1000, 128, seed=6)
    x["q"][..., -1] = 1.0
    x["k"][:, :, -5:, -1] += 10.0 * math.sqrt(128)
    o, lse = run_fwd(cuda_lib, x)
    ro, rl = oracle_fwd(orc, x)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what="late max")


def test_fwd_bf16_no_keys(cuda_lib, orc):
    """Nk = 0 and all-zero seqlens: every row empty."""
    x = W.random_inputs(1, 2, 130, 0, 128, seed=7)
    o, lse = run_fwd(cuda_lib, x)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    x = W.random_inputs(2, 2, 130, 260, 128, seed=8)
    x["seqlens_k"] = torch.zeros(2, dtype=torch.int32)
    o, lse = run_fwd(cuda_lib, x, W.MASK_PADDING)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_fwd_bf16_lse_optional(cuda_lib, orc):
    x = W.random_inputs(1, 1, 200, 200, 128, seed=9)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse = cuda_lib.attn_fwd(q, k, v, want_lse=False)
    assert lse is None
    ro, _ = oracle_fwd(orc, x)
    assert np.abs(_np(o) - ro).max() <= TOL_O_BF16


# ------------------------------------------------------ full-size workloads
def _sample_rows(B, H, Nq, n, seed, diag_heads=()):
    """Random flat rows (b*H+h)*Nq+i, plus fixed rows at tile edges of the
    first and last head, plus -- for the heads in diag_heads -- the rows at
    both edges and the middle of every 128-row tile (the rows whose last
    visible key sits at the start, middle or end of the tile's diagonal
    block under a causal mask)."""
    rng = np.random.default_rng(seed)
    fixed = []
    for bh in (0, B * H - 1):
        for i in (0, 1, 127, 128, 255, 256, Nq // 2, Nq - 129, Nq - 128, Nq - 1):
            if 0 <= i < Nq:
                fixed.append(bh * Nq + i)
    for bh in diag_heads:
        for t0 in range(0, Nq, 128):
            for r in (0, 1, 63, 64, 126, 127):
                if t0 + r < Nq:
                    fixed.append(bh * Nq + t0 + r)
    rand = rng.choice(B * H * Nq, size=n, replace=False)
    return np.unique(np.concatenate([np.array(fixed, np.int64), rand.astype(np.int64)]))


def _run_full_size(cuda_lib, orc, w, rows):
    x = W.generate(w)
    o, lse = run_fwd(cuda_lib, x, w.mask_kind, w.window)
    assert not np.isnan(o).any() and not np.isnan(lse).any()
    if rows is None:
        ro, rl = oracle_fwd(orc, x, w.mask_kind, w.window)
        assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what=w.name)
    else:
        ro, rl = oracle_fwd(orc, x, w.mask_kind, w.window, rows=rows)
        assert_close(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], ro, rl, TOL_O_BF16,
                     TOL_LSE, what=w.name)
    return x, o, lse


def test_full_size_prefill(cuda_lib, orc):
    """The prefill workload (B1 H64 8192^2, no mask) in the benchmark's launch
    configuration: 4096 sampled rows against the oracle one by one (the
    whole tensor is 2.2 TFLOP of FP64 work), no NaN anywhere."""
    w = W.PREFILL
    _run_full_size(cuda_lib, orc, w, _sample_rows(w.B, w.H, w.Nq, 4096, seed=1))


def test_full_size_causal(cuda_lib, orc):
    """The causal workload (B2 H32 8192^2): 16384 random rows plus the edge
    and middle rows of every tile of four heads, against the oracle."""
    w = W.CAUSAL
    bhs = w.B * w.H
    rows = _sample_rows(w.B, w.H, w.Nq, 16384, seed=2, diag_heads=(0, 1, bhs // 2, bhs - 1))
    assert rows.size >= 16384 + 4 * 6 * (w.Nq // 128) - 200
    _run_full_size(cuda_lib, orc, w, rows)


def test_full_size_masked_every_row(cuda_lib, orc):
    """The masked workload (B8 H16 4096^2, window 1024 + padding), every row
    of the output against the oracle (rows see at most 1024 keys, so the
    whole tensor is about 0.27 TFLOP of FP64 work), and the empty rows
    predicted by the mask exactly 0 / -inf."""
    w = W.MASKED
    x, o, lse = _run_full_size(cuda_lib, orc, w, None)
    # row i of batch b sees no key iff i >= L_b + window - 1
    L = x["seqlens_k"].numpy()
    i = np.arange(w.Nq)
    n_empty = 0
    for b in range(w.B):
        empty = i >= L[b] + w.window - 1
        n_empty += int(empty.sum())
        assert np.all(np.isneginf(lse[b][:, empty]))
        assert np.all(o[b][:, empty] == 0)
        assert np.all(np.isfinite(lse[b][:, ~empty]))
    assert n_empty > 0          # the workload exercises rows with no key


# ------------------------------------------------------------ split-KV decode
def run_decode(attn, x, num_splits, scale=None, with_ws=False):
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    sl = x.get("seqlens_k")
    sl = sl.to(dev) if sl is not None else None
    B, H, _, d = q.shape
    ws = torch.empty(attn.attn_decode_workspace_bytes(B, H, d, num_splits), dtype=torch.uint8,
                     device=dev)
    o, lse = attn.attn_decode_splitkv(q, k, v, scale=scale, seqlens_k=sl, num_splits=num_splits,
                                      workspace=ws)
    attn.attn_check_device_error()
    if with_ws:
        return _np(o), _np(lse), ws
    return _np(o), _np(lse)


def test_decode_full_size(cuda_lib, orc):
    w = W.DECODE
    x = W.generate(w)
    o, lse = run_decode(cuda_lib, x, w.num_splits)
    ro, rl = oracle_fwd(orc, x)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what=w.name)


DECODE_SHAPES = [
    # B, H, Nk, d, splits, seqlen_range
    (1, 4, 1000, 128, 8, None),
    (2, 3, 777, 64, 5, None),
    (1, 2, 100, 128, 64, None),          # more splits than 2-key chunks: empty splits
    (3, 2, 4096, 128, 16, (0, 4096)),    # padded, including empty sequences
    (1, 1, 1, 128, 1, None),
    (2, 2, 5000, 128, 1, None),
]


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=[str(s) for s in DECODE_SHAPES])
def test_decode_shapes(cuda_lib, orc, shape):
    B, H, Nk, d, S, sr = shape
    x = W.random_inputs(B, H, 1, Nk, d, seed=Nk % 97, seqlen_range=sr)
    o, lse = run_decode(cuda_lib, x, S)
    mk = W.MASK_PADDING if sr else 0
    ro, rl = oracle_fwd(orc, x, mk)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what=str(shape))


def test_decode_split_partials(cuda_lib, orc):
    """The workspace holds, per (b, h, split), the chunk's normalised output
    and log-sum-exp: compare each with the oracle on that chunk's keys."""
    B, H, Nk, d, S = 1, 2, 1000, 128, 7
    x = W.random_inputs(B, H, 1, Nk, d, seed=21)
    _, _, ws = run_decode(cuda_lib, x, S, with_ws=True)
    slots = B * H * S
    wso = ws[: slots * d * 4].view(torch.float32).reshape(B, H, S, d).cpu().numpy()
    off = ((slots * d * 4 + 255) // 256) * 256
    wsl = ws[off: off + slots * 4].view(torch.float32).reshape(B, H, S).cpu().numpy()
    chunk = -(-Nk // S)
    for s in range(S):
        a, b = s * chunk, min((s + 1) * chunk, Nk)
        y = {"q": x["q"], "k": x["k"][:, :, a:b].contiguous(), "v": x["v"][:, :, a:b].contiguous()}
        ro, rl = oracle_fwd(orc, y)
        assert np.abs(wso[:, :, s] - ro[:, :, 0]).max() <= 1e-3
        assert np.abs(wsl[:, :, s] - rl[:, :, 0]).max() <= 1e-4


# ------------------------------------------------------------ failure path
def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib, orc):
    """A wait on a barrier nothing completes gives up after its limit, the
    error surfaces as ATTN_ERR_TIMEOUT, and the next call still works."""
    cuda_lib.attn_selftest_bounded_wait(2_000_000)
    with pytest.raises(cuda_lib.AttnError) as ei:
        cuda_lib.attn_check_device_error()
    assert ei.value.status == cuda_lib.ATTN_ERR_TIMEOUT
    cuda_lib.attn_check_device_error()          # cleared
    x = W.random_inputs(1, 1, 130, 130, 128, seed=3)
    o, lse = run_fwd(cuda_lib, x)
    ro, rl = oracle_fwd(orc, x)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE)


def test_bad_arguments_raise(cuda_lib):
    dev = torch.device("cuda:0")
    q = torch.zeros(1, 1, 16, 96, dtype=torch.bfloat16, device=dev)
    with pytest.raises(cuda_lib.AttnError) as ei:
        cuda_lib.attn_fwd(q, q, q)
    assert ei.value.status == cuda_lib.ATTN_ERR_UNSUPPORTED
    buf = torch.zeros(1 + 16 * 128, dtype=torch.bfloat16, device=dev)
    qm = buf[1:].view(1, 1, 16, 128)             # 2-byte offset: misaligned
    with pytest.raises(cuda_lib.AttnError) as ei:
        cuda_lib.attn_fwd(qm, qm, qm)
    assert ei.value.status == cuda_lib.ATTN_ERR_INVALID_ARG


def test_decode_bindings_check_output_shapes(cuda_lib):
    """The C entry points see only pointers: the bindings refuse an lse or
    seqlens_k too short for B*H rows / B sequences before calling them."""
    dev = torch.device("cuda:0")
    q = torch.zeros(2, 3, 1, 128, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(2, 3, 64, 128, dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    short_lse = torch.empty(2, 3, dtype=torch.float32, device=dev)[:, :2]
    bad_lens = torch.full((1,), 64, dtype=torch.int32, device=dev)
    for fn in (cuda_lib.attn_decode_splitkv, cuda_lib.attn_decode_splitkv_noalloc):
        with pytest.raises(ValueError):
            fn(q, k, k, o, lse=torch.empty(2, 2, 1, dtype=torch.float32, device=dev),
               num_splits=4)
        with pytest.raises(ValueError):
            fn(q, k, k, o, seqlens_k=bad_lens, num_splits=4)
        with pytest.raises((ValueError, TypeError)):
            fn(q, k, k, o, lse=short_lse.contiguous()[:, :1], num_splits=4)


@pytest.mark.parametrize("d,Nq,mk,sr", [
    (64, 3000, W.MASK_CAUSAL, None),
    (128, 3100, W.MASK_CAUSAL, None),
    (128, 2600, W.MASK_CAUSAL | W.MASK_PADDING, (1, 2600)),
])
def test_fwd_causal_reversed_walk_long(cuda_lib, orc, d, Nq, mk, sr):
    """Causal CTAs whose tile 1 sees the diagonal block more walk their key
    blocks from the diagonal down (tile 0 starting one step later): rows of
    up to 24 key blocks, both head dims (K/V rings of 5 + 4 and 3 + 2
    slots, several wrap-arounds), a ragged last tile, and padded key
    lengths that cut some CTAs' walk short, element by element against the
    oracle."""
    x = W.random_inputs(2, 2, Nq, Nq, d, seed=Nq + d, seqlen_range=sr)
    o, lse = run_fwd(cuda_lib, x, mk)
    ro, rl = oracle_fwd(orc, x, mk)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what="d%d Nq%d" % (d, Nq))


# ------------------------------------------------ host-memory pipelined API
@pytest.mark.parametrize("shape", [
    (2, 3, 300, 300, 128, W.MASK_CAUSAL, 0, None, 4),
    (3, 2, 257, 513, 64, 0, 0, None, 5),
    (2, 4, 400, 400, 128, W.MASK_WINDOW | W.MASK_PADDING, 96, (0, 400), 3),
])
def test_fwd_from_host_matches_device_call(cuda_lib, orc, shape):
    """attn_fwd_from_host (copies pipelined with the kernel by head groups)
    gives bit for bit the device-resident attn_fwd result."""
    B, H, Nq, Nk, d, mk, win, sr, chunks = shape
    x = W.random_inputs(B, H, Nq, Nk, d, seed=B * 100 + H, seqlen_range=sr)
    o_dev, l_dev = run_fwd(cuda_lib, x, mk, win)
    hq, hk, hv = (x[n].pin_memory() for n in ("q", "k", "v"))
    ho = torch.zeros(B, H, Nq, d, dtype=torch.bfloat16).pin_memory()
    hl = torch.zeros(B, H, Nq, dtype=torch.float32).pin_memory()
    cuda_lib.attn_fwd_from_host(hq, hk, hv, ho, hl, mask_kind=mk, window=win,
                                seqlens_k=x["seqlens_k"], chunks=chunks)
    torch.cuda.synchronize()
    cuda_lib.attn_check_device_error()
    assert np.array_equal(ho.float().numpy(), o_dev)
    assert np.array_equal(hl.numpy(), l_dev)
    ro, rl = oracle_fwd(orc, x, mk, win)
    assert_close(ho.float().numpy(), hl.numpy(), ro, rl, TOL_O_BF16, TOL_LSE, what=str(shape))


@pytest.mark.parametrize("chunks,slots", [(5, 2), (7, 4), (3, 1)])
def test_fwd_from_host_slot_counts(cuda_lib, chunks, slots):
    """The host pipeline with fewer or more device slots than the default
    (each slot reused once its previous group has been copied out) gives
    the device-resident result bit for bit."""
    B, H, Nq, Nk, d = 2, 4, 300, 420, 128
    x = W.random_inputs(B, H, Nq, Nk, d, seed=77 + slots)
    o_dev, l_dev = run_fwd(cuda_lib, x, W.MASK_CAUSAL)
    hq, hk, hv = (x[n].pin_memory() for n in ("q", "k", "v"))
    ho = torch.zeros(B, H, Nq, d, dtype=torch.bfloat16).pin_memory()
    hl = torch.zeros(B, H, Nq, dtype=torch.float32).pin_memory()
    pipe = cuda_lib.HostPipeline(B, H, Nq, Nk, d, chunks=chunks, slots=slots)
    for _ in range(2):                       # the pipeline is reusable across calls
        ho.zero_()
        cuda_lib.attn_fwd_from_host(hq, hk, hv, ho, hl, mask_kind=W.MASK_CAUSAL, pipeline=pipe)
        torch.cuda.synchronize()
        cuda_lib.attn_check_device_error()
        assert np.array_equal(ho.float().numpy(), o_dev)
        assert np.array_equal(hl.numpy(), l_dev)


@pytest.mark.parametrize("mk,sr", [(0, None), (W.MASK_CAUSAL | W.MASK_PADDING, (1, 256))])
def test_fwd_from_host_ramped_groups(cuda_lib, mk, sr):
    """Enough heads for the ramped group sizes (2 x 16 heads in groups of at
    most 8: 2, 4, 8, 8, 4, 4, 2 heads): bit for bit the device result,
    including the per-head key lengths of every group."""
    B, H, Nq, Nk, d, chunks = 2, 16, 256, 256, 64, 4
    assert cuda_lib.attn_fwd_host_groups(B, H, chunks) == 7
    x = W.random_inputs(B, H, Nq, Nk, d, seed=4321, seqlen_range=sr)
    o_dev, l_dev = run_fwd(cuda_lib, x, mk)
    hq, hk, hv = (x[n].pin_memory() for n in ("q", "k", "v"))
    ho = torch.zeros(B, H, Nq, d, dtype=torch.bfloat16).pin_memory()
    hl = torch.zeros(B, H, Nq, dtype=torch.float32).pin_memory()
    cuda_lib.attn_fwd_from_host(hq, hk, hv, ho, hl, mask_kind=mk, seqlens_k=x["seqlens_k"],
                                chunks=chunks, slots=3)
    torch.cuda.synchronize()
    cuda_lib.attn_check_device_error()
    assert np.array_equal(ho.float().numpy(), o_dev)
    assert np.array_equal(hl.numpy(), l_dev)


def test_fwd_from_host_pageable_no_lse_and_degenerate(cuda_lib):
    """attn_fwd_host with pageable (not page-locked) host buffers, without
    lse, with more groups than heads, and with no keys at all."""
    B, H, Nq, Nk, d = 1, 3, 200, 330, 64
    x = W.random_inputs(B, H, Nq, Nk, d, seed=91)
    o_dev, _ = run_fwd(cuda_lib, x, W.MASK_WINDOW, 50)
    ho = torch.zeros(B, H, Nq, d, dtype=torch.bfloat16)
    cuda_lib.attn_fwd_from_host(x["q"], x["k"], x["v"], ho, None, mask_kind=W.MASK_WINDOW,
                                window=50, chunks=7, slots=2)
    torch.cuda.synchronize()
    cuda_lib.attn_check_device_error()
    assert np.array_equal(ho.float().numpy(), o_dev)
    # Nk = 0: every row empty
    x0 = W.random_inputs(2, 2, 130, 0, 128, seed=92)
    ho = torch.full((2, 2, 130, 128), 7.0, dtype=torch.bfloat16).pin_memory()
    hl = torch.zeros(2, 2, 130, dtype=torch.float32).pin_memory()
    cuda_lib.attn_fwd_from_host(x0["q"].pin_memory(), x0["k"], x0["v"], ho, hl, chunks=3)
    torch.cuda.synchronize()
    cuda_lib.attn_check_device_error()
    assert torch.all(ho == 0) and torch.all(torch.isneginf(hl))
