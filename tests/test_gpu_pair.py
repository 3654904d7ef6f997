"""The forward on CTA pairs (tcgen05 cta_group::2), a compile-time option.

Built with ATTN_FWD_PAIR=1, the BF16 forward at d = 128 runs each MMA on the
tensor cores of two SMs: M = 256 query rows, 128 from each CTA of a cluster
of two, with each CTA loading half of every K block (64 keys) and half of
every V block (64 head dims) and the first CTA issuing every MMA. The
arithmetic per element is the same as the one-CTA kernel's (the same
products in the same K order, the same softmax code), so this file checks
the pair build against the FP64 oracle at the usual tolerances and against
the default build bit for bit -- except under causal masks, where the
one-CTA kernel walks a CTA's key blocks from the diagonal down and the two
agree to rounding. It is not the default because it measured slower on
GB300: every P hand-off crosses to the other SM.
"""
import math
import os

import numpy as np
import pytest
import torch

from test_gpu_parity import TOL_LSE, TOL_O_BF16, assert_close, oracle_fwd
from online_softmax_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pair_lib(cuda_lib):
    from online_softmax_02_gb300 import build as B
    bdir = os.path.join(ROOT, "_build", "attn_pair")
    path = B.build(extra_flags=("-DATTN_FWD_PAIR=1",), out=os.path.join(bdir, "libattn_pair.so"),
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
    # B, H, Nq, Nk, mask, window, seqlen_range: several 512-row units, ragged
    # tails where the second CTA's rows lie past Nq, masks that leave one CTA
    # of a pair without visible keys in blocks the other needs
    (1, 2, 512, 512, 0, 0, None),
    (1, 2, 300, 700, 0, 0, None),
    (2, 3, 1100, 1000, 0, 0, None),
    (1, 2, 1200, 1200, W.MASK_CAUSAL, 0, None),
    (2, 2, 700, 900, W.MASK_CAUSAL, 0, None),
    (3, 2, 1000, 1000, W.MASK_WINDOW | W.MASK_PADDING, 100, (0, 1000)),
    (2, 2, 640, 640, W.MASK_CAUSAL | W.MASK_PADDING, 0, (50, 640)),
    (2, 2, 600, 600, W.MASK_PADDING, 0, (0, 130)),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_pair_against_oracle_and_default(cuda_lib, pair_lib, orc, shape):
    B, H, Nq, Nk, mk, win, sr = shape
    x = W.random_inputs(B, H, Nq, Nk, 128, seed=sum(shape[:4]) % 997, seqlen_range=sr)
    o, lse = _fwd(cuda_lib, pair_lib, x, mk, win)
    ro, rl = oracle_fwd(orc, x, mk, win)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what=str(shape))
    o0, l0 = _fwd(cuda_lib, None, x, mk, win)
    if mk & (W.MASK_CAUSAL | W.MASK_WINDOW):
        # the one-CTA kernel walks a causal CTA's key blocks from the diagonal
        # down (the pair form in key order): the same sums added in another
        # order, equal up to rounding (O: one BF16 step; lse: FP32 sums)
        fin = np.isfinite(l0)
        assert np.array_equal(fin, np.isfinite(lse))
        assert np.abs(lse[fin] - l0[fin]).max(initial=0.0) <= 1e-5
        assert np.all(np.abs(o - o0) <= 2.0 ** -7 * np.maximum(np.abs(o0), 1.0))
    else:
        assert np.array_equal(o, o0) and np.array_equal(lse, l0), "pair build differs from default"


def test_pair_late_max_and_large_scores(cuda_lib, pair_lib, orc):
    x = W.random_inputs(1, 2, 256, 1000, 128, seed=6)
    x["q"][..., -1] = 1.0
    x["k"][:, :, -5:, -1] += 10.0 * math.sqrt(128)
    o, lse = _fwd(cuda_lib, pair_lib, x)
    ro, rl = oracle_fwd(orc, x)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what="late max")
    x = W.random_inputs(1, 2, 600, 700, 128, seed=5, scale_q=30.0)
    o, lse = _fwd(cuda_lib, pair_lib, x, W.MASK_CAUSAL)
    ro, rl = oracle_fwd(orc, x, W.MASK_CAUSAL)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what="large scores")


def test_pair_d64_uses_one_cta_kernel(cuda_lib, pair_lib, orc):
    """d = 64 is outside the pair form (a V half would be 32 head dims); the
    pair build runs it on the one-CTA kernel."""
    x = W.random_inputs(1, 2, 500, 600, 64, seed=9)
    o, lse = _fwd(cuda_lib, pair_lib, x, W.MASK_CAUSAL)
    ro, rl = oracle_fwd(orc, x, W.MASK_CAUSAL)
    assert_close(o, lse, ro, rl, TOL_O_BF16, TOL_LSE, what="d64")
