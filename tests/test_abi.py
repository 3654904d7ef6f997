"""The C interface without a GPU: libattn.so loads, exports every function
include/attn.h declares, and rejects bad arguments synchronously (these
calls return before any CUDA call, so no device is needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from online_softmax_02_gb300 import build
    build.build()
    import online_softmax_02_gb300 as attn
    return attn.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["attn_fwd", "attn_fwd_f32", "attn_decode_splitkv",
                 "attn_decode_workspace_bytes", "attn_check_device_error",
                 "attn_last_error"]:
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    from online_softmax_02_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (attn_\w+)", out))
    declared = set(declared_functions())
    assert declared <= exported, declared - exported
    # nothing else with the attn_ prefix leaks out
    assert exported == declared, exported - declared
    for name in declared:
        assert hasattr(lib, name)


def test_constants_match_header():
    import online_softmax_02_gb300 as attn
    from online_softmax_02_gb300 import workloads as W
    text = open(HEADER).read()
    vals = dict((k, int(v)) for k, v in re.findall(r"(ATTN_\w+)\s*=\s*(\d+)", text))
    assert vals["ATTN_OK"] == attn.ATTN_OK == 0
    assert vals["ATTN_ERR_INVALID_ARG"] == attn.ATTN_ERR_INVALID_ARG
    assert vals["ATTN_ERR_UNSUPPORTED"] == attn.ATTN_ERR_UNSUPPORTED
    assert vals["ATTN_ERR_CUDA"] == attn.ATTN_ERR_CUDA
    assert vals["ATTN_ERR_TIMEOUT"] == attn.ATTN_ERR_TIMEOUT
    assert vals["ATTN_MASK_CAUSAL"] == W.MASK_CAUSAL
    assert vals["ATTN_MASK_WINDOW"] == W.MASK_WINDOW
    assert vals["ATTN_MASK_PADDING"] == W.MASK_PADDING


def test_version_and_workspace_size(lib):
    assert b"sm_103a" in lib.attn_version()
    # 1*32*64 slots: 2048*128 floats + 2048 floats, each padded to 256 bytes
    assert lib.attn_decode_workspace_bytes(1, 32, 128, 64) == 2048 * 128 * 4 + 2048 * 4
    assert lib.attn_decode_workspace_bytes(1, 1, 64, 3) == 768 + 256
    assert lib.attn_decode_workspace_bytes(1, 1, 64, 5) == 1280 + 256
    assert lib.attn_decode_workspace_bytes(1, 1, 64, 0) == 0
    assert lib.attn_decode_workspace_bytes(1, 1, 64, 1025) == 0


FAKE = 0x10000   # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2),
    (dict(d=64, B=-1), 1),
    (dict(scale=0.0), 1),
    (dict(scale=float("inf")), 1),
    (dict(mask_kind=8), 1),
    (dict(mask_kind=2, window=0), 1),
    (dict(mask_kind=4, seqlens=None), 1),
    (dict(mask_kind=0, seqlens=FAKE), 1),
    (dict(q=FAKE + 8), 1),
    (dict(o=0), 1),
    (dict(H=70000), 2),
])
def test_forward_argument_errors(lib, kw, code):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, H=2, Nq=16, Nk=16, d=128,
             scale=0.125, mask_kind=0, window=0, seqlens=None)
    a.update(kw)
    for fn in (lib.attn_fwd, lib.attn_fwd_f32):
        st = fn(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"],
                a["d"], a["scale"], a["mask_kind"], a["window"], a["seqlens"], None)
        assert st == code
        assert lib.attn_last_error() != b""


def test_forward_empty_problem_is_ok(lib):
    assert lib.attn_fwd(None, None, None, None, None, 0, 4, 16, 16, 128, 0.1, 0, 0, None, None) == 0
    assert lib.attn_fwd(None, None, None, None, None, 1, 4, 0, 16, 64, 0.1, 0, 0, None, None) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(d=32), 2),
    (dict(num_splits=0), 1),
    (dict(num_splits=2000), 1),
    (dict(ws=None), 1),
    (dict(ws_bytes=10), 1),
    (dict(ws=FAKE + 16), 1),
    (dict(k=FAKE + 4), 1),
])
def test_decode_argument_errors(lib, kw, code):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, H=2, Nk=100, d=128, scale=0.1,
             seqlens=None, num_splits=4, ws=FAKE, ws_bytes=1 << 20)
    a.update(kw)
    st = lib.attn_decode_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                                 a["Nk"], a["d"], a["scale"], a["seqlens"], a["num_splits"],
                                 a["ws"], a["ws_bytes"], None)
    assert st == code


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), 2),
    (dict(dq=0.0), 1),
    (dict(dk=float("inf")), 1),
    (dict(dv=-1.0), 1),
    (dict(scale=1e30, dq=1e30), 1),
    (dict(q=FAKE + 8), 1),
    (dict(mask_kind=2, window=0), 1),
])
def test_fwd_fp8_argument_errors(lib, kw, code):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, H=2, Nq=16, Nk=16, d=128,
             scale=0.125, dq=1.0, dk=1.0, dv=1.0, mask_kind=0, window=0, seqlens=None)
    a.update(kw)
    st = lib.attn_fwd_fp8(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"],
                          a["Nk"], a["d"], a["scale"], a["dq"], a["dk"], a["dv"], a["mask_kind"],
                          a["window"], a["seqlens"], None)
    assert st == code
    assert lib.attn_last_error() != b""


@pytest.mark.parametrize("kw,code", [
    (dict(rows=-1), 1),
    (dict(rows=1 << 31), 1),
    (dict(n=0), 1),
    (dict(dtype=7), 2),
    (dict(x=None), 1),
    (dict(x=FAKE + 2), 1),            # FP32 rows must be 4-byte aligned
    (dict(y=FAKE + 1, dtype=1), 1),   # BF16 rows must be 2-byte aligned
    (dict(lse=FAKE + 2), 1),
])
def test_softmax_rows_argument_errors(lib, kw, code):
    a = dict(x=FAKE, y=FAKE, lse=None, rows=4, n=16, dtype=0)
    a.update(kw)
    assert lib.attn_softmax_rows(a["x"], a["y"], a["lse"], a["rows"], a["n"], a["dtype"],
                                 None) == code


def test_softmax_rows_and_exp2_empty_are_ok(lib):
    assert lib.attn_softmax_rows(None, None, None, 0, 16, 0, None) == 0
    assert lib.attn_exp2_soft(None, None, 0, None) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), 1),
    (dict(x=None), 1),
    (dict(y=FAKE + 2), 1),
])
def test_exp2_soft_argument_errors(lib, kw, code):
    a = dict(x=FAKE, y=FAKE, n=8)
    a.update(kw)
    assert lib.attn_exp2_soft(a["x"], a["y"], a["n"], None) == code


def test_host_group_count(lib):
    # groups of at most P = ceil(B*H / groups) heads; with B*H >= 4 P and
    # P >= 4 the first two and the last two groups take P/4 and P/2 heads
    assert lib.attn_fwd_host_groups(1, 64, 16) == 19      # 1, 2, 14 x 4, 2, 2, 1
    assert lib.attn_fwd_host_groups(2, 16, 4) == 7        # 2, 4, 8, 8, 4, 4, 2
    assert lib.attn_fwd_host_groups(1, 16, 4) == 7        # 1, 2, 4, 4, 2, 2, 1
    assert lib.attn_fwd_host_groups(1, 64, 4) == 7        # 4, 8, 16, 16, 8, 8, 4
    assert lib.attn_fwd_host_groups(1, 24, 4) == 7        # 2, 3, 6, 6, 2, 3, 2
    assert lib.attn_fwd_host_groups(2, 3, 3) == 3         # P = 2: no ramp
    assert lib.attn_fwd_host_groups(1, 64, 64) == 64      # P = 1
    assert lib.attn_fwd_host_groups(1, 12, 2) == 2        # B*H < 4 P: no ramp
    assert lib.attn_fwd_host_groups(1, 5, 100) == 5       # more groups than heads
    assert lib.attn_fwd_host_groups(0, 5, 4) == 0
    assert lib.attn_fwd_host_groups(1, 5, 0) == -1
    assert lib.attn_fwd_host_groups(-1, 5, 4) == -1


def test_host_workspace_size(lib):
    # 2*3 heads in groups of 2 (3 groups), 2 slots: per slot q, k, v, o BF16
    # and lse FP32 for 2 heads, each region padded to 256 bytes; then the
    # per-head and per-batch key lengths
    B, H, Nq, Nk, d = 2, 3, 10, 20, 64
    a256 = lambda x: (x + 255) // 256 * 256
    slot = 2 * a256(2 * Nq * d * 2) + 2 * a256(2 * Nk * d * 2) + a256(2 * Nq * 4)
    assert lib.attn_fwd_host_workspace_bytes(B, H, Nq, Nk, d, 3, 2) == 2 * slot + a256(6 * 4 + 2 * 4)
    # more slots than groups: only as many buffer sets as groups
    assert lib.attn_fwd_host_workspace_bytes(B, H, Nq, Nk, d, 3, 8) == 3 * slot + 256
    for bad in ((B, H, Nq, Nk, 96, 3, 2), (B, H, Nq, Nk, d, 0, 2), (B, H, Nq, Nk, d, 3, 0),
                (B, H, Nq, Nk, d, 3, 9), (-1, H, Nq, Nk, d, 3, 2)):
        assert lib.attn_fwd_host_workspace_bytes(*bad) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2),
    (dict(groups=0), 1),
    (dict(slots=0), 1),
    (dict(slots=9), 1),
    (dict(ws=None), 1),
    (dict(ws_bytes=100), 1),
    (dict(ws=FAKE + 16), 1),
    (dict(mask_kind=4, seqlens=None), 1),
    (dict(q=FAKE + 1), 1),
    (dict(lse=FAKE + 2), 1),
    (dict(scale=-1.0), 1),
])
def test_fwd_host_argument_errors(lib, kw, code):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, H=2, Nq=16, Nk=16, d=128,
             scale=0.125, mask_kind=0, window=0, seqlens=None, groups=2, slots=2, ws=FAKE,
             ws_bytes=1 << 24)
    a.update(kw)
    st = lib.attn_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"],
                           a["Nk"], a["d"], a["scale"], a["mask_kind"], a["window"],
                           a["seqlens"], a["groups"], a["slots"], a["ws"], a["ws_bytes"], None)
    assert st == code
    assert lib.attn_last_error() != b""
