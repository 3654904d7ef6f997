"""online_softmax_02_gb300 -- exact fused attention with online softmax on
GB300 (sm_103a).

A thin ctypes binding over ``libattn.so`` (C interface in ``include/attn.h``).
This module only marshals arguments: every step of the computation runs in
the library's CUDA kernels. PyTorch is used for device memory and streams.
There is no CPU or PyTorch fallback: if the library is missing, ``load()``
raises.

Functions (same names as the C entry points):
  attn_fwd(q, k, v, ...)            BF16 fused forward -> (o, lse)
  attn_fwd_f32(q, k, v, ...)        FP32 fused forward -> (o, lse)
  attn_fwd_from_host(q, k, v, o, ...)  BF16 forward on host tensors through
                                    attn_fwd_host (copies pipelined with the
                                    kernel by head groups)
  attn_fwd_host_workspace_bytes(B, H, Nq, Nk, d, groups, slots)
  attn_fwd_host_groups(B, H, groups)  head groups (kernel launches) it uses
  attn_bwd(q, k, v, o, dout, lse, ...)  backward -> (dq, dk, dv)
  attn_bwd_workspace_bytes(B, H, Nq, d)
  attn_decode_workspace_bytes(B, H, d, num_splits)
  attn_decode_splitkv(q, k, v, ...) split-KV decode -> (o, lse)
  attn_decode_splitkv_noalloc(q, k, v, o, ...)  the same, no caller workspace
  attn_softmax_rows(x, ...)         standalone row softmax -> (y, lse)
  attn_check_device_error(stream=None)
  attn_selftest_bounded_wait(limit_cycles, stream=None)
"""
from __future__ import annotations

import ctypes
import math
import os

from .workloads import MASK_CAUSAL, MASK_NONE, MASK_PADDING, MASK_WINDOW  # noqa: F401

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")
_lib = None


class AttnError(RuntimeError):
    """A non-OK status from libattn.so; `.status` holds the code."""

    def __init__(self, status: int, message: str):
        super().__init__("attn status %d: %s" % (status, message))
        self.status = status


def load():
    """Load libattn.so (built by ``__graft_entry__.build()`` or
    ``online_softmax_02_gb300/build.py``). Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libattn.so not found at %s: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
    _lib = _configure(ctypes.CDLL(LIB_PATH))
    return _lib


def open_build(path: str):
    """Load another build of libattn.so -- one compiled with compile-time
    options other than the defaults (``build.build(out=..., extra_flags=...)``)
    -- and return its ctypes handle; pass it as ``lib=`` to attn_fwd or
    attn_fwd_fp8. The default library is not affected."""
    if not os.path.exists(path):
        raise ImportError("no library at %s" % path)
    return _configure(ctypes.CDLL(path))


def _configure(lib):
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, P, P]
    lib.attn_fwd.restype = I
    lib.attn_fwd_f32.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, P, P]
    lib.attn_fwd_f32.restype = I
    lib.attn_fwd_host_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    lib.attn_fwd_host_workspace_bytes.restype = S
    lib.attn_fwd_host_groups.argtypes = [I, I, I]
    lib.attn_fwd_host_groups.restype = I
    lib.attn_fwd_host.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, P, I, I, P, S, P]
    lib.attn_fwd_host.restype = I
    lib.attn_fwd_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, F, F, F, F, I, I, P, P]
    lib.attn_fwd_fp8.restype = I
    lib.attn_decode_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_decode_workspace_bytes.restype = S
    lib.attn_decode_splitkv.argtypes = [P, P, P, P, P, I, I, I, I, F, P, I, P, S, P]
    lib.attn_decode_splitkv.restype = I
    lib.attn_decode_splitkv_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, F, P, I, P]
    lib.attn_decode_splitkv_noalloc.restype = I
    lib.attn_bwd_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_bwd_workspace_bytes.restype = S
    lib.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, I, I, P, P, S, P]
    lib.attn_bwd.restype = I
    lib.attn_softmax_rows.argtypes = [P, P, P, ctypes.c_longlong, I, I, P]
    lib.attn_softmax_rows.restype = I
    lib.attn_check_device_error.argtypes = [P]
    lib.attn_check_device_error.restype = I
    lib.attn_exp2_soft.argtypes = [P, P, ctypes.c_longlong, P]
    lib.attn_exp2_soft.restype = I
    lib.attn_selftest_bounded_wait.argtypes = [ctypes.c_longlong, P]
    lib.attn_selftest_bounded_wait.restype = I
    lib.attn_last_error.argtypes = []
    lib.attn_last_error.restype = ctypes.c_char_p
    lib.attn_version.argtypes = []
    lib.attn_version.restype = ctypes.c_char_p
    return lib


def _check(status: int, lib=None):
    if status != ATTN_OK:
        raise AttnError(status, (lib or load()).attn_last_error().decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _require(t, name, dtype, device=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def _fwd(fn, dtype, q, k, v, o, lse, scale, mask_kind, window, seqlens_k, stream,
         out_dtype=None, descales=(), lib=None):
    import torch
    out_dtype = dtype if out_dtype is None else out_dtype
    _require(q, "q", dtype)
    dev = q.device
    _require(k, "k", dtype, dev)
    _require(v, "v", dtype, dev)
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d] matching q")
    if o is None:
        o = torch.empty(q.shape, dtype=out_dtype, device=dev)
    _require(o, "o", out_dtype, dev)
    if tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must have q's shape")
    if lse is not None:
        _require(lse, "lse", torch.float32, dev)
        if tuple(lse.shape) != (B, H, Nq):
            raise ValueError("lse must be [B, H, Nq]")
    if seqlens_k is not None:
        _require(seqlens_k, "seqlens_k", torch.int32, dev)
        if tuple(seqlens_k.shape) != (B,):
            raise ValueError("seqlens_k must be [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(dev):
        st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                float(scale), *[float(f) for f in descales], int(mask_kind), int(window),
                _ptr(seqlens_k), _stream_handle(stream, dev))
    _check(st, lib)
    return o, lse


def attn_fwd(q, k, v, o=None, lse=None, scale=None, mask_kind=MASK_NONE, window=0,
             seqlens_k=None, stream=None, want_lse=True, lib=None):
    """BF16 fused attention forward through ``attn_fwd``.

    q [B,H,Nq,d], k/v [B,H,Nk,d] contiguous BF16 CUDA tensors; returns
    (o [B,H,Nq,d] BF16, lse [B,H,Nq] FP32 or None). Output buffers may be
    passed in to avoid allocation. ``lib``: a handle from ``open_build``
    (default: the library next to this file)."""
    import torch
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    return _fwd((lib or load()).attn_fwd, torch.bfloat16, q, k, v, o, lse, scale, mask_kind,
                window, seqlens_k, stream, lib=lib)


def attn_fwd_fp8(q, k, v, descale_q, descale_k, descale_v, o=None, lse=None, scale=None,
                 mask_kind=MASK_NONE, window=0, seqlens_k=None, stream=None, want_lse=True,
                 lib=None):
    """E4M3 fused attention forward through ``attn_fwd_fp8``.

    q [B,H,Nq,128], k/v [B,H,Nk,128] contiguous ``torch.float8_e4m3fn`` CUDA
    tensors holding the inputs divided by their per-tensor factors
    ``descale_*``; returns (o [B,H,Nq,128] BF16, lse [B,H,Nq] FP32 or None)."""
    import torch
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    return _fwd((lib or load()).attn_fwd_fp8, torch.float8_e4m3fn, q, k, v, o, lse, scale,
                mask_kind, window, seqlens_k, stream, out_dtype=torch.bfloat16,
                descales=(descale_q, descale_k, descale_v), lib=lib)


def attn_fwd_f32(q, k, v, o=None, lse=None, scale=None, mask_kind=MASK_NONE, window=0,
                 seqlens_k=None, stream=None, want_lse=True):
    """FP32 fused attention forward through ``attn_fwd_f32``."""
    import torch
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    return _fwd(load().attn_fwd_f32, torch.float32, q, k, v, o, lse, scale, mask_kind,
                window, seqlens_k, stream)


def attn_bwd_workspace_bytes(B: int, H: int, Nq: int, d: int, lib=None) -> int:
    return int((lib or load()).attn_bwd_workspace_bytes(B, H, Nq, d))


def attn_bwd(q, k, v, o, dout, lse, dq=None, dk=None, dv=None, scale=None,
             mask_kind=MASK_NONE, window=0, seqlens_k=None, workspace=None, stream=None,
             lib=None):
    """Attention backward through ``attn_bwd``: BF16 q, k, v [B,H,N,d], the
    forward's BF16 output o and FP32 lse [B,H,Nq], and the BF16 gradient
    dout of the loss with respect to o. Returns (dq, dk, dv) in BF16.
    ``lib``: a handle from ``open_build`` (default: the library next to this
    file)."""
    import torch
    lib = lib or load()
    _require(q, "q", torch.bfloat16)
    dev = q.device
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _require(t, n, torch.bfloat16, dev)
    _require(lse, "lse", torch.float32, dev)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d]")
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("o and dout must have q's shape")
    if tuple(lse.shape) != (B, H, Nq):
        raise ValueError("lse must be [B, H, Nq]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _require(t, n, torch.bfloat16, dev)
    if seqlens_k is not None:
        _require(seqlens_k, "seqlens_k", torch.int32, dev)
    need = int(lib.attn_bwd_workspace_bytes(B, H, Nq, d))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _require(workspace, "workspace", torch.uint8, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(dev):
        st = lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                          _ptr(dk), _ptr(dv), B, H, Nq, Nk, d, float(scale), int(mask_kind),
                          int(window), _ptr(seqlens_k), _ptr(workspace), workspace.numel(),
                          _stream_handle(stream, dev))
    _check(st, lib)
    return dq, dk, dv


def attn_decode_workspace_bytes(B: int, H: int, d: int, num_splits: int) -> int:
    return int(load().attn_decode_workspace_bytes(B, H, d, num_splits))


def _check_decode_aux(o, q, lse, seqlens_k, B, H, dev):
    """Shapes of the decode outputs and key lengths: the C entry points see
    only pointers, so a short lse or seqlens_k would be written or read past
    its end by the kernels."""
    import torch
    _require(o, "o", torch.bfloat16, dev)
    if tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must have q's shape [B, H, 1, d]")
    if lse is not None:
        _require(lse, "lse", torch.float32, dev)
        if lse.numel() != B * H or (lse.dim() == 3 and tuple(lse.shape) != (B, H, 1)):
            raise ValueError("lse must be [B, H, 1] (B*H FP32 values)")
    if seqlens_k is not None:
        _require(seqlens_k, "seqlens_k", torch.int32, dev)
        if tuple(seqlens_k.shape) != (B,):
            raise ValueError("seqlens_k must be [B]")


def attn_decode_splitkv(q, k, v, o=None, lse=None, scale=None, seqlens_k=None,
                        num_splits=64, workspace=None, stream=None, want_lse=True):
    """Split-KV decode through ``attn_decode_splitkv``: q [B,H,1,d], k/v
    [B,H,Nk,d] BF16. ``workspace``: a CUDA uint8 tensor of at least
    ``attn_decode_workspace_bytes`` bytes (allocated here if None)."""
    import torch
    lib = load()
    _require(q, "q", torch.bfloat16)
    dev = q.device
    _require(k, "k", torch.bfloat16, dev)
    _require(v, "v", torch.bfloat16, dev)
    if q.dim() != 4 or q.shape[2] != 1:
        raise ValueError("q must be [B, H, 1, d]")
    B, H, _, d = q.shape
    Nk = k.shape[2]
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d]")
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, 1), dtype=torch.float32, device=dev)
    _check_decode_aux(o, q, lse, seqlens_k, B, H, dev)
    need = int(lib.attn_decode_workspace_bytes(B, H, d, num_splits))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _require(workspace, "workspace", torch.uint8, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(dev):
        st = lib.attn_decode_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nk, d,
                                     float(scale), _ptr(seqlens_k), int(num_splits),
                                     _ptr(workspace), workspace.numel(),
                                     _stream_handle(stream, dev))
    _check(st)
    return o, lse


def attn_decode_splitkv_noalloc(q, k, v, o, lse=None, scale=None, seqlens_k=None,
                                num_splits=64, stream=None):
    """Split-KV decode through ``attn_decode_splitkv_noalloc``: the same result
    as ``attn_decode_splitkv`` for callers that cannot allocate device memory
    on their call path. The C entry point allocates nothing; its per-split
    partials live in a fixed 4 MiB array inside libattn.so, shared by every
    call on a device (calls that overlap on the GPU race on it). The output
    buffers ``o`` (and ``lse`` if wanted) must be passed in. Problems whose
    partials need more than 4 MiB raise AttnError (ATTN_ERR_INVALID_ARG)."""
    import torch
    lib = load()
    _require(q, "q", torch.bfloat16)
    dev = q.device
    _require(k, "k", torch.bfloat16, dev)
    _require(v, "v", torch.bfloat16, dev)
    if q.dim() != 4 or q.shape[2] != 1:
        raise ValueError("q must be [B, H, 1, d]")
    B, H, _, d = q.shape
    Nk = k.shape[2]
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d]")
    _check_decode_aux(o, q, lse, seqlens_k, B, H, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(dev):
        st = lib.attn_decode_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                             Nk, d, float(scale), _ptr(seqlens_k),
                                             int(num_splits), _stream_handle(stream, dev))
    _check(st)
    return o, lse


def attn_fwd_host_groups(B: int, H: int, groups: int = 4) -> int:
    """Number of head groups (forward kernel launches) attn_fwd_host uses."""
    return int(load().attn_fwd_host_groups(B, H, groups))


def attn_fwd_host_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int, groups: int = 4,
                                  slots: int = 3) -> int:
    return int(load().attn_fwd_host_workspace_bytes(B, H, Nq, Nk, d, groups, slots))


class HostPipeline:
    """The device workspace of ``attn_fwd_host`` for one shape, kept so that
    repeated calls allocate nothing: ``slots`` buffer sets (q, k, v, o, lse)
    of ceil(B*H / chunks) heads each. Create it once for a shape and reuse it
    across calls ordered on one stream."""

    def __init__(self, B, H, Nq, Nk, d, device=None, chunks=4, slots=3):
        import torch
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.B, self.H, self.Nq, self.Nk, self.d = B, H, Nq, Nk, d
        self.chunks, self.slots = int(chunks), int(slots)
        need = attn_fwd_host_workspace_bytes(B, H, Nq, Nk, d, self.chunks, self.slots)
        if need == 0 and B * H > 0:
            raise ValueError("invalid host pipeline arguments")
        self.workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=self.device)


def _require_host(t, name, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError("%s must be a CPU tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def attn_fwd_from_host(q, k, v, o, lse=None, scale=None, mask_kind=MASK_NONE, window=0,
                       seqlens_k=None, pipeline=None, chunks=4, slots=3, stream=None):
    """Fused attention forward for inputs and outputs in host memory, through
    ``attn_fwd_host``.

    q [B,H,Nq,d], k/v [B,H,Nk,d] and o [B,H,Nq,d] are BF16 CPU tensors (pin
    them, e.g. ``.pin_memory()``, for the copies to overlap the kernels); lse
    an optional FP32 CPU [B,H,Nq]; seqlens_k a CPU int32 [B] (padding mask).
    The heads are cut into ``chunks`` groups whose copy-in, kernel and
    copy-out overlap (``slots`` device buffer sets; ``pipeline`` holds a
    reusable workspace). Returns once the work is queued on ``stream`` (the
    current stream by default); synchronise it before reading o / lse."""
    import torch
    lib = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _require_host(t, n, torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, Nq, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d] matching q")
    if tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must have q's shape")
    if lse is not None:
        _require_host(lse, "lse", torch.float32)
        if tuple(lse.shape) != (B, H, Nq):
            raise ValueError("lse must be [B, H, Nq]")
    if seqlens_k is not None:
        _require_host(seqlens_k, "seqlens_k", torch.int32)
        if tuple(seqlens_k.shape) != (B,):
            raise ValueError("seqlens_k must be [B]")
    if pipeline is None:
        pipeline = HostPipeline(B, H, Nq, Nk, d, device=torch.cuda.current_device(),
                                chunks=chunks, slots=slots)
    P = pipeline
    if (P.B * P.H, P.Nq, P.Nk, P.d) != (B * H, Nq, Nk, d):
        raise ValueError("pipeline was built for another shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(P.device):
        st = lib.attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                               float(scale), int(mask_kind), int(window), _ptr(seqlens_k),
                               P.chunks, P.slots, _ptr(P.workspace), P.workspace.numel(),
                               _stream_handle(stream, P.device))
    _check(st)
    return o, lse


def attn_softmax_rows(x, y=None, lse=None, stream=None, want_lse=True):
    """Row softmax of a 2-D CUDA tensor (FP32 or BF16) through
    ``attn_softmax_rows``; returns (y, lse)."""
    import torch
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be float32 or bfloat16")
    _require(x, "x", x.dtype)
    if x.dim() != 2:
        raise ValueError("x must be [rows, n]")
    y = torch.empty_like(x) if y is None else y
    _require(y, "y", x.dtype, x.device)
    if lse is None and want_lse:
        lse = torch.empty(x.shape[0], dtype=torch.float32, device=x.device)
    if lse is not None:
        _require(lse, "lse", torch.float32, x.device)
    dtype = 1 if x.dtype == torch.bfloat16 else 0
    with torch.cuda.device(x.device):
        st = load().attn_softmax_rows(_ptr(x), _ptr(y), _ptr(lse), x.shape[0], x.shape[1], dtype,
                                      _stream_handle(stream, x.device))
    _check(st)
    return y, lse


def attn_check_device_error(stream=None, lib=None):
    """Synchronise and raise AttnError if a kernel gave up a bounded wait."""
    import torch
    h = _stream_handle(stream, torch.cuda.current_device()) if stream is not None else None
    lib = lib or load()
    _check(lib.attn_check_device_error(h), lib)


def attn_exp2_soft(x, y=None, stream=None):
    """Diagnostic: 2^x of a contiguous FP32 CUDA tensor by the forward
    kernels' software exponential (``attn_exp2_soft``)."""
    import torch
    _require(x, "x", torch.float32)
    y = torch.empty_like(x) if y is None else y
    _require(y, "y", torch.float32, x.device)
    with torch.cuda.device(x.device):
        st = load().attn_exp2_soft(_ptr(x), _ptr(y), x.numel(), _stream_handle(stream, x.device))
    _check(st)
    return y


def attn_selftest_bounded_wait(limit_cycles: int, stream=None):
    import torch
    h = _stream_handle(stream, torch.cuda.current_device()) if stream is not None else None
    _check(load().attn_selftest_bounded_wait(int(limit_cycles), h))


def attn_version() -> str:
    return load().attn_version().decode()
