"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: it only draws tensors. It is the
one piece that both the CUDA path's callers and the FP64 oracle's callers use,
so that both sides see the same stored values. It imports nothing else from
this package.

Recipe (every workload): ``torch.Generator('cpu').manual_seed(seed)``; draw
order seqlens (padded workloads only), then q, k, v; i.i.d. N(0, 1) drawn in
FP32 and, for BF16 workloads, rounded to BF16 once. The oracle is given the
rounded values upcast exactly to FP32.

Named workloads (shapes taken from the pages' worked test and the long-context
figures they discuss):
  tile_test    1 head, 1000 keys (not a block multiple), d = 64, FP32; 128
               query rows placed at tile offset q0 in {0, 300, 872} of an
               Nq = q0 + 128 query array (other rows zero); optional variant
               that raises the scores of the last five keys by exactly 10.
  prefill      B=1, H=64, Nq=Nk=8192, d=128, BF16, no mask.
  causal       B=2, H=32, Nq=Nk=8192, d=128, BF16, causal.
  masked       B=8, H=16, Nq=Nk=4096, d=128, BF16, key lengths uniform in
               [100, 4096], sliding window 1024 plus padding.
  decode       B=1, H=32, one query per head, Nk=131072, d=128, BF16,
               64 key splits.
  softmax      [4096, 32768] FP32 scores, N(0, 1): batches of long vectors
               as in the row-softmax measurements the pages quote.
E4M3 variants of any workload (`generate_fp8`) draw the same FP32 values and
store each of q, k, v as E4M3 with one power-of-two factor per tensor.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import torch

# Mask bit flags (values of the C interface's mask_kind argument).
MASK_NONE = 0
MASK_CAUSAL = 1
MASK_WINDOW = 2
MASK_PADDING = 4


@dataclass
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: torch.dtype
    mask_kind: int = MASK_NONE
    window: int = 0
    seqlen_range: tuple | None = None    # (lo, hi) inclusive, padded masks
    num_splits: int = 0                  # decode only
    q0: int = 0                          # tile_test only
    planted: bool = False                # tile_test only
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def describe(self) -> dict:
        out = {"workload": self.name, "B": self.B, "H": self.H, "Nq": self.Nq,
               "Nk": self.Nk, "d": self.d,
               "dtype": {torch.bfloat16: "bf16", torch.float32: "f32"}[self.dtype],
               "mask_kind": self.mask_kind}
        if self.window:
            out["window"] = self.window
        if self.seqlen_range:
            out["seqlens_k"] = "U[%d,%d]" % self.seqlen_range
        if self.num_splits:
            out["num_splits"] = self.num_splits
        return out


def tile_test(q0: int = 0, causal: bool = False, planted: bool = False) -> Workload:
    return Workload("tile_test_q0_%d%s%s" % (q0, "_causal" if causal else "",
                                            "_planted" if planted else ""),
                    B=1, H=1, Nq=q0 + 128, Nk=1000, d=64, dtype=torch.float32,
                    mask_kind=MASK_CAUSAL if causal else MASK_NONE,
                    q0=q0, planted=planted)


PREFILL = Workload("prefill_B1_H64_N8192_d128_bf16", 1, 64, 8192, 8192, 128,
                   torch.bfloat16)
CAUSAL = Workload("causal_B2_H32_N8192_d128_bf16", 2, 32, 8192, 8192, 128,
                  torch.bfloat16, mask_kind=MASK_CAUSAL)
MASKED = Workload("masked_B8_H16_N4096_d128_bf16_window1024_padded", 8, 16,
                  4096, 4096, 128, torch.bfloat16,
                  mask_kind=MASK_WINDOW | MASK_PADDING, window=1024,
                  seqlen_range=(100, 4096))
DECODE = Workload("decode_B1_H32_Nk131072_d128_bf16_splits64", 1, 32, 1,
                  131072, 128, torch.bfloat16, num_splits=64)


def generate(w: Workload):
    """Draw the inputs of workload `w` on the CPU.

    Returns a dict with q, k, v (CPU tensors in w.dtype, [B,H,N,d],
    contiguous) and seqlens_k (int32 [B] or None).
    """
    g = torch.Generator("cpu").manual_seed(w.seed)
    seqlens = None
    if w.seqlen_range is not None:
        lo, hi = w.seqlen_range
        seqlens = torch.randint(lo, hi + 1, (w.B,), generator=g,
                                dtype=torch.int64).to(torch.int32)
    if w.name.startswith("tile_test"):
        q_rows = torch.randn(128, w.d, generator=g, dtype=torch.float32)
        k = torch.randn(w.Nk, w.d, generator=g, dtype=torch.float32)
        v = torch.randn(w.Nk, w.d, generator=g, dtype=torch.float32)
        if w.planted:
            # Raise the scores of the last five keys by exactly 10: a unit
            # query component times a key component of 10 / scale.
            q_rows[:, w.d - 1] = 1.0
            k[w.Nk - 5:, w.d - 1] += 10.0 / w.scale
        q = torch.zeros(w.Nq, w.d, dtype=torch.float32)
        q[w.q0:w.q0 + 128] = q_rows
        q, k, v = (t.reshape(1, 1, *t.shape).contiguous() for t in (q, k, v))
    else:
        q = torch.randn(w.B, w.H, w.Nq, w.d, generator=g, dtype=torch.float32)
        k = torch.randn(w.B, w.H, w.Nk, w.d, generator=g, dtype=torch.float32)
        v = torch.randn(w.B, w.H, w.Nk, w.d, generator=g, dtype=torch.float32)
    q, k, v = (t.to(w.dtype).contiguous() for t in (q, k, v))
    return {"q": q, "k": k, "v": v, "seqlens_k": seqlens}


E4M3_MAX = 448.0                         # largest finite E4M3 value


def quantize_e4m3(t):
    """Store a tensor as E4M3 with a per-tensor power-of-two factor:
    returns (t8, descale) with t8 = round_e4m3(t / descale) and descale the
    smallest power of two for which max|t| / descale <= 448. t8 * descale is
    then exact in FP32, so both sides see the same real inputs."""
    amax = float(t.abs().max())
    descale = 2.0 ** math.ceil(math.log2(amax / E4M3_MAX)) if amax > 0 else 1.0
    return (t.float() / descale).to(torch.float8_e4m3fn).contiguous(), descale


def generate_fp8(w: Workload):
    """The inputs of workload `w` (same seeded draws as `generate`, in FP32)
    stored as E4M3: dict with q, k, v (float8_e4m3fn), descale_q/k/v, and
    seqlens_k."""
    x = generate(dataclasses.replace(w, dtype=torch.float32))
    out = {"seqlens_k": x["seqlens_k"]}
    for n in ("q", "k", "v"):
        out[n], out["descale_" + n] = quantize_e4m3(x[n])
    return out


SOFTMAX_ROWS, SOFTMAX_N = 4096, 32768    # row softmax workload: [4096, 32768] FP32


def softmax_inputs(rows=SOFTMAX_ROWS, n=SOFTMAX_N, dtype=torch.float32, seed=0, scale=1.0):
    """Seeded [rows, n] matrix of N(0, scale^2) scores (drawn in FP32, rounded
    once to `dtype`), the input of the standalone row softmax."""
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(rows, n, generator=g, dtype=torch.float32) * scale).to(dtype).contiguous()


def random_inputs(B, H, Nq, Nk, d, dtype=torch.bfloat16, seed=0,
                  seqlen_range=None, scale_q=1.0):
    """Generic seeded draw used by the parity tests at reduced sizes.
    Same recipe as `generate` (seqlens, then q, k, v; N(0,1) in FP32, rounded
    to `dtype`). `scale_q` multiplies q before rounding (to widen scores)."""
    g = torch.Generator("cpu").manual_seed(seed)
    seqlens = None
    if seqlen_range is not None:
        lo, hi = seqlen_range
        seqlens = torch.randint(lo, hi + 1, (B,), generator=g,
                                dtype=torch.int64).to(torch.int32)
    q = torch.randn(B, H, Nq, d, generator=g, dtype=torch.float32) * scale_q
    k = torch.randn(B, H, Nk, d, generator=g, dtype=torch.float32)
    v = torch.randn(B, H, Nk, d, generator=g, dtype=torch.float32)
    q, k, v = (t.to(dtype).contiguous() for t in (q, k, v))
    return {"q": q, "k": k, "v": v, "seqlens_k": seqlens}
