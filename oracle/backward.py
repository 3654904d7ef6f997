"""FP64 oracle for the attention backward pass -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module; it shares no code with the CUDA library.

What is computed. For O = softmax(scale * Q K^T + mask) V and a loss whose
gradient with respect to O is dO, the gradients follow from the chain rule
through the row softmax (the backward pass the pages describe under P1 "What
interviewers probe next" -- it stores only the per-row log-sum-exp and
rebuilds P block by block -- and P2's closing paragraph on the backward
pass, which rebuilds the normalised P_j = exp(S_j - LSE) directly):

  per batch b and head h, with S = scale Q K^T (masked entries -inf):
    P   = row softmax of S                 (rows with no visible key: 0)
    dV  = P^T dO
    dP  = dO V^T
    dS  = P * (dP - rowsum(P * dP))        (softmax Jacobian, row by row)
    dQ  = scale dS K
    dK  = scale dS^T Q

The softmax row is the plain definition exp(s - m) / l over the visible keys
(the same three-pass form as the forward oracle). Matrix products use numpy
in float64. Masks follow the forward oracle's readings (causal j <= i;
window i - W < j <= i; padding j < seqlens_k[b]; combined by AND).

Pins: ``tests/test_oracle_backward.py`` (central finite differences of the
pinned FP64 blockwise forward, torch autograd through SDPA in float64, the
shift invariances of softmax, a closed form, and planted mutants).
"""
from __future__ import annotations

import numpy as np

MASK_CAUSAL = 1
MASK_WINDOW = 2
MASK_PADDING = 4


def visible_mask(Nq, Nk, mask_kind, window, Lk):
    """Boolean [Nq, Nk]: key j visible from query i."""
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    vis = j < Lk
    if mask_kind & (MASK_CAUSAL | MASK_WINDOW):
        vis = vis & (j <= i)
    if mask_kind & MASK_WINDOW:
        vis = vis & (j > i - window)
    return np.broadcast_to(vis, (Nq, Nk))


def softmax_rows(S, vis):
    """exp(s - m) / l over the visible entries of each row; empty rows -> 0."""
    P = np.zeros_like(S)
    for r in range(S.shape[0]):
        js = vis[r]
        if not js.any():
            continue
        s = S[r, js]
        m = s.max()
        e = np.exp(s - m)
        P[r, js] = e / e.sum()
    return P


def attention_backward(q, k, v, do, scale, mask_kind=0, window=0, seqlens_k=None):
    """Gradients (dq, dk, dv) in float64, each shaped like its input
    ([B,H,N,d]); inputs may be FP32 or BF16-valued arrays."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        Lk = Nk
        if mask_kind & MASK_PADDING:
            Lk = int(min(max(int(seqlens_k[b]), 0), Nk))
        vis = visible_mask(Nq, Nk, mask_kind, window, Lk)
        for h in range(H):
            S = scale * (q[b, h] @ k[b, h].T)
            P = softmax_rows(S, vis)
            dV = P.T @ do[b, h]
            dP = do[b, h] @ v[b, h].T
            rs = (P * dP).sum(axis=1, keepdims=True)
            dS = P * (dP - rs)
            dq[b, h] = scale * (dS @ k[b, h])
            dk[b, h] = scale * (dS.T @ q[b, h])
            dv[b, h] = dV
    return dq, dk, dv
