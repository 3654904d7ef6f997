"""Host logic of bench.py (CPU): FLOP accounting by visible pairs, and the
multi-rank timing path (max over ranks, whole-job rate) on two gloo ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
from online_softmax_02_gb300 import workloads as W


def _brute_pairs(Nq, Nk, mask_kind, window, L):
    n = 0
    for i in range(Nq):
        for j in range(Nk):
            ok = j < L
            if mask_kind & (W.MASK_CAUSAL | W.MASK_WINDOW):
                ok = ok and j <= i
            if mask_kind & W.MASK_WINDOW:
                ok = ok and j > i - window
            n += ok
    return n


@pytest.mark.parametrize("mask_kind,window,seqlens", [
    (0, 0, None), (W.MASK_CAUSAL, 0, None), (W.MASK_WINDOW, 7, None),
    (W.MASK_WINDOW | W.MASK_PADDING, 5, [30, 3, 0]), (W.MASK_PADDING, 0, [11, 40, 1]),
    (W.MASK_CAUSAL | W.MASK_PADDING, 0, [17, 33, 2]),
])
def test_visible_pairs_matches_brute_force(mask_kind, window, seqlens):
    w = W.Workload("t", B=3, H=2, Nq=33, Nk=37, d=8, dtype=torch.float32,
                   mask_kind=mask_kind, window=window)
    got = bench.visible_pairs(w, seqlens)
    want = sum(_brute_pairs(33, 37, mask_kind, window, 37 if seqlens is None else seqlens[b])
               for b in range(3)) * 2
    assert got == want
    assert bench.flops(w, seqlens) == 4.0 * 8 * want
    # the per-row count the CPU baselines use sums to the same total
    rows = np.arange(3 * 2 * 33)
    per_row = bench.row_visible_keys(w, rows, seqlens)
    assert int(per_row.sum()) == want
    for r in (0, 5, 32, 33, 100, 197):
        b, i = r // (2 * 33), r % 33
        L = 37 if seqlens is None else seqlens[b]
        assert per_row[r] == sum(
            1 for j in range(37) if j < L
            and (not mask_kind & (W.MASK_CAUSAL | W.MASK_WINDOW) or j <= i)
            and (not mask_kind & W.MASK_WINDOW or j > i - window))


def test_workload_flop_counts():
    assert bench.flops(W.PREFILL) == 4.0 * 128 * 64 * 8192 * 8192
    # causal: 8192 * 8193 / 2 visible pairs per head
    assert bench.flops(W.CAUSAL) == 4.0 * 128 * 64 * (8192 * 8193 // 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + 5.0 * rank, True, device="cpu")
        out[rank] = t
    finally:
        torch.distributed.destroy_process_group()


def test_two_rank_max_and_rate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 15.0
    # 2 ranks x 3 steps x 1e12 units in 15 ms
    assert bench.whole_job_rate(1e12, world, 3, out[0]) == pytest.approx(4e14)


def test_traffic_records_follow_their_source_hash(monkeypatch):
    import bench
    for key, rec in bench.NCU_TRAFFIC.items():
        assert rec["bytes_per_launch"] > 0 and rec["file"].endswith(".cu")
        got = bench.traffic_for(key)
        assert got in (None, rec["bytes_per_launch"])
        if got is not None:
            assert bench.traffic_for(key, 0.25) == rec["bytes_per_launch"] * 0.25
    monkeypatch.setitem(bench.NCU_TRAFFIC, "fwd_bf16",
                        dict(bench.NCU_TRAFFIC["fwd_bf16"], sha256="0" * 64))
    assert bench.traffic_for("fwd_bf16") is None
    assert bench.traffic_for("no such kernel") is None


def test_build_cli_needs_out_with_options():
    """A build with compile-time options must name its own library (the
    default libattn.so is never overwritten by an option build)."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "-m", "online_softmax_02_gb300.build", "-D",
                        "ATTN_FWD_PAIR=1"], capture_output=True, text=True,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode != 0 and "--out" in r.stderr
