"""Stream and graph behaviour of the C interface (GPU only): calls on
separate streams run concurrently without interfering, and the forward,
backward and split-KV decode launches can be captured into a CUDA graph and
replayed (they allocate nothing and do not synchronise), each replay giving
the eager result bit for bit."""
import numpy as np
import pytest
import torch

from online_softmax_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_concurrent_streams_match_serial(cuda_lib):
    dev = torch.device("cuda:0")
    xs = [W.random_inputs(1, 4, 700, 900, 128, seed=s) for s in range(4)]
    ins = [tuple(x[n].to(dev) for n in "qkv") for x in xs]
    serial = []
    for q, k, v in ins:
        o, lse = cuda_lib.attn_fwd(q, k, v, mask_kind=W.MASK_CAUSAL)
        serial.append((o.clone(), lse.clone()))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in ins]
    outs = [(torch.empty_like(q), torch.empty(q.shape[:3], device=dev)) for q, _, _ in ins]
    for _ in range(3):
        for (q, k, v), (o, lse), s in zip(ins, outs, streams):
            cuda_lib.attn_fwd(q, k, v, o=o, lse=lse, mask_kind=W.MASK_CAUSAL, stream=s)
        # a decode on the default stream at the same time
        xd = W.random_inputs(1, 2, 1, 5000, 128, seed=9)
        od, ld = cuda_lib.attn_decode_splitkv(*(xd[n].to(dev) for n in "qkv"), num_splits=16)
        torch.cuda.synchronize()
        cuda_lib.attn_check_device_error()
        for (o, lse), (so, sl) in zip(outs, serial):
            assert torch.equal(o, so) and torch.equal(lse, sl)


def test_cuda_graph_replay_matches_eager(cuda_lib):
    dev = torch.device("cuda:0")
    x = W.random_inputs(1, 2, 384, 384, 128, seed=21)
    q, k, v = (x[n].to(dev) for n in "qkv")
    g = torch.Generator("cpu").manual_seed(22)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16).to(dev)
    xd = W.random_inputs(1, 4, 1, 3000, 128, seed=23)
    qd, kd, vd = (xd[n].to(dev) for n in "qkv")
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(cuda_lib.attn_bwd_workspace_bytes(1, 2, 384, 128), dtype=torch.uint8,
                     device=dev)
    od = torch.empty_like(qd)
    ld = torch.empty(qd.shape[:3], device=dev)
    wsd = torch.empty(cuda_lib.attn_decode_workspace_bytes(1, 4, 128, 8), dtype=torch.uint8,
                      device=dev)
    s = torch.cuda.Stream()

    def step():
        cuda_lib.attn_fwd(q, k, v, o=o, lse=lse, mask_kind=W.MASK_CAUSAL, stream=s)
        cuda_lib.attn_bwd(q, k, v, o, do, lse, dq=dq, dk=dk, dv=dv, mask_kind=W.MASK_CAUSAL,
                          workspace=ws, stream=s)
        cuda_lib.attn_decode_splitkv(qd, kd, vd, o=od, lse=ld, num_splits=8, workspace=wsd,
                                     stream=s)

    with torch.cuda.stream(s):
        step()                       # warm up (kernel attributes, device error word)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, dq, dk, dv, od, ld)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for t in (o, lse, dq, dk, dv, od, ld):
        t.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    cuda_lib.attn_check_device_error()
    for name, got, ref in zip(("o", "lse", "dq", "dk", "dv", "od", "ld"),
                              (o, lse, dq, dk, dv, od, ld), eager):
        if name == "dq":
            # dQ sums one FP32 contribution per key block in whatever order
            # the blocks' reductions reach memory: equal up to that order,
            # i.e. within one BF16 rounding step of the result
            diff = (got.float() - ref.float()).abs()
            assert torch.all(diff <= 2.0 ** -7 * ref.float().abs() +
                             1e-3 * ref.float().abs().max()), name
        else:
            assert torch.equal(got, ref), name
    assert not np.isnan(o.float().cpu().numpy()).any()
