"""CUDA-graph capture of b4_fused_moe (b12x PR #136: decode graph capture with
caller-owned buffers; flashinfer PR #4255 review: work must follow the
caller's stream).

The call is captured on a non-default stream into a torch CUDA graph.  During
capture nothing is allocated; every replay rewrites `out` (a sentinel written
before the replay is gone) and reproduces the eager result -- bit for bit on
the decode path, whose top-k sum has a fixed order, and within the parity
tolerance on the grouped path, whose fp32 combine order follows atomics.
"""

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import DeviceLayer, assert_parity, bf16_to_np, host_layer, oracle_out

pytestmark = pytest.mark.gpu

CASES = [("decode", W.WORKLOADS["decode"].scaled(hidden=512, inter=384, experts=16), 4, 1),
         ("grouped", W.WORKLOADS["prefill"].scaled(hidden=512, inter=320, experts=12), 100, 2),
         ("mxfp4", W.WORKLOADS["mxfp4"].scaled(hidden=352, inter=160, experts=7), 3, 0)]


@pytest.mark.parametrize("name,wl,m,path", CASES, ids=[c[0] for c in CASES])
def test_capture_and_replay(name, wl, m, path):
    hl = host_layer(wl, m, seed=21)
    dl = DeviceLayer(hl, path=path)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dl.run(stream=s)
    s.synchronize()
    eager = dl.out.clone()
    ref = oracle_out(hl)
    assert_parity(bf16_to_np(eager), ref, f"{name} eager")

    # torch's first capture in a process registers its RNG state on the device;
    # do that with a throwaway graph so the check below sees only this call
    warm = torch.cuda.CUDAGraph()
    scratch = torch.zeros(4, device="cuda")
    with torch.cuda.graph(warm, stream=s):
        scratch.add_(1)
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dl.run(stream=s)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before, "the library allocated during capture"

    for _ in range(5):
        dl.out.fill_(123.0)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        got = dl.out.clone()
        assert not torch.any(got == 123.0), "replay did not rewrite out (empty graph?)"
        if path == 2:
            assert_parity(bf16_to_np(got), ref, f"{name} replay")
        else:
            assert torch.equal(got, eager)
    dl.b4.check_status(dl.ws)


def test_timing_events_capture():
    """The timing hook records one event per kernel boundary, also inside a graph."""
    import w4a16_moe_gb300 as b4

    wl = CASES[1][1]
    hl = host_layer(wl, 40, seed=22)
    dl = DeviceLayer(hl, path=2)  # grouped: route pack, FC1, FC2, finalize
    s = torch.cuda.Stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in ev:
        e.record(s)
    with torch.cuda.stream(s):
        dl.run(stream=s)
    s.synchronize()
    b4.set_timing_events(ev)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dl.run(stream=s)
    finally:
        b4.set_timing_events(None)
    g.replay()
    torch.cuda.synchronize()
    ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(4)]
    assert all(t > 0 for t in ms) and sum(ms) < 1000.0, ms
    assert_parity(bf16_to_np(dl.out), oracle_out(hl), "timed replay")
    with pytest.raises(b4.B4Error):
        b4.set_timing_events(ev[:1])


def test_timing_events_decode():
    """The decode path is one launch: events[0] before it, events[1] after."""
    import w4a16_moe_gb300 as b4

    hl = host_layer(CASES[0][1], 2, seed=23)
    dl = DeviceLayer(hl, path=1)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    b4.set_timing_events(ev)
    try:
        dl.run()
    finally:
        b4.set_timing_events(None)
    torch.cuda.synchronize()
    t = ev[0].elapsed_time(ev[1])
    assert 0 < t < 1000.0, t
    assert_parity(bf16_to_np(dl.out), oracle_out(hl), "timed decode")
