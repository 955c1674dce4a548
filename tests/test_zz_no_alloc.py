"""b4_fused_moe_noalloc: the fused layer for callers that cannot allocate.

Plugin hooks of inference runtimes and custom-op slots of frameworks get only
their input and output buffers; the host's allocator owns the device memory
and a cudaMalloc from inside the hook is not allowed.  The library serves them
from a static device array instead of a caller workspace.  These tests check
that two calls in a row through that entry point give the result of
b4_fused_moe with a workspace (bit for bit on the decode path, whose top-k sum
has a fixed order; within the parity tolerance on the grouped path, whose fp32
combine order follows atomics), that the second call leaves the device's free
memory unchanged, and that a shape too large for the array is refused.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""

import ctypes

import pytest
import torch

import workloads as W
from gpu_util import DeviceLayer, assert_parity, bf16_to_np, host_layer

CASES = [("decode", W.WORKLOADS["decode"].scaled(hidden=512, inter=384, experts=16), 4, 1),
         ("grouped", W.WORKLOADS["prefill"].scaled(hidden=512, inter=320, experts=12), 100, 2),
         ("mxfp4", W.WORKLOADS["mxfp4"].scaled(hidden=352, inter=160, experts=7), 3, 0),
         ("decode_full", W.WORKLOADS["decode"], 1, 0)]


def _noalloc(dl, out, status, stream=None):
    dl.b4.fused_moe_noalloc(dl.cfg, dl.x, dl.w13, dl.s13, dl.g13, dl.w2, dl.s2, dl.g2, dl.ids, dl.wts, dl.act, out,
                            device_status=status, stream=stream)


@pytest.mark.gpu
@pytest.mark.parametrize("name,wl,m,path", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry_point(name, wl, m, path):
    # the full-size case compares two GPU entry points only: random codes (no quantiser run)
    hl = host_layer(wl, m, seed=31, weights="random" if name.endswith("_full") else "quantized")
    dl = DeviceLayer(hl, path=path)
    assert dl.b4.workspace_bytes(dl.cfg, dl.act) <= dl.b4.NOALLOC_SCRATCH_BYTES
    dl.run()
    want = dl.result()  # synchronises and checks the workspace status word

    out = torch.empty_like(dl.out)
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out.fill_(123.0)
        status.fill_(-1)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        _noalloc(dl, out, status)
        torch.cuda.synchronize()
        if call == 1:  # the first call may load the library's device code
            assert torch.cuda.mem_get_info()[0] == free_before, "device memory changed during the call"
        assert status.tolist() == [0, 0], f"device status {status.tolist()}"
        assert not torch.any(out == 123.0), "out was not written in full"
        if path == 2:
            assert_parity(bf16_to_np(out), want, f"{name} call {call}")
        else:
            assert torch.equal(out, dl.out), f"{name} call {call} differs from b4_fused_moe"


AFTER = [("grouped", CASES[1][1], 120, 9, 2), ("decode", CASES[0][1], 64, 4, 1)]


@pytest.mark.gpu
@pytest.mark.parametrize("name,wl,m_big,m_small,path", AFTER, ids=[a[0] for a in AFTER])
def test_noalloc_after_another_shape(name, wl, m_big, m_small, path):
    """A call on a smaller shape after a larger one reads nothing the larger
    left (partials, markers, counters), and reports a clear status word.  On
    the decode path the larger call runs the route-grouped kernel and the
    smaller one the per-route kernel."""
    big = DeviceLayer(host_layer(wl, m_big, seed=32), path=path)
    small = DeviceLayer(host_layer(wl, m_small, seed=33), path=path)
    small.run()
    want = small.result()
    tmp = torch.empty_like(big.out)
    out = torch.empty_like(small.out)
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    _noalloc(big, tmp, status)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0], f"device status after the larger call {status.tolist()}"
    status.fill_(-1)
    _noalloc(small, out, status)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0], f"device status after the smaller call {status.tolist()}"
    if path == 2:
        assert_parity(bf16_to_np(out), want, f"{name}: small after big")
    else:
        assert torch.equal(out, small.out), f"{name}: small after big differs from b4_fused_moe"


def test_noalloc_refuses_oversized_shape():
    """The prefill shape (m = 2048, H = 4096, I = 1536, top_k = 8) needs more
    scratch than the static array holds; the call is refused before any launch
    (no device is touched, so this runs without a GPU)."""
    import w4a16_moe_gb300 as b4

    wl = W.WORKLOADS["prefill"]
    cfg = b4.MoEConfig(m=2048, top_k=wl.top_k, num_global_experts=wl.num_global_experts,
                       num_local_experts=wl.num_local_experts, hidden=wl.hidden, inter=wl.inter)
    need = b4.workspace_bytes(cfg, b4.SILU)
    assert need > b4.NOALLOC_SCRATCH_BYTES
    # raw C call with null buffers: the size check comes before any pointer is used
    st = b4.raw_lib().b4_fused_moe_noalloc(ctypes.byref(cfg._c()), None, None, None, None, None, None, None, None,
                                           None, b4.SILU, None, None, None)
    assert st == b4.B4_ERR_WORKSPACE_TOO_SMALL
    msg = b4.last_error()
    assert str(need) in msg and str(b4.NOALLOC_SCRATCH_BYTES) in msg, msg
    # the binding's constant is the header's
    import os
    import re

    header = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                               "b4moe.h")).read()
    shift = int(re.search(r"#define B4_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << 20\)", header).group(1))
    assert shift << 20 == b4.NOALLOC_SCRATCH_BYTES
