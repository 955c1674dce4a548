"""The device failure path, exercised without a GPU fault.

Every wait in the library's kernels is bounded: when its limit runs out it
records B4_ERR_TIMEOUT and the wait site in the workspace's status word,
raises the CTA's abort flag and returns.  b4_wait_self_test runs that exact
routine on an mbarrier phase that no thread completes, with a short limit;
these tests check that the status comes back through b4_check_status, that
the wait ends near its limit (no trap, no hang) and that the context is still
usable afterwards.
"""

import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b4():
    import w4a16_moe_gb300 as b4mod

    return b4mod


@pytest.mark.parametrize("limit_us", [1000, 5000])
def test_bounded_wait_runs_out_into_the_status_word(b4, limit_us):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        start.record(stream)
        b4.wait_self_test(ws, limit_us, stream=stream)
        end.record(stream)
    with pytest.raises(b4.B4Error) as ei:
        b4.check_status(ws, stream=stream)
    wall = time.perf_counter() - t0
    assert ei.value.status == b4.B4_ERR_TIMEOUT
    assert "wait site 90" in str(ei.value)
    # the wait ran out near its limit: not earlier, and not much later
    ms = start.elapsed_time(end)
    assert limit_us / 1e3 * 0.9 <= ms <= limit_us / 1e3 + 2.0, ms
    assert wall < 10.0
    # check_status reset the word; the context still works
    b4.check_status(ws, stream=stream)
    y = torch.arange(8, device="cuda", dtype=torch.float32)
    assert float(y.sum()) == 28.0


def test_a_layer_call_after_a_timeout_clears_the_word(b4):
    """The fused layer's first kernel clears the status word, so a call after
    a recorded timeout reports B4_OK."""
    import workloads as W
    from gpu_util import DeviceLayer, assert_parity, host_layer, oracle_out

    wl = W.WORKLOADS["tiny"]
    hl = host_layer(wl, 4, seed=9)
    dl = DeviceLayer(hl)
    b4.wait_self_test(dl.ws, 1000)
    torch.cuda.synchronize()
    dl.run()
    assert_parity(dl.result(), oracle_out(hl), "after a timeout")  # result() calls check_status


def test_self_test_rejects_bad_arguments(b4):
    ws = torch.zeros(4, dtype=torch.uint8, device="cuda")
    with pytest.raises(b4.B4Error) as ei:
        b4.wait_self_test(ws, 1000)
    assert ei.value.status == b4.B4_ERR_INVALID_ARGUMENT
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    for bad in (0, 1000001):
        with pytest.raises(b4.B4Error) as ei:
            b4.wait_self_test(ws, bad)
        assert ei.value.status == b4.B4_ERR_INVALID_ARGUMENT
