"""Parity of b4_fused_moe with the oracle.

Tolerance: max|gpu - oracle| <= 1e-2 * max|oracle|
and sum|gpu - oracle| / sum|oracle| <= 5e-3, per call.

* scaled-down workloads with N(0, 0.02) weights quantised by the oracle,
  spanning several tiles and ragged tails, both paths and both activations;
* the five workloads at full size (random codes), compared on sampled tokens
  the oracle computes one by one, in the launch configuration the benchmark
  times;
* edge cases: m = 0, every route dropped, top-1 single expert, repeated
  calls with one workspace (capacity reuse), a workspace one byte short.
"""

import zlib

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import DeviceLayer, assert_parity, host_layer, oracle_out

pytestmark = pytest.mark.gpu

# scaled workloads: same structure as the five, sizes the oracle finishes fast
SCALED = {
    "tiny": W.WORKLOADS["tiny"],
    "decode_s": W.WORKLOADS["decode"].scaled(hidden=512, inter=384, experts=16),
    "small_s": W.WORKLOADS["small"].scaled(hidden=320, inter=192, experts=16),
    "prefill_s": W.WORKLOADS["prefill"].scaled(hidden=512, inter=320, experts=12),
    "mxfp4_s": W.WORKLOADS["mxfp4"].scaled(hidden=352, inter=160, experts=7),
}
CASES = [
    ("tiny", "silu", 4), ("tiny", "silu", 1),
    ("decode_s", "relu2", 1), ("decode_s", "relu2", 2), ("decode_s", "relu2", 4), ("decode_s", "silu", 3),
    ("small_s", "silu", 16), ("small_s", "silu", 64),
    ("prefill_s", "silu", 200), ("prefill_s", "relu2", 200), ("prefill_s", "silu", 37),
    ("mxfp4_s", "silu", 100), ("mxfp4_s", "relu2", 9),
    # many routes per expert: the weights-on-M grouped kernel (m * top_k >= 96 * E_l)
    ("mxfp4_s", "silu", 300), ("tiny", "relu2", 512),
]


@pytest.fixture(scope="module")
def b4():
    import w4a16_moe_gb300 as b4mod

    return b4mod


@pytest.mark.parametrize("name,act,m", CASES, ids=[f"{n}-{a}-m{m}" for n, a, m in CASES])
@pytest.mark.parametrize("path", ["auto", "decode", "grouped"])
def test_parity_scaled(b4, name, act, m, path):
    if path == "decode" and m > b4.DECODE_MAX_M:
        pytest.skip("decode path caps m")
    wl = SCALED[name].with_act(act)
    hl = host_layer(wl, m, seed=zlib.crc32(f"{name}/{act}/{m}".encode()) % 1000)
    dl = DeviceLayer(hl, path={"auto": b4.PATH_AUTO, "decode": b4.PATH_DECODE, "grouped": b4.PATH_GROUPED}[path])
    dl.run()
    got = dl.result()
    ref = oracle_out(hl)
    assert_parity(got, ref, f"{name}/{act}/m={m}/{path}")


FULL = [("tiny", "silu", 4), ("decode", "relu2", 1), ("decode", "relu2", 2), ("decode", "relu2", 4),
        ("small", "silu", 16), ("small", "silu", 64), ("prefill", "silu", 2048), ("prefill", "relu2", 2048),
        ("mxfp4", "silu", 512)]


@pytest.mark.parametrize("name,act,m", FULL, ids=[f"{n}-{a}-m{m}" for n, a, m in FULL])
def test_parity_full_size_sampled(b4, name, act, m):
    wl = W.WORKLOADS[name].with_act(act)
    hl = host_layer(wl, m, seed=7, weights="random")
    dl = DeviceLayer(hl)
    dl.run()
    got = dl.result()
    rng = np.random.default_rng(11)
    toks = np.unique(np.concatenate([[0, m - 1], rng.choice(m, size=min(m, 2 if m > 64 else 6), replace=False)]))
    ref = oracle_out(hl, tokens=toks)
    assert_parity(got[toks], ref, f"{name}/{act}/m={m} tokens {toks.tolist()}")


def test_m_zero_is_a_noop(b4):
    wl = SCALED["tiny"]
    hl = host_layer(wl, 4, seed=1)
    dl = DeviceLayer(hl)
    dl.cfg.m = 0
    dl.out.fill_(7.0)
    dl.run()
    torch.cuda.synchronize()
    assert torch.all(dl.out == 7.0)


@pytest.mark.parametrize("path", [1, 2])
def test_all_routes_dropped_gives_zero(b4, path):
    wl = SCALED["mxfp4_s"]
    hl = host_layer(wl, 5, seed=2)
    hl.ids[:] = -1
    hl.ids[1, 2] = wl.num_global_experts  # out of range
    hl.ids[3, 0] = 3  # mapped to -1 by expert_map
    dl = DeviceLayer(hl, path=path)
    dl.out.fill_(7.0)
    dl.run()
    got = dl.result()
    assert np.all(got == 0)


def test_top1_single_expert(b4):
    wl = W.Workload("dense", "nvfp4_e4m3_k16", 1, 1, 1, 256, 128, "silu", (8,))
    for m, path in ((8, 2), (3, 1)):
        hl = host_layer(wl, m, seed=3)
        dl = DeviceLayer(hl, path=path)
        dl.run()
        assert_parity(dl.result(), oracle_out(hl), f"dense m={m}")


def test_workspace_capacity_reuse_and_size_contract(b4):
    wl = SCALED["prefill_s"]
    hl = host_layer(wl, 60, seed=4)
    dl = DeviceLayer(hl)
    # one workspace sized for m=60 (capacity 64) serves m in (32, 64]
    assert b4.workspace_bytes(dl.cfg, dl.act) == b4.workspace_bytes(
        b4.MoEConfig(64, wl.top_k, wl.num_global_experts, wl.num_local_experts, wl.hidden, wl.inter), dl.act)
    for m in (60, 33, 64):
        sub = host_layer(wl, m, seed=5 + m)
        d2 = DeviceLayer(sub)
        d2.ws = dl.ws
        d2.run()
        assert_parity(d2.result(), oracle_out(sub), f"reuse m={m}")
    short = dl.ws[: dl.ws.numel() - 1]
    with pytest.raises(b4.B4Error) as ei:
        b4.fused_moe(dl.cfg, dl.x, dl.w13, dl.s13, dl.g13, dl.w2, dl.s2, dl.g2, dl.ids, dl.wts, dl.act, dl.out, short)
    assert ei.value.status == b4.B4_ERR_WORKSPACE_TOO_SMALL


def test_decode_path_is_bitwise_reproducible(b4):
    wl = SCALED["decode_s"]
    hl = host_layer(wl, 4, seed=6)
    dl = DeviceLayer(hl, path=1)
    outs = []
    for _ in range(3):
        dl.run()
        torch.cuda.synchronize()
        outs.append(dl.out.clone())
    assert all(torch.equal(outs[0], o) for o in outs[1:])
