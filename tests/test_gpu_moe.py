"""Parity of b4_fused_moe with the oracle.

Tolerance: max|gpu - oracle| <= 1e-2 * max|oracle|
and sum|gpu - oracle| / sum|oracle| <= 5e-3, per call.

* scaled-down workloads with N(0, 0.02) weights quantised by the oracle,
  spanning several tiles and ragged tails, both paths and both activations;
* the five workloads at full size (random codes), in the launch
  configuration the benchmark times, compared on every token up to m = 64 and
  on 64 chosen tokens above (the most and least loaded experts, both sides of
  every route-chunk boundary); the MXFP4 shape at full size with the small-m
  path forced;
* the clamped swiglu on every kernel, with a limit the FC1 outputs cross,
  and at full size on the MXFP4 shape with the gpt-oss parameters;
* tokens that select one expert in several top-k slots, on every path;
* edge cases: m = 0, every route dropped, top-1 single expert, repeated
  calls with one workspace (capacity reuse), a workspace one byte short.
"""

import zlib

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import DeviceLayer, assert_parity, host_layer, oracle_out
from oracle import moe as M

pytestmark = pytest.mark.gpu

# scaled workloads: same structure as the five, sizes the oracle finishes fast
SCALED = {
    "tiny": W.WORKLOADS["tiny"],
    "decode_s": W.WORKLOADS["decode"].scaled(hidden=512, inter=384, experts=16),
    "small_s": W.WORKLOADS["small"].scaled(hidden=320, inter=192, experts=16),
    "prefill_s": W.WORKLOADS["prefill"].scaled(hidden=512, inter=320, experts=12),
    "mxfp4_s": W.WORKLOADS["mxfp4"].scaled(hidden=352, inter=160, experts=7),
    # many experts, few routes each: the small-m path's per-route kernel above m = 4
    "decode_w": W.WORKLOADS["decode"].scaled(hidden=256, inter=192, experts=128),
    # more local experts than the route pack's 2 x 152 CTAs: CTAs that place and
    # copy the rows of several experts each
    "many_e": W.WORKLOADS["decode"].scaled(hidden=128, inter=64, experts=320),
    # the largest top_k the layer takes (32 routes per token)
    "topk32": W.WORKLOADS["decode"].scaled(hidden=128, inter=128, experts=64, top_k=32),
}
CASES = [
    ("tiny", "silu", 4), ("tiny", "silu", 1),
    ("decode_s", "relu2", 1), ("decode_s", "relu2", 2), ("decode_s", "relu2", 4), ("decode_s", "silu", 3),
    ("small_s", "silu", 16), ("small_s", "silu", 64),
    ("prefill_s", "silu", 200), ("prefill_s", "relu2", 200), ("prefill_s", "silu", 37),
    ("mxfp4_s", "silu", 100), ("mxfp4_s", "relu2", 9),
    # routes repeating experts on the per-route kernel: its grouped units (E8M0 scales)
    ("mxfp4_s", "relu2", 4),
    # many routes per expert: the weights-on-M grouped kernel (m * top_k >= 96 * E_l)
    ("mxfp4_s", "silu", 300), ("tiny", "relu2", 512),
    ("decode_w", "relu2", 6), ("decode_w", "silu", 8), ("decode_w", "relu2", 9),
    # as many routes as local experts: the per-route kernel's boundary (m * top_k = E_l)
    ("decode_w", "relu2", 16),
    # AUTO above m = 16 while an expert gets at most two routes: the small-m
    # path, on the per-route kernel's grouped units; m = 32 fills the group
    # table (256 routes, one thread each)
    ("decode_w", "relu2", 24), ("decode_w", "silu", 32),
    ("many_e", "silu", 100),
    # top_k = 32: per-route grouped units (m = 2 and 4: 64 and 128 routes), the
    # route-grouped kernel (m = 16: 512 routes), the grouped GEMMs (m = 80)
    ("topk32", "relu2", 2), ("topk32", "silu", 4), ("topk32", "relu2", 16), ("topk32", "silu", 80),
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


# the clamped swiglu (swiglu-oai) on every kernel's gated epilogue: the
# per-route small-m kernel with one-route units (decode_s m=1) and grouped
# units (decode_s m=4, decode_w m=24), the route-grouped small-m kernel
# (small_s m=16), the weights-on-N GEMMs (prefill_s m=37, mxfp4_s m=9 on the
# grouped path) and the weights-on-M GEMMs (tiny m=512, mxfp4_s m=300).  The
# limit is one the FC1 outputs of these sizes cross (their spread is about
# 0.02 sqrt(H) = 0.3 .. 0.45), so both clamps act.
OAI_PARAMS = (1.702, 1.0, 0.4)
OAI_CASES = [("decode_s", 1), ("decode_s", 4), ("decode_w", 24), ("small_s", 16), ("prefill_s", 37),
             ("tiny", 512), ("mxfp4_s", 9), ("mxfp4_s", 300)]


@pytest.mark.parametrize("name,m", OAI_CASES, ids=[f"{n}-m{m}" for n, m in OAI_CASES])
@pytest.mark.parametrize("path", ["auto", "decode", "grouped"])
def test_parity_clamped_swiglu(b4, name, m, path):
    if path == "decode" and m > b4.DECODE_MAX_M:
        pytest.skip("decode path caps m")
    wl = SCALED[name].with_act("swiglu_oai", OAI_PARAMS)
    hl = host_layer(wl, m, seed=zlib.crc32(f"oai/{name}/{m}".encode()) % 1000)
    dl = DeviceLayer(hl, path={"auto": b4.PATH_AUTO, "decode": b4.PATH_DECODE, "grouped": b4.PATH_GROUPED}[path])
    dl.run()
    assert_parity(dl.result(), oracle_out(hl), f"swiglu_oai {name}/m={m}/{path}")


FULL = [("tiny", "silu", 4), ("decode", "relu2", 1), ("decode", "relu2", 2), ("decode", "relu2", 4),
        ("small", "silu", 16), ("small", "silu", 64), ("prefill", "silu", 2048), ("prefill", "relu2", 2048),
        ("mxfp4", "silu", 512),
        # the gpt-oss-like MXFP4 shape with the gpt-oss clamped swiglu (1.702, 1, 7)
        ("mxfp4", "swiglu_oai", 512)]


def pick_tokens(hl, n=64, seed=11):
    """At most n tokens for a full-size comparison: every token when m <= n;
    otherwise the first and last token, for the two most loaded local experts
    the tokens of their first and last route and of the routes on both sides
    of every 128- and 160-route chunk boundary (the grouped kernels' route
    chunks, in packed route order), two tokens of each of the three least
    loaded experts, then random tokens."""
    m, k = hl.ids.shape
    if m <= n:
        return np.arange(m)
    loc = M.local_experts(hl.ids, hl.wl.num_global_experts, hl.wl.num_local_experts, hl.em)
    routes = {}
    for t in range(m):
        for j in range(k):
            if loc[t, j] >= 0:
                routes.setdefault(int(loc[t, j]), []).append(t)
    by_load = sorted(routes, key=lambda e: (len(routes[e]), e))
    pick = [0, m - 1]
    for e in by_load[-2:]:
        r = routes[e]
        idx = [0, len(r) - 1]
        for chunk in (128, 160):
            for c in range(chunk, len(r), chunk):
                idx += [c - 1, c]
        pick += [r[i] for i in idx]
    for e in by_load[:3]:
        pick += routes[e][:2]
    pick = list(dict.fromkeys(pick))[:n]
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(m), pick)
    pick += rng.choice(rest, size=n - len(pick), replace=False).tolist()
    return np.array(sorted(pick))


@pytest.mark.parametrize("name,act,m", FULL, ids=[f"{n}-{a}-m{m}" for n, a, m in FULL])
def test_parity_full_size_sampled(b4, name, act, m):
    wl = W.WORKLOADS[name].with_act(act)
    hl = host_layer(wl, m, seed=7, weights="random")
    dl = DeviceLayer(hl)
    dl.run()
    got = dl.result()
    toks = pick_tokens(hl)
    assert len(toks) == min(m, 64)
    ref = oracle_out(hl, tokens=toks)
    assert_parity(got[toks], ref, f"{name}/{act}/m={m} ({len(toks)} tokens)")


FORCED = [("mxfp4", "silu", 4), ("mxfp4", "relu2", 4), ("mxfp4", "silu", 24), ("decode", "silu", 8),
          ("decode", "relu2", 16), ("mxfp4", "silu", 12), ("mxfp4", "swiglu_oai", 12)]


@pytest.mark.parametrize("name,act,m", FORCED, ids=[f"{n}-{a}-m{m}" for n, a, m in FORCED])
def test_parity_full_size_decode_forced(b4, name, act, m):
    """Full-size shapes on the small-m path whatever AUTO would pick: the
    MXFP4 workload (E8M0 scales per 32, H = 2880 and I = 1440 not multiples of
    128, an expert_map dropping experts, invalid ids) on the per-route kernel
    with one route per unit (m = 4), with grouped units (m = 12: 48 routes on
    28 local experts) and on the route-grouped kernel (m = 24); the decode
    workload with grouped units at m = 16 (128 routes on 128 experts)."""
    wl = W.WORKLOADS[name].with_act(act)
    hl = host_layer(wl, m, seed=13, weights="random")
    dl = DeviceLayer(hl, path=b4.PATH_DECODE)
    dl.run()
    assert_parity(dl.result(), oracle_out(hl), f"{name}/{act}/m={m} decode forced")


DUP = [("decode_s", "relu2", 3), ("decode_s", "silu", 4), ("small_s", "silu", 16), ("mxfp4_s", "silu", 40)]


@pytest.mark.parametrize("name,act,m", DUP, ids=[f"{n}-{a}-m{m}" for n, a, m in DUP])
@pytest.mark.parametrize("path", ["auto", "decode", "grouped"])
def test_duplicate_expert_ids_within_a_token(b4, name, act, m, path):
    """A token may select the same expert in several top-k slots: each slot is
    its own route, weighted by its own router weight."""
    wl = SCALED[name].with_act(act)
    hl = host_layer(wl, m, seed=zlib.crc32(f"dup/{name}/{m}".encode()) % 1000)
    k = wl.top_k
    hl.ids[0, 1] = hl.ids[0, 0]                       # two slots, one expert
    hl.ids[m - 1, :] = hl.ids[m - 1, 0]               # every slot the same expert
    if m > 2:
        hl.ids[1, k - 1] = hl.ids[1, 0]               # first and last slot
    dl = DeviceLayer(hl, path={"auto": b4.PATH_AUTO, "decode": b4.PATH_DECODE, "grouped": b4.PATH_GROUPED}[path])
    dl.run()
    assert_parity(dl.result(), oracle_out(hl), f"dup {name}/{act}/m={m}/{path}")


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
