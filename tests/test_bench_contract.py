"""bench.py's output contract, on CPU: the reference arm's JSON line, the
argument guards, and the per-call byte / flop accounting the roofline uses."""

import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def _run(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          cwd=ROOT, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["higher_is_better"] is False and d["unit"] == "us/call"
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"].startswith("decode NVFP4 MoE") and d["config"]["workload"].endswith("m=1")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["value"] > 0 and abs(d["ms_per_step"] - d["value"] / 1e3) < 1e-3


def test_argument_guards():
    r = _run("--warmup", "2")
    assert r.returncode != 0 and "warmup" in r.stderr
    r = _run("--workload", "linear:none:1")
    assert r.returncode != 0 and "secondary" in r.stderr


def test_call_accounting_counts_each_hit_expert_once():
    wl = W.WORKLOADS["decode"]
    b1 = wl.inter * wl.hidden // 2 + wl.inter * wl.hidden // 16 + 4  # W1 codes + E4M3 scales + fp32 gs
    b2 = wl.hidden * wl.inter // 2 + wl.hidden * wl.inter // 16 + 4
    ids = np.array([[0, 1, 2, 3, 4, 5, 6, 7], [7, 6, 5, 4, 3, 2, 1, 0]], np.int32)  # 8 distinct experts, twice
    a = bench.call_accounting(wl, 2, ids, None)
    assert a["experts_hit"] == 8 and a["routes"] == 16
    assert a["weight_bytes"] == 8 * (b1 + b2)
    assert a["bytes"] == 8 * (b1 + b2) + 2 * wl.hidden * 2 * 2 + 2 * wl.top_k * 8
    assert a["flops"] == 2.0 * 16 * (wl.inter * wl.hidden + wl.hidden * wl.inter)
    # invalid ids and experts mapped away carry no bytes
    wl_mx = W.WORKLOADS["mxfp4"]
    em = W.expert_map(wl_mx)
    ids = np.array([[-1, 32, 3, 11]], np.int32)  # invalid, invalid, dropped by the map, dropped by the map
    a = bench.call_accounting(wl_mx, 1, ids, em)
    assert a["experts_hit"] == 0 and a["weight_bytes"] == 0 and a["routes"] == 0


def test_traffic_hash_ignores_comments():
    """The measured traffic stays attached to unchanged kernel code."""
    h1 = bench.source_hash(["int f() { return 1; }  // one\n/* block\n comment */\n", "x"])
    h2 = bench.source_hash(["// a new comment\n\nint f() { return 1; }\n", "x  "])
    h3 = bench.source_hash(["int f() { return 2; }\n", "x"])
    assert h1 == h2 != h3
    for fam in bench.KERNEL_SOURCES:
        assert len(bench.kernel_source_hash(fam)) == 16


def test_traffic_table_families_follow_the_dispatch_rule():
    """Each recorded ncu traffic figure is keyed by the kernel family that
    serves its workload under AUTO (the small-m path up to m = 16, and up to
    m = 64 while m * top_k <= 2 E_local; within it the per-route kernel for
    m <= 4, m * top_k <= E_local, or <= 2 E_local and <= 256 routes; else the
    grouped GEMMs, weights on N below 96 routes per local expert)."""
    from types import SimpleNamespace

    for (fam, key, m) in bench.NCU_TRAFFIC:
        name, act = key.split(":")
        wl = W.WORKLOADS[name].with_act(act)
        r, e = m * wl.top_k, wl.num_local_experts
        decode = m <= 16 or (m <= 64 and r <= 2 * e)
        b = SimpleNamespace(decode=decode, wl=wl, m=m)
        assert bench.kernel_family(b) == fam, (fam, key, m)
        if not decode:
            assert (fam == "grouped_wn") == (r < 96 * e)


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    """The N > 1 host logic (replicas, max over ranks) on CPU with gloo."""
    import socket

    import torch.multiprocessing as mp

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def test_reference_arm_prints_nothing_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, cwd=ROOT, timeout=600, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""
