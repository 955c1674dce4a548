"""GPU parity of the dense W4A16 linear layer (b4_linear) with the oracle.

Every execution path: the fused small-m kernel (K-split GEMV units, then
output units that sum the split partials) for m <= 4 (or forced up to 64);
the weights-on-N tcgen05 GEMM with K split across units and fp32 partial sums
(few units: small m, moderate N); the weights-on-M GEMM storing bf16 (m >=
96), including N not a multiple of 64 (a strided copy into out).  Also:
capture in a CUDA graph, and the paths agreeing with each other.
"""

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import assert_parity, bf16_to_np, dev
from oracle import linear as L
from oracle import quant as Q

NV, MX = W.NV, W.MX

CASES = [
    # name, fmt, m, n, k, path ("auto" / "decode" / "grouped"), weights
    ("nv_m1_full", NV, 1, 4096, 4096, "auto", "random"),
    ("nv_m2", NV, 2, 768, 1536, "auto", "quantized"),      # per-route small-m kernel
    ("nv_m3", NV, 3, 640, 1024, "auto", "quantized"),      # per-route kernel, three tokens in one grouped unit
    ("nv_m16", NV, 16, 384, 2048, "auto", "quantized"),    # route-grouped small-m kernel
    ("nv_m64", NV, 64, 256, 512, "auto", "quantized"),
    ("nv_m40_decode", NV, 40, 256, 1024, "decode", "quantized"),
    ("nv_m16_full", NV, 16, 4096, 4096, "auto", "random"),
    ("nv_m65_wn", NV, 65, 512, 256, "auto", "quantized"),
    ("nv_m300_wm", NV, 300, 1024, 512, "auto", "quantized"),
    ("nv_m7_grouped", NV, 7, 256, 512, "grouped", "quantized"),
    ("mx_m3_tail", MX, 3, 1440, 2880, "auto", "quantized"),
    ("mx_m200_tail", MX, 200, 1440, 2880, "auto", "quantized"),
    ("nv_m2048_full", NV, 2048, 4096, 4096, "auto", "random"),
]


def _workload(fmt, n, k):
    return W.Workload("linear", fmt, 1, 1, 1, k, n, "relu2", ())


def _inputs(fmt, m, n, k, weights, seed):
    wl = _workload(fmt, n, k)
    x_bits, x = W.activations(wl, m, seed)
    if weights == "quantized":
        g = torch.Generator().manual_seed(seed)
        w = (torch.randn(1, n, k, generator=g) * 0.02).numpy()
        codes, scales, gs = Q.quantize(w, fmt)
    else:
        codes, scales, gs = W.random_codes(wl, seed, 0)
    return x_bits, x, codes, scales, gs


class DeviceLinear:
    def __init__(self, fmt, m, n, k, path, codes, scales, gs, x_bits):
        import w4a16_moe_gb300 as b4

        self.b4 = b4
        paths = {"auto": b4.PATH_AUTO, "decode": b4.PATH_DECODE, "grouped": b4.PATH_GROUPED}
        self.cfg = b4.linear_config(m, n, k, format=b4.FORMATS[fmt], path=paths[path])
        self.w, self.s = b4.prepare_linear_weights(self.cfg, dev(codes), dev(scales))
        self.gs = None if gs is None else dev(np.asarray(gs, np.float32).reshape(1))
        self.x = dev(x_bits).view(torch.bfloat16)
        self.out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.ws = torch.empty(b4.linear_workspace_bytes(self.cfg), dtype=torch.uint8, device="cuda")

    def run(self, stream=None):
        self.b4.linear(self.cfg, self.x, self.w, self.s, self.gs, self.out, self.ws, stream=stream)

    def result(self):
        torch.cuda.synchronize()
        self.b4.check_status(self.ws)
        return bf16_to_np(self.out)


@pytest.mark.gpu
@pytest.mark.parametrize("name,fmt,m,n,k,path,weights", CASES, ids=[c[0] for c in CASES])
def test_linear_matches_oracle(name, fmt, m, n, k, path, weights):
    x_bits, x, codes, scales, gs = _inputs(fmt, m, n, k, weights, seed=41)
    dl = DeviceLinear(fmt, m, n, k, path, codes, scales, gs, x_bits)
    dl.run()
    got = dl.result()
    rows = np.arange(m) if m <= 256 else np.linspace(0, m - 1, 64).astype(np.int64)  # sampled rows at m = 2048
    want = L.linear(x[rows], codes, scales, None if gs is None else gs[0], fmt)
    assert_parity(got[rows], want, name)


@pytest.mark.gpu
def test_linear_paths_agree_and_capture():
    """m = 16 through both paths: each within parity, and a CUDA-graph replay
    with new x equals an eager call."""
    fmt, m, n, k = NV, 16, 512, 1024
    x_bits, x, codes, scales, gs = _inputs(fmt, m, n, k, "quantized", seed=42)
    want = L.linear(x, codes, scales, gs[0], fmt)
    outs = {}
    for path in ("decode", "grouped"):
        dl = DeviceLinear(fmt, m, n, k, path, codes, scales, gs, x_bits)
        dl.run()
        outs[path] = dl.result()
        assert_parity(outs[path], want, path)
        # graph capture: replay after changing x in place
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            dl.run(stream=s)  # eager first: kernel attributes are set outside capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dl.run(stream=s)
        x2_bits, x2 = W.activations(_workload(fmt, n, k), m, 43)
        dl.x.copy_(dev(x2_bits).view(torch.bfloat16))
        dl.out.fill_(float("nan"))
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        assert_parity(dl.result(), L.linear(x2, codes, scales, gs[0], fmt), f"{path} graph replay")
    assert_parity(outs["decode"], outs["grouped"], "decode vs grouped")


@pytest.mark.gpu
def test_linear_small_path_is_reproducible():
    """The small-m path sums split partials in a fixed order: bitwise equal runs."""
    fmt, m, n, k = NV, 4, 1024, 4096
    x_bits, _, codes, scales, gs = _inputs(fmt, m, n, k, "random", seed=44)
    dl = DeviceLinear(fmt, m, n, k, "decode", codes, scales, gs, x_bits)
    dl.run()
    first = dl.out.clone()
    for _ in range(3):
        dl.run()
    torch.cuda.synchronize()
    assert torch.equal(first, dl.out)
