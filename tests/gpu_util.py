"""Shared helpers of the GPU tests: inputs, device copies, library calls, parity.

Inputs come from ``workloads`` (seeded, no arithmetic of the layer); quantised
test weights come from the oracle's quantiser; expected values come from the
oracle only.  Nothing here feeds a CUDA result back into the oracle.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

import workloads as W
from oracle import formats as F
from oracle import moe as M
from oracle import quant as Q

MAX_TOL = 1e-2   # max|gpu - oracle| <= 1e-2 * max|oracle|
MEAN_TOL = 5e-3  # sum|gpu - oracle| / sum|oracle| <= 5e-3


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def parity_errors(gpu: np.ndarray, ref: np.ndarray):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(gpu)), "non-finite GPU output"
    diff = np.abs(gpu - ref)
    scale = np.abs(ref).max()
    max_rel = diff.max() / scale if scale > 0 else diff.max()
    denom = np.abs(ref).sum()
    mean_rel = diff.sum() / denom if denom > 0 else diff.sum()
    return float(max_rel), float(mean_rel)


def assert_parity(gpu, ref, what=""):
    mx, mean = parity_errors(gpu, ref)
    assert mx <= MAX_TOL and mean <= MEAN_TOL, f"{what}: max_rel={mx:.3e} mean_rel={mean:.3e}"
    return mx, mean


@dataclasses.dataclass
class HostLayer:
    wl: W.Workload
    x_bits: np.ndarray
    x: np.ndarray
    ids: np.ndarray
    wts: np.ndarray
    em: np.ndarray | None
    c13: np.ndarray
    s13: np.ndarray
    g13: np.ndarray | None
    c2: np.ndarray
    s2: np.ndarray
    g2: np.ndarray | None

    @property
    def m(self):
        return self.x.shape[0]


def host_layer(wl: W.Workload, m: int, seed: int, weights: str = "quantized") -> HostLayer:
    x_bits, x = W.activations(wl, m, seed)
    ids, wts = W.routing(wl, m, seed)
    em = W.expert_map(wl)
    if weights == "quantized":
        w13, w2 = W.float_weights(wl, seed)
        c13, s13, g13 = Q.quantize(w13, wl.fmt)
        c2, s2, g2 = Q.quantize(w2, wl.fmt)
    else:
        c13, s13, g13 = W.random_codes(wl, seed, 0)
        c2, s2, g2 = W.random_codes(wl, seed, 1)
    return HostLayer(wl, x_bits, x, ids, wts, em, c13, s13, g13, c2, s2, g2)


def oracle_out(hl: HostLayer, tokens=None):
    return M.fused_moe(hl.x, hl.c13, hl.s13, hl.g13, hl.c2, hl.s2, hl.g2, hl.ids, hl.wts, hl.wl.act, hl.wl.fmt,
                       hl.wl.num_global_experts, expert_map=hl.em, tokens=tokens, swiglu=hl.wl.swiglu)


class DeviceLayer:
    """Device copies, prepared weights and a workspace for one HostLayer."""

    def __init__(self, hl: HostLayer, path: int | None = None):
        import w4a16_moe_gb300 as b4

        self.b4 = b4
        self.hl = hl
        wl = hl.wl
        self.act = b4.ACTIVATIONS[wl.act]
        self.em = None if hl.em is None else dev(hl.em)
        self.cfg = b4.MoEConfig(
            m=hl.m, top_k=wl.top_k, num_global_experts=wl.num_global_experts,
            num_local_experts=wl.num_local_experts, hidden=wl.hidden, inter=wl.inter,
            format=b4.FORMATS[wl.fmt], path=b4.PATH_AUTO if path is None else path, expert_map=self.em,
            swiglu_alpha=wl.swiglu[0], swiglu_beta=wl.swiglu[1], swiglu_limit=wl.swiglu[2])
        self.x = dev(hl.x_bits).view(torch.bfloat16)
        self.ids = dev(hl.ids)
        self.wts = dev(hl.wts)
        self.w13, self.s13 = b4.prepare_weights(self.cfg, 0, self.act, dev(hl.c13), dev(hl.s13))
        self.w2, self.s2 = b4.prepare_weights(self.cfg, 1, self.act, dev(hl.c2), dev(hl.s2))
        self.g13 = None if hl.g13 is None else dev(hl.g13)
        self.g2 = None if hl.g2 is None else dev(hl.g2)
        self.ws = torch.empty(b4.workspace_bytes(self.cfg, self.act), dtype=torch.uint8, device="cuda")
        self.out = torch.empty(hl.m, wl.hidden, dtype=torch.bfloat16, device="cuda")

    def run(self, stream=None):
        self.b4.fused_moe(self.cfg, self.x, self.w13, self.s13, self.g13, self.w2, self.s2, self.g2, self.ids,
                          self.wts, self.act, self.out, self.ws, stream=stream)

    def result(self):
        torch.cuda.synchronize()
        self.b4.check_status(self.ws)
        return bf16_to_np(self.out)


def bf16_bits_of(values: np.ndarray) -> np.ndarray:
    return F.bf16_bits(values)
