"""Seeded synthetic inputs for the fused W4A16 MoE workloads.

This module holds no arithmetic of the layer: it draws random numbers and
routing decisions, and nothing else.  It is the one module shared by the
oracle-side tests and the CUDA-side tests and benchmark; neither side's code
lives here.

Workloads (the pages name a "Nemotron variant" MoE shape without printing its
sizes, so these synthetic shapes stand in for it):

========  ==========================================================  ============
name      shape                                                       m
========  ==========================================================  ============
tiny      NVFP4, E=8, top_k=2, H=256, I=512, SiLU-SwiGLU               4
decode    NVFP4, E=128, top_k=8, H=4096, I=1536, ReLU^2                1, 2, 4
small     NVFP4, E=64, top_k=6, H=2048, I=1408, SwiGLU, 8 hot experts  16, 64
prefill   NVFP4, E=128, top_k=8, H=4096, I=1536, SwiGLU and ReLU^2     2048
mxfp4     MXFP4, E_g=32 -> E_l=28, top_k=4, H=2880, I=1440, SwiGLU      512
linear    NVFP4 dense linear layer, N = K = 4096 (one weight matrix,    1, 16, 2048
          top-1, no activation: "hidden" is K, "inter" is N)
========  ==========================================================  ============

Recipe: x ~ N(0, 1) rounded to bf16; weights ~ N(0, 0.02) in float32 (the
tests quantise them with the oracle's quantiser); router logits ~ N(0, 1)
(+2 on experts 0..7 for "small"), softmax, top-k, weights renormalised to sum
to 1.  "mxfp4" maps global experts {3, 11, 19, 27} to -1 and the rest in
ascending order to 0..27, then sets round(1% of the routes) to -1 and 32
alternately (invalid ids).  At full size the weights are drawn directly as
random codes and scales (see ``random_codes``), since quantising gigabytes of
float weights on the host would take minutes; the kernels' timing does not
depend on the values.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    fmt: str  # "nvfp4_e4m3_k16" or "mxfp4_e8m0_k32"
    num_global_experts: int
    num_local_experts: int
    top_k: int
    hidden: int
    inter: int
    act: str  # "silu", "relu2" or "swiglu_oai"
    ms: tuple
    hot_experts: int = 0
    drop_globals: tuple = ()
    invalid_frac: float = 0.0
    # (alpha, beta, limit) of "swiglu_oai": the gpt-oss values by default
    swiglu: tuple = (1.702, 1.0, 7.0)

    @property
    def group(self) -> int:
        return 16 if self.fmt.startswith("nvfp4") else 32

    @property
    def n1(self) -> int:
        return 2 * self.inter if self.act in ("silu", "swiglu_oai") else self.inter

    def with_act(self, act: str, swiglu=None) -> "Workload":
        if swiglu is None:
            return dataclasses.replace(self, act=act)
        return dataclasses.replace(self, act=act, swiglu=tuple(swiglu))

    def scaled(self, hidden=None, inter=None, experts=None, top_k=None) -> "Workload":
        """Same structure, smaller sizes (for fast parity cases).

        A workload that drops global experts keeps the same number of drops,
        spread over the smaller global range.
        """
        e = experts or self.num_local_experts
        n_drop = len(self.drop_globals)
        eg = e + n_drop
        drops = ()
        if n_drop:
            step = max(1, eg // n_drop)
            drops = tuple(range(min(3, step - 1), eg, step))[:n_drop]
        return dataclasses.replace(
            self,
            hidden=hidden or self.hidden,
            inter=inter or self.inter,
            num_local_experts=e,
            num_global_experts=eg,
            drop_globals=drops,
            top_k=top_k or self.top_k,
            hot_experts=min(self.hot_experts, e // 2),
        )


NV = "nvfp4_e4m3_k16"
MX = "mxfp4_e8m0_k32"

WORKLOADS = {
    "tiny": Workload("tiny", NV, 8, 8, 2, 256, 512, "silu", (4,)),
    "decode": Workload("decode", NV, 128, 128, 8, 4096, 1536, "relu2", (1, 2, 4)),
    "small": Workload("small", NV, 64, 64, 6, 2048, 1408, "silu", (16, 64), hot_experts=8),
    "prefill": Workload("prefill", NV, 128, 128, 8, 4096, 1536, "silu", (2048,)),
    "linear": Workload("linear", NV, 1, 1, 1, 4096, 4096, "relu2", (1, 16, 2048)),
    "mxfp4": Workload(
        "mxfp4", MX, 32, 28, 4, 2880, 1440, "silu", (512,),
        drop_globals=(3, 11, 19, 27), invalid_frac=0.01,
    ),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def activations(wl: Workload, m: int, seed: int):
    """x ~ N(0, 1) rounded to bf16.  Returns (bits uint16 [m, H], float64 values)."""
    g = _gen(seed * 7919 + 1)
    x = torch.randn(m, wl.hidden, generator=g, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16).copy()
    return bits, x.to(torch.float64).numpy()


def expert_map(wl: Workload):
    """Global -> local expert map (int32 [E_g]) or None when E_g == E_l and no drops."""
    if not wl.drop_globals and wl.num_global_experts == wl.num_local_experts:
        return None
    em = np.full(wl.num_global_experts, -1, dtype=np.int32)
    nxt = 0
    for gidx in range(wl.num_global_experts):
        if gidx in wl.drop_globals:
            continue
        em[gidx] = nxt
        nxt += 1
    if nxt != wl.num_local_experts:
        raise ValueError("expert_map does not cover the local experts")
    return em


def routing(wl: Workload, m: int, seed: int):
    """Softmax top-k routing.  Returns (topk_ids int32 [m, k], topk_weights float32 [m, k])."""
    g = _gen(seed * 7919 + 2)
    logits = torch.randn(m, wl.num_global_experts, generator=g, dtype=torch.float32)
    if wl.hot_experts:
        logits[:, : wl.hot_experts] += 2.0
    probs = torch.softmax(logits, dim=-1)
    w, ids = torch.topk(probs, wl.top_k, dim=-1)
    w = w / w.sum(dim=-1, keepdim=True)
    ids = ids.to(torch.int32).numpy().copy()
    w = w.to(torch.float32).numpy().copy()
    if wl.invalid_frac and m:
        n_bad = int(round(wl.invalid_frac * m * wl.top_k))
        perm = torch.randperm(m * wl.top_k, generator=g)[:n_bad].numpy()
        flat = ids.reshape(-1)
        for i, r in enumerate(sorted(perm.tolist())):
            flat[r] = -1 if i % 2 == 0 else wl.num_global_experts
    return ids, w


def float_weights(wl: Workload, seed: int, experts=None):
    """fp32 weights ~ N(0, 0.02): (w13 [E, N1, H], w2 [E, H, I]).

    ``experts`` restricts generation to a list of local experts (the arrays then
    hold only those experts, in that order); every expert has its own stream,
    so an expert's weights do not depend on which others are drawn.
    """
    ex = range(wl.num_local_experts) if experts is None else experts
    w13, w2 = [], []
    for e in ex:
        g = _gen(seed * 1_000_003 + 17 * int(e) + 3)
        w13.append(torch.randn(wl.n1, wl.hidden, generator=g) * 0.02)
        w2.append(torch.randn(wl.hidden, wl.inter, generator=g) * 0.02)
    return torch.stack(w13).numpy(), torch.stack(w2).numpy()


# plausible block-scale codes for N(0, 0.02) weights: NVFP4 scales near the
# top of the E4M3 range (amax-normalised blocks), MXFP4 exponents near 2^-6.
_NV_SCALE_CODES = np.arange(0x68, 0x7F, dtype=np.uint8)  # 64 .. 448
_MX_SCALE_CODES = np.arange(117, 125, dtype=np.uint8)  # 2^-10 .. 2^-3


def random_codes(wl: Workload, seed: int, which: int):
    """Random packed codes, block scales and global scales for one tensor.

    which = 0: W13 / W1 ([E, N1, H]); which = 1: W2 ([E, H, I]).
    Returns (codes uint8 [E, N, K/2], scales uint8 [E, N, K/g], gs float32 [E] or None).
    """
    n, k = (wl.n1, wl.hidden) if which == 0 else (wl.hidden, wl.inter)
    e = wl.num_local_experts
    rng = np.random.Generator(np.random.Philox(key=seed * 31 + which))
    codes = rng.integers(0, 256, size=(e, n, k // 2), dtype=np.uint8)
    pool = _NV_SCALE_CODES if wl.fmt == NV else _MX_SCALE_CODES
    scales = pool[rng.integers(0, len(pool), size=(e, n, k // wl.group))]
    gs = None
    if wl.fmt == NV:
        gs = (0.02 * 3.0 / (6.0 * 448.0) * (1.0 + 0.1 * rng.random(e))).astype(np.float32)
    return codes, scales, gs
