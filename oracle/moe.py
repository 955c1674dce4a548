"""The fused W4A16 mixture-of-experts layer, restated in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix (flashinfer PR #4255, Description and Performance):

* weights are FP4 (NVFP4 or MXFP4), activations bf16;
* FC1 is a grouped GEMM over the routed tokens with the SiLU-SwiGLU ("silu")
  or ReLU^2 ("relu2") activation fused into its epilogue;
* FC2 is a grouped GEMM whose store epilogue folds in the top-k sum;
* a separate small-m decode path computes the same thing.

This module is the plain definition of what those kernels compute.  Readings
taken where the pages are silent:

* W13 rows [0, I) are the gate projection and rows [I, 2I) the up projection;
  ReLU^2 is non-gated with W1 of I rows;
* the FC1 global scale gs13 multiplies the FC1 accumulator before the
  activation; the FC2 global scale gs2 multiplies the FC2 accumulator;
* silu(z) = z / (1 + exp(-z)), no clamp and no alpha;
* "swiglu_oai" -- swiglu-oai, which the Description lists as not included
  and the b12x PR's CodeRabbit summary alludes to ("SwiGLU parameters"),
  defined by neither -- is read as the clamped swiglu of the gpt-oss models:
  g' = min(gate, limit), u' = clip(up, -limit, limit),
  h = g' * sigmoid(alpha * g') * (u' + beta), with alpha, beta and limit
  given by the caller (gpt-oss: 1.702, 1, 7).  Gate and up are the same W13
  row halves as for "silu".  SiTU is not built: neither the pages nor a
  standard source fixes its formula;
* the intermediate h is rounded to bf16 once, after the activation and
  before FC2 -- the one place the GPU rounds it;
* the router weight multiplies each route's FC2 output in the combine (the
  "top-k sum" of the FC2 store epilogue), accumulated in ascending j, then
  rounded to bf16 once;
* a token with no valid route produces +0.

The matrix products are float64 ``numpy.matmul`` calls; nothing is blocked,
fused or reordered beyond grouping the routes of one expert into one product,
which computes the same independent dot products.
"""

from __future__ import annotations

import numpy as np

from .formats import bf16_rn
from .quant import GROUP, MXFP4, NVFP4, dequant
from .routing import local_experts

SILU = "silu"
RELU2 = "relu2"
SWIGLU_OAI = "swiglu_oai"
GATED = (SILU, SWIGLU_OAI)  # activations whose W13 holds gate and up rows


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_oai(gate, up, alpha, beta, limit):
    """The clamped swiglu (the reading stated in the module docstring).

    The gate is bounded above only, the up projection on both sides; a limit
    of +inf leaves both as they are.
    """
    g = np.minimum(np.asarray(gate, dtype=np.float64), limit)
    u = np.clip(np.asarray(up, dtype=np.float64), -limit, limit)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-alpha * g)) * (u + beta)


def activation_fn(a, act, inter, swiglu=None):
    """Apply the FC1 epilogue activation to fp64 FC1 outputs a [..., N1].

    ``swiglu`` = (alpha, beta, limit), required for "swiglu_oai".
    """
    if act in GATED and a.shape[-1] != 2 * inter:
        raise ValueError("a gated activation expects N1 = 2 * inter")
    if act == SILU:
        return silu(a[..., :inter]) * a[..., inter:]
    if act == SWIGLU_OAI:
        if swiglu is None:
            raise ValueError("swiglu_oai needs (alpha, beta, limit)")
        alpha, beta, limit = swiglu
        return swiglu_oai(a[..., :inter], a[..., inter:], alpha, beta, limit)
    if act == RELU2:
        if a.shape[-1] != inter:
            raise ValueError("ReLU^2 expects N1 = inter")
        return np.maximum(a, 0.0) ** 2
    raise ValueError(f"unknown activation {act!r}")


def _check_inputs(x, w13, s13, gs13, w2, s2, gs2, fmt, act):
    m, hidden = x.shape
    e_l, n1, half_h = w13.shape
    if half_h * 2 != hidden:
        raise ValueError("w13 K dimension does not match hidden")
    inter = n1 // 2 if act in GATED else n1
    if w2.shape != (e_l, hidden, inter // 2):
        raise ValueError(f"w2 shape {w2.shape} != {(e_l, hidden, inter // 2)}")
    g = GROUP[fmt]
    if s13.shape != (e_l, n1, hidden // g) or s2.shape != (e_l, hidden, inter // g):
        raise ValueError("scale shapes do not match the weights")
    if fmt == NVFP4 and (gs13 is None or gs2 is None):
        raise ValueError("NVFP4 needs fp32 global scales")
    if fmt == MXFP4 and (gs13 is not None or gs2 is not None):
        raise ValueError("MXFP4 has no global scales")
    return m, hidden, inter, e_l


def expert_route_outputs(x, w13, s13, gs13, w2, s2, gs2, fmt, act, expert, rows, swiglu=None):
    """FC1 -> activation -> bf16 -> FC2 for the routes of one local expert.

    x rows ``rows`` (token indices) -> y [len(rows), H] in float64, including
    gs2 but not the router weight.  Also returns h, the bf16-rounded
    intermediate, for tests that pin it.
    """
    hidden = x.shape[1]
    inter = w2.shape[2] * 2
    g13 = None if gs13 is None else float(gs13[expert])
    g2 = None if gs2 is None else float(gs2[expert])
    wq13 = dequant(w13[expert], s13[expert], fmt)  # [N1, H], no global scale
    wq2 = dequant(w2[expert], s2[expert], fmt)  # [H, I]
    xa = x[rows]  # [r, H]
    a = xa @ wq13.T
    if g13 is not None:
        a = a * g13
    h = bf16_rn(activation_fn(a, act, inter, swiglu))
    y = h @ wq2.T
    if g2 is not None:
        y = y * g2
    assert y.shape == (len(rows), hidden)
    return y, h


def fused_moe(
    x,
    w13,
    s13,
    gs13,
    w2,
    s2,
    gs2,
    topk_ids,
    topk_weights,
    act,
    fmt,
    num_global_experts,
    expert_map=None,
    tokens=None,
    return_prerounded=False,
    swiglu=None,
):
    """Reference output of the fused W4A16 MoE layer.

    x : [m, H] float64 holding bf16 values.  w13/s13/gs13 and w2/s2/gs2 are the
    packed codes, block scales and (NVFP4) fp32 global scales of the local
    experts.  topk_ids [m, k] int, topk_weights [m, k] float32.
    ``tokens`` optionally restricts the computation to a subset of rows (the
    output then has one row per listed token, in the given order).

    ``swiglu`` = (alpha, beta, limit) of the "swiglu_oai" activation.

    Returns out [len(tokens), H] float64 holding bf16 values; with
    ``return_prerounded`` also the float64 combine before its bf16 rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    m, hidden, inter, e_l = _check_inputs(x, w13, s13, gs13, w2, s2, gs2, fmt, act)
    ids = np.asarray(topk_ids, dtype=np.int64)
    wts = np.asarray(topk_weights, dtype=np.float64)
    k = ids.shape[1]
    loc = local_experts(ids, num_global_experts, e_l, expert_map)
    toks = np.arange(m) if tokens is None else np.asarray(tokens, dtype=np.int64)

    # group the selected routes by expert, compute each route's FC2 output
    y_of_route = {}
    for e in sorted({int(loc[t, j]) for t in toks for j in range(k) if loc[t, j] >= 0}):
        routes = [(int(t), j) for t in toks for j in range(k) if loc[t, j] == e]
        rows = np.array([t for t, _ in routes], dtype=np.int64)
        y, _ = expert_route_outputs(x, w13, s13, gs13, w2, s2, gs2, fmt, act, e, rows, swiglu)
        for (t, j), yr in zip(routes, y):
            y_of_route[(t, j)] = yr

    pre = np.zeros((len(toks), hidden), dtype=np.float64)
    for i, t in enumerate(toks):
        for j in range(k):  # ascending j
            if loc[t, j] >= 0:
                pre[i] += wts[t, j] * y_of_route[(int(t), j)]
    out = bf16_rn(pre)
    if return_prerounded:
        return out, pre
    return out
