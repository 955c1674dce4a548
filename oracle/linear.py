"""The dense W4A16 linear layer, restated in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix: b12x PR #136, "fix(gemm): restore capture-safe K6 small-M
dispatch" (Summary), is a dense W4A16 GEMM -- one low-bit weight matrix times
16-bit activations -- with a small-M dispatch and caller-owned output
buffers.  Here the weight matrix is stored in the FP4 formats of the MoE
layer (flashinfer PR #4255, Description): NVFP4 (E2M1 codes, an E4M3 scale
per 16 elements along K, an fp32 global scale) or MXFP4 (E2M1 codes, an E8M0
scale per 32 elements along K).

Readings taken where the pages are silent:

* out = x . W^T, W[n, k] the dequantised weight of output n and input k,
  i.e. the FC1 product of a one-expert, top-1 MoE layer with no activation;
* the NVFP4 global scale multiplies the accumulator, as for FC1;
* the product is exact (float64 here) and rounded to bf16 once.

The matrix product is one float64 ``numpy.matmul``; nothing is blocked or
reordered.
"""

from __future__ import annotations

import numpy as np

from .formats import bf16_rn
from .quant import GROUP, MXFP4, NVFP4, dequant


def linear(x, codes, scales, gs, fmt, return_prerounded=False):
    """Reference output of the dense W4A16 linear layer.

    x : [m, K] float64 holding bf16 values.  codes [N, K/2] uint8 (two E2M1
    codes per byte, element 2j in the low nibble), scales [N, K/g] uint8,
    gs a float (NVFP4) or None (MXFP4).  A leading axis of one expert on
    codes / scales / gs is accepted.

    Returns out [m, N] float64 holding bf16 values; with ``return_prerounded``
    also the float64 product before its rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    codes = np.asarray(codes)
    scales = np.asarray(scales)
    if codes.ndim == 3:
        if codes.shape[0] != 1 or scales.shape[0] != 1:
            raise ValueError("the linear layer has one weight matrix")
        codes, scales = codes[0], scales[0]
        if gs is not None:
            gs = np.asarray(gs).reshape(-1)[0]
    n, half_k = codes.shape
    if x.ndim != 2 or x.shape[1] != 2 * half_k:
        raise ValueError(f"x shape {x.shape} does not match K = {2 * half_k}")
    if scales.shape != (n, 2 * half_k // GROUP[fmt]):
        raise ValueError("scale shape does not match the codes")
    if fmt == NVFP4 and gs is None:
        raise ValueError("NVFP4 needs the fp32 global scale")
    if fmt == MXFP4 and gs is not None:
        raise ValueError("MXFP4 has no global scale")
    w = dequant(codes, scales, fmt)  # [N, K]
    pre = x @ w.T
    if gs is not None:
        pre = pre * float(gs)
    out = bf16_rn(pre)
    if return_prerounded:
        return out, pre
    return out
