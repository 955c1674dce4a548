"""NVFP4 and MXFP4 weight quantisation and dequantisation, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix (flashinfer PR #4255, Description and review comments):

* NVFP4 weights: E2M1 codes with one FP8-E4M3 block scale per 16 elements
  along K (scale format ``e4m3_k16``) and, for the ModelOpt layout, one fp32
  global scale per expert.
* MXFP4 weights, source format ``fp4_e8m0_k32``: E2M1 codes with one E8M0
  power-of-two scale per 32 elements along K, "including scale-tail handling
  for TP shards that are not 128-aligned".

Readings taken where the pages are silent:

* packing: element 2j of a row sits in the low nibble of byte j, element
  2j+1 in the high nibble (the ModelOpt convention);
* the global scale multiplies the dequantised value, one fp32 per expert per
  tensor;
* NVFP4 quantiser: gs = amax|W_e| / (6 * 448) (1 when amax is 0);
  s_b = e4m3_rn_satfinite(amax_b / (6 * gs)); code = e2m1_rn_sat(w / (e4m3(s_b) * gs)),
  or +0 when s_b decodes to 0 (safe handling of zero-valued scales, named in
  the CodeRabbit summary of PR #4255);
* MXFP4 quantiser: e = clamp(127 + ceil(log2(amax_b / 6)), 0, 254), e = 0 when
  amax_b = 0 (a power-of-two ceiling, the only E8M0 rounding the pages name:
  ``pow2_ceil_ue8m0_torch`` in a review comment of PR #4255);
  code = e2m1_rn_sat(w / 2^(e-127)).

The quantisers only build test inputs: the layer itself consumes codes and
scales and never quantises.
"""

from __future__ import annotations

import numpy as np

from .formats import (
    E2M1_MAX,
    E4M3_MAX,
    e2m1_decode,
    e2m1_rn_sat,
    e4m3_decode,
    e4m3_rn_satfinite,
    e8m0_decode,
)

NVFP4 = "nvfp4_e4m3_k16"
MXFP4 = "mxfp4_e8m0_k32"
GROUP = {NVFP4: 16, MXFP4: 32}


# ---------------------------------------------------------------------------
# nibble packing
# ---------------------------------------------------------------------------


def pack_nibbles(codes) -> np.ndarray:
    """[..., K] codes 0..15 -> [..., K/2] bytes, element 2j in the low nibble."""
    c = np.asarray(codes).astype(np.uint8)
    if c.shape[-1] % 2:
        raise ValueError("K must be even to pack two codes per byte")
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] codes, inverse of ``pack_nibbles``."""
    p = np.asarray(packed).astype(np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# ---------------------------------------------------------------------------
# dequantisation (the definition the layer computes, step a2 / a3)
# ---------------------------------------------------------------------------


def dequant(codes_packed, scales, fmt, gs=None) -> np.ndarray:
    """Dequantise one expert's weight matrix to float64.

    codes_packed : [N, K/2] uint8, scales : [N, K/g] uint8.
    NVFP4: W[n, k] = e2m1(c[n, k]) * e4m3(s[n, k // 16]) * gs (gs omitted when None).
    MXFP4: W[n, k] = e2m1(c[n, k]) * 2^(s[n, k // 32] - 127); gs must be None.
    """
    g = GROUP[fmt]
    c = e2m1_decode(unpack_nibbles(codes_packed))
    n, k = c.shape
    if k % g:
        raise ValueError(f"K={k} is not a multiple of the scale group {g}")
    s = np.asarray(scales)
    if s.shape != (n, k // g):
        raise ValueError(f"scales shape {s.shape} != {(n, k // g)}")
    if fmt == NVFP4:
        sv = e4m3_decode(s)
    else:
        if gs is not None:
            raise ValueError("MXFP4 has no global scale")
        sv = e8m0_decode(s)
    w = c * np.repeat(sv, g, axis=1)
    if gs is not None:
        w = w * float(gs)
    return w


# ---------------------------------------------------------------------------
# quantisers (test-input builders)
# ---------------------------------------------------------------------------


def quantize_nvfp4(w):
    """Quantise [E, N, K] weights to NVFP4.

    Returns (codes [E, N, K/2] uint8, scales [E, N, K/16] uint8, gs [E] float32).
    The global scale is rounded to float32 first, because that is the type the
    layer receives; the block scales and codes are then chosen against that
    float32 value, in float64 arithmetic.
    """
    w = np.asarray(w, dtype=np.float64)
    e, n, k = w.shape
    if k % 16:
        raise ValueError("K must be a multiple of 16 for NVFP4")
    amax_e = np.abs(w).reshape(e, -1).max(axis=1)
    gs = np.where(amax_e > 0, amax_e / (E2M1_MAX * E4M3_MAX), 1.0).astype(np.float32)
    gs64 = gs.astype(np.float64)
    blocks = w.reshape(e, n, k // 16, 16)
    amax_b = np.abs(blocks).max(axis=-1)
    s = e4m3_rn_satfinite(amax_b / (E2M1_MAX * gs64[:, None, None]))
    sv = e4m3_decode(s)
    denom = sv * gs64[:, None, None]
    safe = np.where(denom > 0, denom, 1.0)
    q = e2m1_rn_sat(blocks / safe[..., None])
    q = np.where((denom > 0)[..., None], q, 0).astype(np.uint8)
    return pack_nibbles(q.reshape(e, n, k)), s.astype(np.uint8), gs


def quantize_mxfp4(w):
    """Quantise [E, N, K] weights to MXFP4 (fp4_e8m0_k32).

    Returns (codes [E, N, K/2] uint8, scales [E, N, K/32] uint8 E8M0).
    """
    w = np.asarray(w, dtype=np.float64)
    e, n, k = w.shape
    if k % 32:
        raise ValueError("K must be a multiple of 32 for MXFP4")
    blocks = w.reshape(e, n, k // 32, 32)
    amax_b = np.abs(blocks).max(axis=-1)
    with np.errstate(divide="ignore"):
        ex = 127 + np.ceil(np.log2(np.where(amax_b > 0, amax_b / E2M1_MAX, 1.0)))
    ex = np.where(amax_b > 0, np.clip(ex, 0, 254), 0).astype(np.int64)
    scale = np.ldexp(1.0, ex - 127)
    q = e2m1_rn_sat(blocks / scale[..., None])
    return pack_nibbles(q.reshape(e, n, k)), ex.astype(np.uint8)


def quantize(w, fmt):
    """Dispatch to the quantiser of ``fmt``; returns (codes, scales, gs-or-None)."""
    if fmt == NVFP4:
        return quantize_nvfp4(w)
    if fmt == MXFP4:
        c, s = quantize_mxfp4(w)
        return c, s, None
    raise ValueError(f"unknown format {fmt!r}")
