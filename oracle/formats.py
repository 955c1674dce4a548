"""Number formats of the W4A16 layer, decoded and encoded in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The formats are named, not defined, on the pages:

* flashinfer PR #4255, Description: "NVFP4 weights, bf16 activations" and the
  new "fp4_e8m0_k32 (MXFP4 K/32) weight source format";
* flashinfer PR #4255, review comments: the scale formats ``e4m3_k16`` and
  ``e8m0_k32``.

NVFP4 and MXFP4 share the 4-bit element E2M1.  Their block scales are FP8
E4M3 (the "fn" variant: no infinities, one NaN pattern per sign) and E8M0 (a
bare biased exponent).  The definitions below are the public ones (OCP
Microscaling Formats v1.0, section 5.3 for E2M1 and E8M0; the OCP 8-bit
floating point specification for E4M3) written out from their bit fields.
The pages print none of these tables; the pins in ``tests/test_oracle_formats.py``
check each decoder against an independent definition or library cast.
"""

from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
# Exponent field 0 is subnormal: value = mantissa * 0.5.
# Magnitudes of codes 0..7 are therefore 0, 0.5, 1, 1.5, 2, 3, 4, 6; codes
# 8..15 are their negatives (code 8 is -0.0).
# ---------------------------------------------------------------------------
_E2M1_MAGNITUDE = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
E2M1_VALUES = np.array(
    list(_E2M1_MAGNITUDE) + [-v for v in _E2M1_MAGNITUDE], dtype=np.float64
)
E2M1_MAX = 6.0


def e2m1_decode(codes) -> np.ndarray:
    """Decode 4-bit E2M1 codes (values 0..15, any integer array) to float64."""
    c = np.asarray(codes).astype(np.int64)
    if np.any((c < 0) | (c > 15)):
        raise ValueError("E2M1 codes must lie in [0, 15]")
    return E2M1_VALUES[c]


def e2m1_rn_sat(v) -> np.ndarray:
    """Round float64 values to the nearest E2M1 code, ties to even, saturating.

    Reading taken (the pages are silent on E2M1 rounding): round to nearest,
    ties to the code whose mantissa bit is 0, magnitudes above 6 saturate to
    6.  The sign bit of the input is kept, so a negative value that rounds to
    zero gives code 8 (-0.0).  NaN inputs are rejected.
    """
    v = np.asarray(v, dtype=np.float64)
    if np.any(np.isnan(v)):
        raise ValueError("cannot encode NaN as E2M1")
    a = np.abs(v)
    grid = np.array(_E2M1_MAGNITUDE)
    # distance to every grid point; pick the nearest, then break ties to the
    # even code (codes 0, 2, 4, 6 have mantissa bit 0).
    d = np.abs(a[..., None] - grid)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    even = (np.arange(8) % 2) == 0
    pick_even = cand & even
    has_even = pick_even.any(axis=-1, keepdims=True)
    chosen = np.where(has_even, pick_even, cand)
    mag_code = np.argmax(chosen, axis=-1)
    mag_code = np.where(a >= E2M1_MAX, 7, mag_code)
    sign = np.signbit(v).astype(np.int64)
    return (mag_code + 8 * sign).astype(np.uint8)


# ---------------------------------------------------------------------------
# E4M3 ("fn"): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits.
# Exponent field 0 is subnormal: value = m * 2^-9.  The pattern S.1111.111 is
# NaN; there are no infinities, so the largest finite magnitude is 448.
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Decode FP8 E4M3 (fn) bytes to float64; 0x7F and 0xFF decode to NaN."""
    b = np.asarray(codes).astype(np.int64)
    if np.any((b < 0) | (b > 255)):
        raise ValueError("E4M3 codes must lie in [0, 255]")
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    sub = m * 2.0 ** -9
    nrm = (1.0 + m / 8.0) * np.ldexp(1.0, e - 7)
    val = sign * np.where(e == 0, sub, nrm)
    return np.where((b & 0x7F) == 0x7F, np.nan, val)


def _e4m3_positive_grid():
    codes = np.arange(0x7F)  # 0x00 .. 0x7E, all finite and non-negative
    return codes, e4m3_decode(codes)


def e4m3_rn_satfinite(v) -> np.ndarray:
    """Round non-negative float64 values to E4M3 (fn), nearest, ties to even.

    Magnitudes at or above 448 saturate to 448 (code 0x7E), the
    "satfinite" behaviour of FP8 conversions.  Block scales are computed from
    magnitudes, so only inputs >= 0 are accepted.
    """
    v = np.asarray(v, dtype=np.float64)
    if np.any(np.isnan(v)) or np.any(v < 0):
        raise ValueError("e4m3_rn_satfinite takes finite values >= 0")
    codes, grid = _e4m3_positive_grid()
    d = np.abs(v[..., None] - grid)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    even = (codes % 2) == 0
    pick_even = cand & even
    has_even = pick_even.any(axis=-1, keepdims=True)
    chosen = np.where(has_even, pick_even, cand)
    out = codes[np.argmax(chosen, axis=-1)]
    out = np.where(v >= E4M3_MAX, 0x7E, out)
    return out.astype(np.uint8)


# ---------------------------------------------------------------------------
# E8M0: an unsigned biased exponent.  value = 2^(b - 127) for b in [0, 254];
# b = 255 is NaN.
# ---------------------------------------------------------------------------


def e8m0_decode(codes) -> np.ndarray:
    """Decode E8M0 bytes to float64 powers of two; 255 decodes to NaN."""
    b = np.asarray(codes).astype(np.int64)
    if np.any((b < 0) | (b > 255)):
        raise ValueError("E8M0 codes must lie in [0, 255]")
    val = np.ldexp(1.0, b - 127)
    return np.where(b == 255, np.nan, val)


# ---------------------------------------------------------------------------
# bf16: 1 sign, 8 exponent bits (bias 127), 7 mantissa bits.
# ---------------------------------------------------------------------------
_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_rn(v) -> np.ndarray:
    """Round float64 values to bf16 once, nearest-even; returns float64 values.

    This is a single rounding from the float64 value.  It does not go through
    float32 first, so it never double-rounds.  Subnormal bf16 values (spacing
    2^-133) are produced exactly; magnitudes that round above the largest
    finite bf16 become infinities, as IEEE round-to-nearest prescribes.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty_like(v)
    finite = np.isfinite(v)
    a = np.abs(np.where(finite, v, 0.0))
    # exponent of the leading bit; subnormals share the quantum 2^-133
    _, e = np.frexp(a)  # a = f * 2^e with f in [0.5, 1)
    exp = np.maximum(e - 1, -126)
    quantum = np.ldexp(1.0, exp - 7)
    q = np.rint(a / quantum) * quantum  # np.rint rounds half to even
    q = np.where(a == 0, 0.0, q)
    overflow = q > _BF16_MAX
    q = np.where(overflow, np.inf, q)
    out[...] = np.where(finite, np.copysign(q, v), v)
    return out


def bf16_bits(v) -> np.ndarray:
    """bf16 bit patterns (uint16) of float64 values already on the bf16 grid."""
    v = np.asarray(v, dtype=np.float64)
    f32 = v.astype(np.float32)
    if not np.array_equal(f32.astype(np.float64), v, equal_nan=True):
        raise ValueError("values are not representable in bf16")
    u32 = f32.view(np.uint32)
    if np.any(u32 & 0xFFFF):
        raise ValueError("values are not representable in bf16")
    return (u32 >> 16).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    """float64 values of bf16 bit patterns."""
    b = np.asarray(bits).astype(np.uint32)
    return (b << 16).astype(np.uint32).view(np.float32).astype(np.float64)
