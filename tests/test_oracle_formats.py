"""Pins for oracle.formats: every decoder and encoder against an independent source.

Sources: the published E2M1 table (tests/golden), torch's float8 casts (a
library routine), the E2M1 bit-field definition, and exact rational arithmetic
(``fractions.Fraction``) for rounding.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_e2m1_table():
    rows = []
    with open(os.path.join(GOLDEN, "e2m1_ocp_mx_v1.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            c, v = line.split()
            rows.append((int(c), float(v)))
    return rows


def test_e2m1_decode_matches_published_table():
    rows = _load_e2m1_table()
    assert [c for c, _ in rows] == list(range(16))
    got = F.e2m1_decode(np.arange(16))
    for (c, v), g in zip(rows, got):
        assert g == v and math.copysign(1, g) == math.copysign(1, v), c


def test_e2m1_decode_matches_bit_fields():
    # 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; exponent 0 subnormal
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        ref = -mag if s else mag
        assert F.e2m1_decode([c])[0] == ref


def test_e4m3_decode_all_codes_match_torch():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))
    assert np.isnan(got[[0x7F, 0xFF]]).all() and F.e4m3_decode([0x7E])[0] == 448.0


def test_e8m0_decode_all_codes():
    got = F.e8m0_decode(np.arange(256))
    for b in range(255):
        assert got[b] == math.ldexp(1.0, b - 127)
    assert np.isnan(got[255])
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert np.array_equal(got[:255], ref[:255]) and np.isnan(ref[255])


def _nearest_even(value: Fraction, grid, even):
    """Exact nearest grid point, ties to the 'even' candidate."""
    best = min(abs(value - g) for g in grid)
    cands = [i for i, g in enumerate(grid) if abs(value - g) == best]
    evens = [i for i in cands if even[i]]
    return (evens or cands)[0]


def test_e2m1_rounding_ties_and_saturation():
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, want in ties.items():
        assert F.e2m1_decode(F.e2m1_rn_sat([v]))[0] == want
        assert F.e2m1_decode(F.e2m1_rn_sat([-v]))[0] == -want
    assert F.e2m1_decode(F.e2m1_rn_sat([7.0, 1e30, -9.0])).tolist() == [6.0, 6.0, -6.0]
    assert F.e2m1_rn_sat([-0.1])[0] == 8  # sign kept on a value rounding to zero


def test_e2m1_rounding_brute_force():
    grid = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    even = [i % 2 == 0 for i in range(8)]
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(0, 7, 2000), np.arange(0, 6.5, 0.125)])
    got = F.e2m1_rn_sat(vals)
    for v, c in zip(vals, got):
        want = 7 if v >= 6 else _nearest_even(Fraction(float(v)), grid, even)
        assert c == want, v


def test_e4m3_rounding_matches_torch_in_range():
    rng = np.random.default_rng(2)
    vals = np.concatenate([
        rng.uniform(0, 448, 4000),
        np.exp(rng.uniform(np.log(1e-4), np.log(448), 4000)),
        F.e4m3_decode(np.arange(0x7F)),  # exact grid points
    ])
    ref = torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # compare only where the float32 copy is exact (no double rounding in the reference)
    exact = vals.astype(np.float32).astype(np.float64) == vals
    got = F.e4m3_rn_satfinite(vals)
    assert np.array_equal(got[exact], ref[exact])


def test_e4m3_rounding_ties_and_saturation():
    grid = [Fraction(float(v)) for v in F.e4m3_decode(np.arange(0x7F))]
    even = [c % 2 == 0 for c in range(0x7F)]
    mids = [(grid[i] + grid[i + 1]) / 2 for i in range(len(grid) - 1)]
    got = F.e4m3_rn_satfinite(np.array([float(x) for x in mids]))
    for x, c in zip(mids, got):
        assert c == _nearest_even(x, grid, even)
    assert F.e4m3_rn_satfinite([448.0, 460.0, 1e9]).tolist() == [0x7E, 0x7E, 0x7E]


def _bf16_exact(v: float) -> float:
    """Reference bf16 rounding by exact rational arithmetic."""
    if v == 0:
        return v
    fv = Fraction(v)
    a = abs(fv)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (max(e, -126) - 7)
    n = a / q
    lo = math.floor(n)
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    r = lo * q
    if r > Fraction((2 - 2 ** -7)) * Fraction(2) ** 127:
        return math.copysign(math.inf, v)
    return math.copysign(float(r), v)


def test_bf16_rn_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        rng.standard_normal(5000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-38).astype(np.float32),  # subnormal range
        np.array([3.3895e38, -3.39e38, 1e-45, 0.0], dtype=np.float32),
    ]).astype(np.float64)
    ref = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    got = F.bf16_rn(vals)
    assert np.array_equal(got, ref)


def test_bf16_rn_is_a_single_rounding():
    # b + half an ulp + a tiny bit: direct rounding goes up; rounding through
    # float32 first would drop the tiny bit, land on the tie and go to even.
    b = 1.0  # bf16 ulp at 1.0 is 2^-7
    v = b + 2.0 ** -8 + 2.0 ** -40
    assert F.bf16_rn([v])[0] == b + 2.0 ** -7
    through_f32 = float(torch.tensor(v, dtype=torch.float32).to(torch.bfloat16))
    assert through_f32 == b  # shows the test value really distinguishes the two
    rng = np.random.default_rng(4)
    for v in rng.standard_normal(300) * np.exp(rng.uniform(-80, 80, 300)):
        assert F.bf16_rn([v])[0] == _bf16_exact(float(v))


def test_bf16_bits_roundtrip():
    vals = F.bf16_rn(np.random.default_rng(5).standard_normal(1000))
    assert np.array_equal(F.bf16_from_bits(F.bf16_bits(vals)), vals)
    with pytest.raises(ValueError):
        F.bf16_bits([1.0 + 2.0 ** -12])
