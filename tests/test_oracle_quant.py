"""Pins for oracle.quant: packing, dequantisation and the two quantisers."""

import numpy as np
import pytest

from oracle import formats as F
from oracle import quant as Q

E4M3_ONE = 0x38  # exponent 7, mantissa 0 -> 1.0
E8M0_ONE = 127


def test_nibble_order_low_nibble_is_even_element():
    # byte 0x21: low nibble 1 (0.5) is element 0, high nibble 2 (1.0) element 1
    codes = Q.unpack_nibbles(np.array([[0x21, 0xF8]], dtype=np.uint8))
    assert codes.tolist() == [[1, 2, 8, 15]]
    assert F.e2m1_decode(codes).tolist() == [[0.5, 1.0, -0.0, -6.0]]
    rng = np.random.default_rng(0)
    c = rng.integers(0, 16, size=(5, 64), dtype=np.uint8)
    assert np.array_equal(Q.unpack_nibbles(Q.pack_nibbles(c)), c)


def test_dequant_with_unit_scales_is_the_e2m1_table():
    rng = np.random.default_rng(1)
    c = rng.integers(0, 16, size=(4, 64), dtype=np.uint8)
    nv = Q.dequant(Q.pack_nibbles(c), np.full((4, 4), E4M3_ONE, np.uint8), Q.NVFP4, gs=1.0)
    mx = Q.dequant(Q.pack_nibbles(c), np.full((4, 2), E8M0_ONE, np.uint8), Q.MXFP4)
    assert np.array_equal(nv, F.e2m1_decode(c)) and np.array_equal(mx, F.e2m1_decode(c))


@pytest.mark.parametrize("fmt,g,one,step", [(Q.NVFP4, 16, E4M3_ONE, 8), (Q.MXFP4, 32, E8M0_ONE, 1)])
def test_dequant_scale_block_locality_and_scaling(fmt, g, one, step):
    rng = np.random.default_rng(2)
    n, k = 3, 4 * g
    c = Q.pack_nibbles(rng.integers(0, 16, size=(n, k), dtype=np.uint8))
    s = np.full((n, k // g), one, np.uint8)
    gs = 1.0 if fmt == Q.NVFP4 else None
    base = Q.dequant(c, s, fmt, gs)
    s2 = s.copy()
    s2[1, 2] = one + step  # doubles block (row 1, k in [2g, 3g))
    out = Q.dequant(c, s2, fmt, gs)
    changed = out != base
    want = np.zeros_like(changed)
    want[1, 2 * g : 3 * g] = base[1, 2 * g : 3 * g] != 0
    assert np.array_equal(changed, want)
    assert np.array_equal(out[1, 2 * g : 3 * g], 2 * base[1, 2 * g : 3 * g])
    if fmt == Q.NVFP4:
        assert np.array_equal(Q.dequant(c, s, fmt, gs=0.25), base * 0.25)


def test_dequant_requeantise_roundtrip_keeps_codes_and_signed_zero():
    # dequant -> divide by the same scale -> E2M1 encode returns the same codes
    rng = np.random.default_rng(3)
    c = rng.integers(0, 16, size=(6, 64), dtype=np.uint8)
    s = rng.integers(0x20, 0x7E, size=(6, 4)).astype(np.uint8)
    w = Q.dequant(Q.pack_nibbles(c), s, Q.NVFP4, gs=0.5)
    back = F.e2m1_rn_sat(w / (np.repeat(F.e4m3_decode(s), 16, axis=1) * 0.5))
    assert np.array_equal(back, c)


def _half_step_bound(u):
    """Half the E2M1 grid spacing at magnitude u (u already divided by the scale)."""
    u = np.abs(u)
    return np.select([u <= 2, u <= 4], [0.25, 0.5], 1.0)


def test_nvfp4_quantiser_error_bound_and_structure():
    rng = np.random.default_rng(4)
    w = rng.standard_normal((3, 32, 128)) * 0.02
    w[2, 5, 16:32] = 0.0  # an all-zero block
    c, s, gs = Q.quantize_nvfp4(w)
    assert gs.dtype == np.float32 and c.shape == (3, 32, 64) and s.shape == (3, 32, 8)
    # the expert's largest block gets exactly the largest finite scale 448
    for e in range(3):
        assert F.e4m3_decode(s[e]).max() == 448.0
    sv = np.repeat(F.e4m3_decode(s), 16, axis=2) * gs.astype(np.float64)[:, None, None]
    deq = np.stack([Q.dequant(c[e], s[e], Q.NVFP4, gs[e]) for e in range(3)])
    u = w / np.where(sv > 0, sv, 1)
    bound = np.maximum(_half_step_bound(u), np.abs(u) - 6.0) * sv
    assert np.all(np.abs(w - deq) <= bound * (1 + 1e-12))
    # every block with a normal-range scale encodes its largest element as +-6
    codes = Q.unpack_nibbles(c).reshape(3, 32, 8, 16)
    mags = (codes & 7).max(axis=-1)
    normal = F.e4m3_decode(s) >= 2.0 ** -6
    assert np.all(mags[normal] == 7)
    assert s[2, 5, 1] == 0 and np.all(codes[2, 5, 1] == 0)


def test_mxfp4_quantiser_error_bound_and_structure():
    rng = np.random.default_rng(5)
    w = rng.standard_normal((2, 16, 96)) * 0.02  # K = 96: three blocks, not 128-aligned
    w[1, 3, 32:64] = 0.0
    c, s = Q.quantize_mxfp4(w)
    assert c.shape == (2, 16, 48) and s.shape == (2, 16, 3)
    deq = np.stack([Q.dequant(c[e], s[e], Q.MXFP4) for e in range(2)])
    sv = np.repeat(F.e8m0_decode(s), 32, axis=2)
    u = w / sv
    assert np.all(np.abs(u) <= 6.0)  # the power-of-two ceiling never saturates
    assert np.all(np.abs(w - deq) <= _half_step_bound(u) * sv * (1 + 1e-12))
    amax = np.abs(w.reshape(2, 16, 3, 32)).max(axis=-1)
    nz = amax > 0
    assert np.all(amax[nz] / F.e8m0_decode(s)[nz] > 3.0)  # tight: the scale is the ceiling
    assert s[1, 3, 1] == 0


def test_quantiser_rejects_bad_k():
    with pytest.raises(ValueError):
        Q.quantize_nvfp4(np.zeros((1, 2, 24)))
    with pytest.raises(ValueError):
        Q.quantize_mxfp4(np.zeros((1, 2, 48)))
