"""Pins for oracle.linear: closed forms, brute force on tiny inputs with an
independent decoder (torch's own E4M3 cast), and linearity."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import linear as L
from oracle import quant as Q

E4M3_ONE = 0x38   # 1.0
E2M1_ONE = 0x2    # +1.0
E2M1_SIX = 0x7    # +6.0
E2M1_MSIX = 0xF   # -6.0


def test_closed_form_ones():
    """Codes +1, block scales 1, gs = 0.5, x = 1: every output is K / 2."""
    n, k, m = 5, 96, 3
    codes = np.full((n, k // 2), E2M1_ONE | (E2M1_ONE << 4), np.uint8)
    scales = np.full((n, k // 16), E4M3_ONE, np.uint8)
    out = L.linear(np.ones((m, k)), codes, scales, 0.5, Q.NVFP4)
    assert out.shape == (m, n)
    assert np.all(out == k / 2)


def test_closed_form_rectangular_rows():
    """Row n holds +6 at even k and -6 at odd k, times 2^(n - 127) (MXFP4);
    x[t][k] = (-1)^k (t + 1): out[t][n] = 6 K (t + 1) 2^(n - 127).  A
    transposed operand or a dropped scale changes the shape or the values."""
    n, k, m = 3, 64, 2
    byte = E2M1_SIX | (E2M1_MSIX << 4)  # element 2j = +6, element 2j+1 = -6
    codes = np.full((n, k // 2), byte, np.uint8)
    scales = np.array([[127 + r] * (k // 32) for r in range(n)], np.uint8)
    sign = np.array([(-1.0) ** j for j in range(k)])
    x = np.stack([sign * (t + 1) for t in range(m)])
    out = L.linear(x, codes, scales, None, Q.MXFP4)
    want = np.array([[6.0 * k * (t + 1) * 2.0 ** r for r in range(n)] for t in range(m)])
    assert np.array_equal(out, want)


def _torch_dequant(codes, scales, fmt, gs):
    """Independent decoder: E2M1 by its value table, E4M3 by torch's
    float8_e4m3fn cast, E8M0 by ldexp, then a python triple loop."""
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    n, half = codes.shape
    k = 2 * half
    g = 16 if fmt == Q.NVFP4 else 32
    if fmt == Q.NVFP4:
        sv = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    else:
        sv = np.ldexp(1.0, scales.astype(np.int64) - 127)
    w = np.zeros((n, k))
    for r in range(n):
        for c in range(k):
            byte = int(codes[r, c // 2])
            code = byte & 15 if c % 2 == 0 else byte >> 4
            w[r, c] = table[code] * sv[r, c // g]
    return w * (1.0 if gs is None else float(gs))


@pytest.mark.parametrize("fmt", [Q.NVFP4, Q.MXFP4])
def test_brute_force_tiny(fmt):
    rng = np.random.default_rng(5)
    m, n, k = 3, 7, 64
    w = rng.standard_normal((1, n, k)) * 0.05
    codes, scales, gs = Q.quantize(w, fmt)
    x = F.bf16_rn(rng.standard_normal((m, k)))
    out, pre = L.linear(x, codes, scales, gs, fmt, return_prerounded=True)
    wd = _torch_dequant(codes[0], scales[0], fmt, None if gs is None else gs[0])
    want = np.zeros((m, n))
    for t in range(m):
        for r in range(n):
            acc = 0.0
            for c in range(k):
                acc += x[t, c] * wd[r, c]
            want[t, r] = acc
    assert np.allclose(pre, want, rtol=1e-12, atol=1e-15)
    assert np.array_equal(out, F.bf16_rn(want))


def test_linearity_and_scaling():
    rng = np.random.default_rng(6)
    m, n, k = 4, 9, 128
    codes, scales, gs = Q.quantize(rng.standard_normal((1, n, k)) * 0.02, Q.NVFP4)
    x1 = F.bf16_rn(rng.standard_normal((m, k)))
    x2 = F.bf16_rn(rng.standard_normal((m, k)))
    _, p1 = L.linear(x1, codes, scales, gs, Q.NVFP4, return_prerounded=True)
    _, p2 = L.linear(x2, codes, scales, gs, Q.NVFP4, return_prerounded=True)
    _, p12 = L.linear(x1 + x2, codes, scales, gs, Q.NVFP4, return_prerounded=True)
    _, p4 = L.linear(4.0 * x1, codes, scales, gs, Q.NVFP4, return_prerounded=True)
    assert np.allclose(p12, p1 + p2, rtol=1e-12, atol=1e-15)
    assert np.array_equal(p4, 4.0 * p1)  # a power of two scales every product exactly
    # the global scale multiplies the whole product
    _, pg = L.linear(x1, codes, scales, gs * 2.0, Q.NVFP4, return_prerounded=True)
    assert np.allclose(pg, 2.0 * p1, rtol=1e-12, atol=0)


def test_rejects_bad_inputs():
    codes = np.zeros((4, 16), np.uint8)
    scales = np.full((4, 2), E4M3_ONE, np.uint8)
    with pytest.raises(ValueError):
        L.linear(np.ones((2, 32)), codes, scales, None, Q.NVFP4)  # NVFP4 without gs
    with pytest.raises(ValueError):
        L.linear(np.ones((2, 30)), codes, scales, 1.0, Q.NVFP4)  # K mismatch
    with pytest.raises(ValueError):
        L.linear(np.ones((2, 32)), codes, np.ones((4, 1), np.uint8), 1.0, Q.MXFP4)  # MXFP4 with gs
