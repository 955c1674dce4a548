"""Pins for oracle.moe: special cases with independent answers, and invariances."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import moe as M
from oracle import quant as Q
from oracle import routing as R

E4M3_ONE = 0x38


def _rand_layer(rng, e, hidden, inter, act, fmt=Q.NVFP4):
    n1 = 2 * inter if act in M.GATED else inter
    w13 = rng.standard_normal((e, n1, hidden)) * 0.05
    w2 = rng.standard_normal((e, hidden, inter)) * 0.05
    c13, s13, g13 = Q.quantize(w13, fmt)
    c2, s2, g2 = Q.quantize(w2, fmt)
    return c13, s13, g13, c2, s2, g2


def _bf16_x(rng, m, hidden):
    return F.bf16_rn(rng.standard_normal((m, hidden)))


@pytest.mark.parametrize("act", [M.SILU, M.RELU2])
def test_top1_single_expert_is_a_dense_mlp(act):
    """E = 1, top-1, weight 1: the layer reduces to a dense MLP (torch fp64)."""
    rng = np.random.default_rng(0)
    hidden, inter, m = 64, 48, 7
    c13, s13, g13, c2, s2, g2 = _rand_layer(rng, 1, hidden, inter, act)
    x = _bf16_x(rng, m, hidden)
    ids = np.zeros((m, 1), np.int32)
    wts = np.ones((m, 1), np.float32)
    out, pre = M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids, wts, act, Q.NVFP4, 1, return_prerounded=True)

    # independent restatement with torch: table lookup, torch matmul, torch silu
    table = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float64)
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)

    def deq(c, s, g):
        c = torch.from_numpy(c.astype(np.int64))
        codes = torch.stack([c & 15, c >> 4], dim=-1).reshape(c.shape[0], -1)
        sc = e4m3[torch.from_numpy(s.astype(np.int64))].repeat_interleave(16, dim=1)
        return table[codes] * sc * float(g)

    W13, W2 = deq(c13[0], s13[0], g13[0]), deq(c2[0], s2[0], g2[0])
    xt = torch.from_numpy(x)
    a = xt @ W13.T
    h = torch.nn.functional.silu(a[:, :inter]) * a[:, inter:] if act == M.SILU else torch.relu(a) ** 2
    h = torch.from_numpy(F.bf16_rn(h.numpy()))
    y = h @ W2.T
    assert np.allclose(pre, y.numpy(), rtol=1e-12, atol=1e-12)
    assert np.array_equal(out, F.bf16_rn(y.numpy()))


def test_exact_integer_case_relu2():
    """Integer x, unit scales, ReLU^2: every intermediate is an exact small
    integer in bf16, so the output is known exactly from integer arithmetic."""
    rng = np.random.default_rng(1)
    e, k, hidden, inter, m = 3, 2, 16, 16, 5
    # FC1 codes restricted to magnitudes {0, 1} -> codes {0, 2} with signs, and
    # x in {-1, 0, 1}, so |a| <= 16 and h = a^2 <= 256 is an exact bf16 integer
    mag = rng.choice([0, 2], size=(e, inter, hidden))
    sgn = rng.integers(0, 2, size=mag.shape) * 8
    c13 = Q.pack_nibbles((mag | sgn).astype(np.uint8))
    mag2 = rng.choice([0, 2, 4], size=(e, hidden, inter))
    c2 = Q.pack_nibbles((mag2 | rng.integers(0, 2, size=mag2.shape) * 8).astype(np.uint8))
    s13 = np.full((e, inter, hidden // 16), E4M3_ONE, np.uint8)
    s2 = np.full((e, hidden, inter // 16), E4M3_ONE, np.uint8)
    g13 = np.ones(e, np.float32)
    g2 = np.ones(e, np.float32)
    xi = rng.integers(-1, 2, size=(m, hidden))
    ids = rng.integers(0, e, size=(m, k)).astype(np.int32)
    wts = np.full((m, k), 0.5, np.float32)
    out = M.fused_moe(xi.astype(np.float64), c13, s13, g13, c2, s2, g2, ids, wts, M.RELU2, Q.NVFP4, e)

    vals = {0: 0, 2: 1, 4: 2}
    W1 = np.vectorize(vals.get)(mag) * np.where(sgn, -1, 1)
    W2 = np.vectorize(vals.get)(mag2) * np.where(c2_sign := (Q.unpack_nibbles(c2) >> 3), -1, 1)
    want = np.zeros((m, hidden), dtype=object)
    for t in range(m):
        for j in range(k):
            ex = ids[t, j]
            a = [int(sum(int(xi[t, q]) * int(W1[ex, i, q]) for q in range(hidden))) for i in range(inter)]
            h = [max(v, 0) ** 2 for v in a]
            assert all(v <= 256 for v in h), "case must stay exactly representable in bf16"
            for n in range(hidden):
                want[t, n] += sum(h[i] * int(W2[ex, n, i]) for i in range(inter))
    want = np.array([[float(v) / 2 for v in row] for row in want])  # weights 0.5 each
    assert np.array_equal(out, F.bf16_rn(want))
    assert c2_sign is not None


def test_invariances_permutation_linearity_and_dropped_routes():
    rng = np.random.default_rng(2)
    e, k, hidden, inter, m = 5, 3, 32, 32, 6
    c13, s13, g13, c2, s2, g2 = _rand_layer(rng, e, hidden, inter, M.SILU)
    x = _bf16_x(rng, m, hidden)
    ids = rng.integers(0, e, size=(m, k)).astype(np.int32)
    wts = rng.random((m, k)).astype(np.float32)
    base, pre = M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids, wts, M.SILU, Q.NVFP4, e, return_prerounded=True)

    # permuting the local experts together with expert_map leaves the output unchanged
    perm = rng.permutation(e)  # local slot perm[l] holds global expert l
    inv = np.argsort(perm)
    em = perm.astype(np.int32)
    out_p = M.fused_moe(x, c13[inv], s13[inv], g13[inv], c2[inv], s2[inv], g2[inv], ids, wts, M.SILU, Q.NVFP4, e, expert_map=em)
    assert np.array_equal(out_p, base)

    # linear in the router weights before the final rounding (x2 and a sum of
    # two weight sets are exact in float32, so the check is not blurred by it)
    _, pre2 = M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids, (wts * 2).astype(np.float32), M.SILU, Q.NVFP4, e, return_prerounded=True)
    assert np.allclose(pre2, 2 * pre, rtol=1e-13, atol=1e-15)
    wa = np.where(rng.random((m, k)) < 0.5, wts, 0).astype(np.float32)
    _, pa = M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids, wa, M.SILU, Q.NVFP4, e, return_prerounded=True)
    _, pb = M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids, (wts - wa).astype(np.float32), M.SILU, Q.NVFP4, e, return_prerounded=True)
    assert np.allclose(pa + pb, pre, rtol=1e-12, atol=1e-15)

    # a dropped route (invalid id) equals the same route with weight 0
    ids_d = ids.copy()
    ids_d[1, 2] = -1
    ids_d[4, 0] = e  # out of range
    wts_0 = wts.copy()
    wts_0[1, 2] = 0
    wts_0[4, 0] = 0
    a = M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids_d, wts, M.SILU, Q.NVFP4, e)
    b = M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids, wts_0, M.SILU, Q.NVFP4, e)
    assert np.array_equal(a, b)

    # a token subset reproduces the matching rows
    sub = M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids, wts, M.SILU, Q.NVFP4, e, tokens=[4, 0])
    assert np.array_equal(sub, base[[4, 0]])

    # a token whose routes are all invalid gives +0
    ids_z = ids.copy()
    ids_z[2] = -1
    z = M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids_z, wts, M.SILU, Q.NVFP4, e)
    assert np.all(z[2] == 0) and not np.any(np.signbit(z[2]))


def test_mxfp4_tail_layer_matches_dense_restatement():
    """MXFP4 with K = 96 and I = 48 (neither 128-aligned): dense torch check."""
    rng = np.random.default_rng(3)
    e, k, hidden, inter, m = 4, 2, 96, 64, 5
    c13, s13, _, c2, s2, _ = _rand_layer(rng, e, hidden, inter, M.SILU, Q.MXFP4)
    em = np.array([2, -1, 0, 3, 1], np.int32)  # 5 global experts, one dropped
    x = _bf16_x(rng, m, hidden)
    ids = rng.integers(-1, 6, size=(m, k)).astype(np.int32)
    wts = rng.random((m, k)).astype(np.float32)
    out, pre = M.fused_moe(x, c13, s13, None, c2, s2, None, ids, wts, M.SILU, Q.MXFP4, 5, expert_map=em, return_prerounded=True)
    want = np.zeros((m, hidden))
    for t in range(m):
        for j in range(k):
            gid = ids[t, j]
            if not (0 <= gid < 5) or em[gid] < 0:
                continue
            l = em[gid]
            W13 = torch.from_numpy(F.e2m1_decode(Q.unpack_nibbles(c13[l])) * np.ldexp(1.0, np.repeat(s13[l].astype(int) - 127, 32, axis=1)))
            W2 = torch.from_numpy(F.e2m1_decode(Q.unpack_nibbles(c2[l])) * np.ldexp(1.0, np.repeat(s2[l].astype(int) - 127, 32, axis=1)))
            a = torch.from_numpy(x[t]) @ W13.T
            h = F.bf16_rn((torch.nn.functional.silu(a[:inter]) * a[inter:]).numpy())
            want[t] += float(wts[t, j]) * (torch.from_numpy(h) @ W2.T).numpy()
    assert np.allclose(pre, want, rtol=1e-12, atol=1e-14)


def test_route_pack_and_layer_agree_on_validity():
    rng = np.random.default_rng(4)
    ids = rng.integers(-3, 12, size=(9, 4)).astype(np.int32)
    em = rng.integers(-1, 6, size=10).astype(np.int32)
    c, o, s = R.route_pack(ids, 10, 6, em)
    loc = R.local_experts(ids, 10, 6, em)
    assert int(o[-1]) == int((loc >= 0).sum())


# ---------------------------------------------------------------- swiglu-oai
OAI = (1.702, 1.0, 7.0)


def _torch_clamped_swiglu(gate, up, alpha, beta, limit):
    """Independent form: g sigmoid(alpha g) = silu(alpha g) / alpha (torch's
    silu and clamp), so no line of the oracle's formula is retyped."""
    g = torch.clamp(torch.as_tensor(gate, dtype=torch.float64), max=limit)
    u = torch.clamp(torch.as_tensor(up, dtype=torch.float64), min=-limit, max=limit)
    return (torch.nn.functional.silu(alpha * g) / alpha * (u + beta)).numpy()


def test_clamped_swiglu_matches_the_silu_identity():
    rng = np.random.default_rng(11)
    gate = rng.standard_normal(4096) * 6
    up = rng.standard_normal(4096) * 6
    for alpha, beta, limit in (OAI, (1.0, 0.0, np.inf), (0.5, -2.0, 3.0), (2.5, 1.0, 0.25)):
        got = M.swiglu_oai(gate, up, alpha, beta, limit)
        assert np.allclose(got, _torch_clamped_swiglu(gate, up, alpha, beta, limit), rtol=1e-13, atol=1e-300)


def test_clamped_swiglu_without_clamp_is_swiglu():
    """alpha 1, beta 0, no limit: silu(gate) * up, torch's silu."""
    rng = np.random.default_rng(12)
    gate, up = rng.standard_normal(1000) * 8, rng.standard_normal(1000) * 8
    want = (torch.nn.functional.silu(torch.from_numpy(gate)) * torch.from_numpy(up)).numpy()
    assert np.allclose(M.swiglu_oai(gate, up, 1.0, 0.0, np.inf), want, rtol=1e-14, atol=0)


def test_clamped_swiglu_special_values():
    alpha, beta, limit = OAI
    f = lambda g, u: float(M.swiglu_oai(g, u, alpha, beta, limit))
    # zero gate, and an up projection of exactly -beta, give exact zeros
    assert f(0.0, 3.0) == 0.0 and f(2.0, -beta) == 0.0
    # the gate saturates above the limit only
    assert f(limit, 0.5) == f(3 * limit, 0.5) == f(1e30, 0.5)
    assert f(-limit, 0.5) != f(-3 * limit, 0.5)
    assert abs(f(-1e3, 0.5)) < 1e-300
    # the up projection saturates on both sides
    assert f(1.0, limit) == f(1.0, 50.0) and f(1.0, -limit) == f(1.0, -50.0)
    # at the limit: limit * sigmoid(alpha limit) * (limit + beta), sigmoid from math.exp
    import math
    want = limit / (1 + math.exp(-alpha * limit)) * (limit + beta)
    assert math.isclose(f(limit, limit), want, rel_tol=1e-15)
    # NaN stays NaN
    assert np.isnan(M.swiglu_oai(np.nan, 1.0, alpha, beta, limit))


def test_activation_fn_gate_and_up_halves():
    """Rows [0, I) are the gate and [I, 2I) the up projection, as for silu:
    swapping the halves changes the result."""
    rng = np.random.default_rng(13)
    a = rng.standard_normal((3, 2 * 40)) * 5
    got = M.activation_fn(a, M.SWIGLU_OAI, 40, OAI)
    assert np.allclose(got, _torch_clamped_swiglu(a[:, :40], a[:, 40:], *OAI), rtol=1e-13)
    assert not np.allclose(got, _torch_clamped_swiglu(a[:, 40:], a[:, :40], *OAI))
    with pytest.raises(ValueError):
        M.activation_fn(a, M.SWIGLU_OAI, 40)  # parameters are required


@pytest.mark.parametrize("fmt", [Q.NVFP4, Q.MXFP4])
def test_clamped_swiglu_layer_is_a_dense_mlp(fmt):
    """E = 1, top-1, weight 1, with a limit the FC1 outputs cross: the layer
    is a dense clamped-swiglu MLP (torch fp64, dequantised by table)."""
    rng = np.random.default_rng(14)
    hidden, inter, m = 64, 64, 9
    c13, s13, g13, c2, s2, g2 = _rand_layer(rng, 1, hidden, inter, M.SWIGLU_OAI, fmt)
    x = _bf16_x(rng, m, hidden) * 8
    ids = np.zeros((m, 1), np.int32)
    wts = np.ones((m, 1), np.float32)
    params = (1.702, 1.0, 0.5)
    out, pre = M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids, wts, M.SWIGLU_OAI, fmt, 1, return_prerounded=True,
                           swiglu=params)
    table = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float64)
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)

    def deq(c, s, g):
        c = torch.from_numpy(c.astype(np.int64))
        codes = torch.stack([c & 15, c >> 4], dim=-1).reshape(c.shape[0], -1)
        s = torch.from_numpy(s.astype(np.int64))
        if fmt == Q.NVFP4:
            return table[codes] * e4m3[s].repeat_interleave(16, dim=1) * float(g)
        return table[codes] * torch.pow(2.0, (s - 127).to(torch.float64)).repeat_interleave(32, dim=1)

    W13 = deq(c13[0], s13[0], None if g13 is None else g13[0])
    W2 = deq(c2[0], s2[0], None if g2 is None else g2[0])
    a = torch.from_numpy(x) @ W13.T
    assert (a[:, :inter] > params[2]).any() and (a[:, inter:].abs() > params[2]).any()  # the clamps act
    h = torch.from_numpy(F.bf16_rn(_torch_clamped_swiglu(a[:, :inter], a[:, inter:], *params)))
    y = h @ W2.T
    assert np.allclose(pre, y.numpy(), rtol=1e-12, atol=1e-12)
    assert np.array_equal(out, F.bf16_rn(y.numpy()))
