"""GPU pins of the building blocks: tcgen05 layouts, the dequantiser, route packing.

* a single tcgen05.mma with A written to tensor memory by tcgen05.st and B in
  the library's shared-memory layout equals a float64 matmul (bf16 inputs);
* the register dequantiser applied to b4_prepare_weights output reproduces
  the oracle's dequantised weights (times 2^-63) bit for bit, over all E2M1
  codes and a spread of E4M3 / E8M0 scales, including zero scales, subnormal
  E4M3 scales and the K / row padding;
* b4_route_pack is bit-exact against the oracle.
"""

import ctypes
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import formats as F  # noqa: E402
from oracle import quant as Q  # noqa: E402
from oracle import routing as R  # noqa: E402

from gpu_util import dev  # noqa: E402

PROBE = os.path.join(os.path.dirname(__file__), "csrc", "libb4probe.so")


@pytest.fixture(scope="module")
def probe():
    if not os.path.exists(PROBE):
        pytest.fail("tests/csrc/libb4probe.so missing: run __graft_entry__.build()")
    lib = ctypes.CDLL(PROBE)
    for name in ("probe_mma_ts", "probe_mma_rowb", "probe_dequant", "probe_dequant_f16", "probe_bf16_mul", "probe_tma",
                 "probe_mma_sw128"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


@pytest.fixture(scope="module")
def b4():
    import w4a16_moe_gb300 as b4mod

    return b4mod


@pytest.mark.parametrize("n", [16, 48, 128, 192, 256])
def test_tcgen05_mma_a_in_tmem_matches_matmul(probe, n):
    rng = np.random.default_rng(n)
    a = F.bf16_rn(rng.standard_normal((128, 64)))
    b = F.bf16_rn(rng.standard_normal((n, 64)))
    A = dev(F.bf16_bits(a).view(np.int16))
    B = dev(F.bf16_bits(b).view(np.int16))
    D = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    rc = probe.probe_mma_ts(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()), n,
                            ctypes.c_void_p(D.data_ptr()), ctypes.c_void_p(status.data_ptr()))
    assert rc == 0 and status.cpu().tolist() == [0, 0]
    want = a @ b.T
    got = D.cpu().numpy().astype(np.float64)
    assert np.allclose(got, want, rtol=1e-5, atol=1e-4), np.abs(got - want).max()


def test_tcgen05_single_row_b_descriptor(probe):
    """The decode path's B operand: one natural-order row, K stride 16 B, N stride 0."""
    rng = np.random.default_rng(5)
    a = F.bf16_rn(rng.standard_normal((128, 64)))
    x = F.bf16_rn(rng.standard_normal(64))
    A = dev(F.bf16_bits(a).view(np.int16))
    X = dev(F.bf16_bits(x).view(np.int16))
    D = torch.full((128, 16), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert probe.probe_mma_rowb(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(X.data_ptr()),
                                ctypes.c_void_p(D.data_ptr()), ctypes.c_void_p(status.data_ptr())) == 0
    assert status.cpu().tolist() == [0, 0]
    got = D.cpu().numpy().astype(np.float64)
    want = a @ x
    assert np.allclose(got[:, 0], want, rtol=1e-5, atol=1e-4), np.abs(got[:, 0] - want).max()
    assert np.array_equal(got[:, 8], got[:, 0])  # rows 8..15 repeat rows 0..7


def _sw128_expect(rows_data, first_slot):
    """128-byte swizzle: 16-byte chunk c of the row in atom slot q lands at chunk c ^ (q % 8)."""
    out = {}
    for j, row in enumerate(rows_data):
        q = first_slot + j
        for c in range(8):
            out[(q, c ^ (q % 8))] = row[8 * c: 8 * c + 8]
    return out


def _tma_call(probe, src, mode, c0, rows4, box_rows, dst_off):
    out = torch.zeros(256 * 128, dtype=torch.uint8, device="cuda")
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    r4 = (ctypes.c_int * 4)(*rows4)
    rc = probe.probe_tma(ctypes.c_void_p(src.data_ptr()), src.shape[0], src.shape[1], mode, c0, r4, box_rows, dst_off,
                         ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(status.data_ptr()))
    assert rc == 0 and status.cpu().tolist() == [0, 0], rc
    return out.cpu().numpy().view(np.uint16)  # 16-bit elements


def test_tma_tile_box_lands_in_128b_swizzle(probe):
    rng = np.random.default_rng(7)
    src_np = rng.integers(0, 1 << 16, size=(300, 128), dtype=np.uint16)
    src = dev(src_np.view(np.int16))
    for r0, c0, box in ((100, 64, 40), (280, 0, 32)):  # second box runs past the last row
        got = _tma_call(probe, src, 0, c0, (r0, 0, 0, 0), box, 0)
        rows = [src_np[r0 + j, c0:c0 + 64] if r0 + j < 300 else np.zeros(64, np.uint16) for j in range(box)]
        for (q, c), want in _sw128_expect(rows, 0).items():
            assert np.array_equal(got[q * 64 + c * 8: q * 64 + c * 8 + 8], want), (r0, q, c)


@pytest.mark.parametrize("dst_off", [0, 512])
def test_tma_gather4_rows(probe, dst_off):
    rng = np.random.default_rng(8)
    src_np = rng.integers(0, 1 << 16, size=(300, 128), dtype=np.uint16)
    src = dev(src_np.view(np.int16))
    rows4 = (5, 250, 17, 99)
    got = _tma_call(probe, src, 1, 64, rows4, 1, dst_off)
    rows = [src_np[r, 64:128] for r in rows4]
    addr_based = all(np.array_equal(got[q * 64 + c * 8: q * 64 + c * 8 + 8], w)
                     for (q, c), w in _sw128_expect(rows, dst_off // 128).items())
    box_based = all(np.array_equal(got[(dst_off // 128 + j) * 64 + (c ^ j) * 8:(dst_off // 128 + j) * 64 + (c ^ j) * 8 + 8],
                                   rows[j][8 * c:8 * c + 8]) for j in range(4) for c in range(8))
    assert addr_based, f"swizzle follows the shared-memory address: {addr_based}; follows the box row: {box_based}"


@pytest.mark.parametrize("n", [16, 128, 160])
def test_tcgen05_mma_with_sw128_b(probe, n):
    rng = np.random.default_rng(9 + n)
    a = F.bf16_rn(rng.standard_normal((128, 64)))
    b = F.bf16_rn(rng.standard_normal((n, 64)))
    A = dev(F.bf16_bits(a).view(np.int16))
    B = dev(F.bf16_bits(b).view(np.int16))
    D = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert probe.probe_mma_sw128(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()), n,
                                 ctypes.c_void_p(D.data_ptr()), ctypes.c_void_p(status.data_ptr())) == 0
    assert status.cpu().tolist() == [0, 0]
    got = D.cpu().numpy().astype(np.float64)
    assert np.allclose(got, a @ b.T, rtol=1e-5, atol=1e-4), np.abs(got - a @ b.T).max()


def test_bf16_mul_keeps_subnormal_inputs(probe):
    # the dequantiser multiplies e2m1 * 2^-126 patterns (0.5 -> subnormal 0x0040)
    a = np.array([0x00400040, 0x80400040, 0x00C00080, 0x01C00000], dtype=np.uint32)
    b = np.array([0x5F005F00, 0x5F005F00, 0x63606360, 0x5A805A80], dtype=np.uint32)  # 2^63, 2^63, 448*2^63, 2^54
    d = torch.zeros(4, dtype=torch.int32, device="cuda")
    A, B = dev(a.view(np.int32)), dev(b.view(np.int32))
    assert probe.probe_bf16_mul(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                                ctypes.c_void_p(d.data_ptr()), 4) == 0
    got = d.cpu().numpy().view(np.uint32)

    def val(bits):
        return F.bf16_from_bits(np.array([bits & 0xFFFF, bits >> 16]))

    for ai, bi, gi in zip(a, b, got):
        want = F.bf16_rn(val(int(ai)) * val(int(bi)))
        assert np.array_equal(val(int(gi)), want), (hex(ai), hex(bi), hex(gi))


def _serving_expected(codes, scales, fmt, which, act, hidden, inter):
    """Expected dequantiser output in serving order: [E, tiles, stages, 128, 64] bf16 bits."""
    e_l = codes.shape[0]
    kvalid = hidden if which == 0 else inter
    inter_pad = -(-inter // 64) * 64
    if which == 0:
        tiles = inter_pad // 64 if act == 0 else -(-inter // 128)
    else:
        tiles = -(-hidden // 128)
    stages = -(-kvalid // 64)
    out = np.zeros((e_l, tiles, stages, 128, 64), dtype=np.float64)
    for e in range(e_l):
        w = Q.dequant(codes[e], scales[e], fmt, gs=None if fmt == Q.MXFP4 else 1.0)
        wpad = np.zeros((w.shape[0], stages * 64))
        wpad[:, :kvalid] = w
        for t in range(tiles):
            for r in range(128):
                if which == 0 and act == 0:
                    q, l = divmod(r, 32)
                    i = t * 64 + q * 16 + (l % 16)
                    src = (i if l < 16 else inter + i) if i < inter else -1
                else:
                    n = t * 128 + r
                    src = n if n < w.shape[0] else -1
                if src >= 0:
                    out[e, t, :, r, :] = wpad[src].reshape(stages, 64)
    return F.bf16_bits(F.bf16_rn(out * 2.0 ** -63)), (tiles, stages)


@pytest.mark.parametrize("fmt,which,act,hidden,inter", [
    (Q.NVFP4, 0, 0, 128, 96),    # SwiGLU interleave, I not a multiple of 64
    (Q.NVFP4, 0, 1, 80, 144),    # ReLU^2 W1, K tail (80 = 64 + 16)
    (Q.NVFP4, 1, 0, 144, 96),    # W2, rows tail, K tail
    (Q.MXFP4, 0, 0, 96, 64),     # MXFP4, K = 96 not 128-aligned
    (Q.MXFP4, 1, 0, 160, 96),    # MXFP4 W2 tails
])
def test_prepare_and_dequant_bit_exact(probe, b4, fmt, which, act, hidden, inter):
    rng = np.random.default_rng(hidden * 7 + inter + which)
    e_l = 3
    n, k = ((2 * inter if act == 0 else inter), hidden) if which == 0 else (hidden, inter)
    g = Q.GROUP[fmt]
    codes = Q.pack_nibbles(rng.integers(0, 16, size=(e_l, n, k), dtype=np.uint8))
    if fmt == Q.NVFP4:
        # every finite E4M3 code, both signs, zero and subnormal scales included
        pool = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    else:
        pool = np.arange(65, 192, dtype=np.uint8)
    scales = pool[rng.integers(0, len(pool), size=(e_l, n, k // g))]
    expect, (tiles, stages) = _serving_expected(codes, scales, fmt, which, act, hidden, inter)
    cfg = b4.MoEConfig(m=1, top_k=1, num_global_experts=e_l, num_local_experts=e_l, hidden=hidden, inter=inter,
                       format=0 if fmt == Q.NVFP4 else 1)
    pc, ps = b4.prepare_weights(cfg, which, act, dev(codes), dev(scales))
    nblk = e_l * tiles * stages
    out = torch.zeros(nblk * 128 * 64, dtype=torch.int16, device="cuda")
    assert probe.probe_dequant(ctypes.c_void_p(pc.data_ptr()), ctypes.c_void_p(ps.data_ptr()),
                               0 if fmt == Q.NVFP4 else 1, nblk, ctypes.c_void_p(out.data_ptr())) == 0
    got = out.cpu().numpy().view(np.uint16).reshape(expect.shape)
    # signed zeros are equal here: a zero-scale block is stored with +0 codes
    zg, ze = (got & 0x7FFF) == 0, (expect & 0x7FFF) == 0
    bad = np.argwhere((got != expect) & ~(zg & ze))
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[0].tolist()}: got {got[tuple(bad[0])]:#06x} want {expect[tuple(bad[0])]:#06x}"


@pytest.mark.parametrize("fmt,which,act,hidden,inter", [
    (Q.NVFP4, 0, 0, 128, 96),
    (Q.NVFP4, 1, 0, 144, 96),
    (Q.MXFP4, 0, 0, 96, 64),
    (Q.MXFP4, 1, 0, 160, 96),
])
def test_prepare_and_f16_dequant_exact(probe, b4, fmt, which, act, hidden, inter):
    """The small-m kernels' dequantiser (bit-pair exchange of the serving
    word, hardware E2M1 -> f16 conversion, fp32 block scale) reproduces the
    oracle's dequantised weights exactly: every E2M1 value times an E4M3 or
    E8M0 scale is exact in fp32."""
    rng = np.random.default_rng(hidden * 5 + inter + which)
    e_l = 3
    n, k = ((2 * inter if act == 0 else inter), hidden) if which == 0 else (hidden, inter)
    g = Q.GROUP[fmt]
    codes = Q.pack_nibbles(rng.integers(0, 16, size=(e_l, n, k), dtype=np.uint8))
    if fmt == Q.NVFP4:
        pool = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    else:
        pool = np.arange(65, 192, dtype=np.uint8)
    scales = pool[rng.integers(0, len(pool), size=(e_l, n, k // g))]
    expect_bits, (tiles, stages) = _serving_expected(codes, scales, fmt, which, act, hidden, inter)
    # the bf16 expectation is exact (times 2^-63): undo the factor
    expect = F.bf16_from_bits(expect_bits).astype(np.float64) * 2.0 ** 63
    cfg = b4.MoEConfig(m=1, top_k=1, num_global_experts=e_l, num_local_experts=e_l, hidden=hidden, inter=inter,
                       format=0 if fmt == Q.NVFP4 else 1)
    pc, ps = b4.prepare_weights(cfg, which, act, dev(codes), dev(scales))
    nblk = e_l * tiles * stages
    out = torch.zeros(nblk * 128 * 64, dtype=torch.float32, device="cuda")
    assert probe.probe_dequant_f16(ctypes.c_void_p(pc.data_ptr()), ctypes.c_void_p(ps.data_ptr()),
                                   0 if fmt == Q.NVFP4 else 1, nblk, ctypes.c_void_p(out.data_ptr())) == 0
    got = out.cpu().numpy().astype(np.float64).reshape(expect.shape)
    bad = np.argwhere(got != expect)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[0].tolist()}: got {got[tuple(bad[0])]} want {expect[tuple(bad[0])]}"


def test_prepare_rejects_invalid_scales(b4):
    cfg = b4.MoEConfig(m=1, top_k=1, num_global_experts=1, num_local_experts=1, hidden=64, inter=64, format=0)
    codes = torch.full((1, 64, 32), 0x11, dtype=torch.uint8, device="cuda")
    scales = torch.full((1, 64, 4), 0x38, dtype=torch.uint8, device="cuda")
    b4.prepare_weights(cfg, 1, 1, codes, scales)
    scales[0, 3, 1] = 0x7F  # E4M3 NaN
    with pytest.raises(b4.B4Error) as ei:
        b4.prepare_weights(cfg, 1, 1, codes, scales)
    assert ei.value.status == b4.B4_ERR_INVALID_ARGUMENT
    cfgm = b4.MoEConfig(m=1, top_k=1, num_global_experts=1, num_local_experts=1, hidden=64, inter=64, format=1)
    sm = torch.full((1, 64, 2), 127, dtype=torch.uint8, device="cuda")
    b4.prepare_weights(cfgm, 1, 1, codes, sm)
    sm[0, 0, 0] = 255
    with pytest.raises(b4.B4Error):
        b4.prepare_weights(cfgm, 1, 1, codes, sm)
    sm[0, 0, 0] = 10  # tiny scale with nonzero codes
    with pytest.raises(b4.B4Error):
        b4.prepare_weights(cfgm, 1, 1, codes, sm)
    codes[0, 0, :16] = 0  # the block (k < 32) is all zero -> accepted
    b4.prepare_weights(cfgm, 1, 1, codes, sm)


def _route_case(seed):
    rng = np.random.default_rng(seed)
    m = int(rng.choice([0, 1, 2, 3, 4, 5, 16, 17, 63, 64, 65, 257, 1000, 2048, 4096]))
    k = int(rng.integers(1, 9))
    eg = int(rng.choice([1, 2, 8, 33, 128, 256]))
    el = int(rng.integers(1, eg + 1))
    em = None
    if seed % 3 == 1 or el != eg:
        em = rng.integers(-1, el + 1, size=eg).astype(np.int32)
    bad_frac = rng.choice([0.0, 0.01, 0.5, 1.0])
    ids = rng.integers(0, eg, size=(m, k)).astype(np.int32)
    mask = rng.random((m, k)) < bad_frac
    ids[mask] = rng.choice([-1, eg, -7, eg + 100], size=int(mask.sum()))
    return m, k, eg, el, em, ids


@pytest.mark.parametrize("seed", range(24))
def test_route_pack_bit_exact(b4, seed):
    m, k, eg, el, em, ids = _route_case(seed)
    cfg = b4.MoEConfig(m=m, top_k=k, num_global_experts=eg, num_local_experts=el, hidden=64, inter=64,
                       expert_map=None if em is None else dev(em))
    cap = b4.route_capacity_tokens(m) * k
    assert cap == R.route_capacity(m, k)
    counts = torch.full((el,), -5, dtype=torch.int32, device="cuda")
    offsets = torch.full((el + 1,), -5, dtype=torch.int32, device="cuda")
    srt = torch.full((cap,), -5, dtype=torch.int32, device="cuda")
    ids_d = dev(ids) if m else torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        b4.route_pack(cfg, ids_d, counts, offsets, srt, stream=stream)
    stream.synchronize()
    c, o, s = R.route_pack(ids, eg, el, em)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(srt.cpu().numpy(), s)
