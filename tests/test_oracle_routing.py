"""Pins for oracle.routing: hand-worked cases, brute force and invariants."""

import os

import numpy as np
import pytest

from oracle import routing as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ints(s):
    return [int(v) for v in s.split(",")] if s else []


def _cases():
    with open(os.path.join(GOLDEN, "route_pack_cases.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            name, m, k, eg, el, ids, em, counts, offsets, srt = line.strip().split("|")
            yield name, int(m), int(k), int(eg), int(el), _ints(ids), (None if em == "none" else _ints(em)), _ints(counts), _ints(offsets), _ints(srt)


@pytest.mark.parametrize("case", list(_cases()), ids=lambda c: c[0])
def test_route_pack_hand_worked(case):
    name, m, k, eg, el, ids, em, counts, offsets, srt = case
    ids = np.array(ids, dtype=np.int32).reshape(m, k)
    c, o, s = R.route_pack(ids, eg, el, em)
    assert c.tolist() == counts and o.tolist() == offsets and s.tolist() == srt


def test_capacity_is_next_pow2_and_ignores_top_k():
    assert [R.route_capacity_tokens(m) for m in (0, 1, 2, 3, 4, 5, 1023, 1024, 1025)] == [1, 1, 2, 4, 4, 8, 1024, 1024, 2048]
    assert R.route_capacity(0, 8) == 8 and R.route_capacity(3, 8) == 32


def _brute(ids, eg, el, em):
    m, k = ids.shape
    pairs = []
    for t in range(m):
        for j in range(k):
            i = int(ids[t, j])
            if not (0 <= i < eg):
                continue
            l = i if em is None else int(em[i])
            if 0 <= l < el:
                pairs.append((l, t * k + j))
    pairs.sort()
    counts = [sum(1 for l, _ in pairs if l == e) for e in range(el)]
    return counts, [r for _, r in pairs]


@pytest.mark.parametrize("seed", range(40))
def test_route_pack_brute_force(seed):
    rng = np.random.default_rng(seed)
    m = int(rng.integers(0, 40))
    k = int(rng.integers(1, 9))
    eg = int(rng.integers(1, 20))
    el = int(rng.integers(1, eg + 1))
    em = None
    if seed % 2:
        em = rng.integers(-2, el + 2, size=eg).astype(np.int32)
    ids = rng.integers(-2, eg + 2, size=(m, k)).astype(np.int32)
    c, o, s = R.route_pack(ids, eg, el, em)
    counts, order = _brute(ids, eg, el, em)
    assert c.tolist() == counts
    assert o[0] == 0 and o.tolist()[1:] == np.cumsum(counts).tolist()
    assert s[: len(order)].tolist() == order
    assert np.all(s[len(order):] == -1) and len(s) == R.route_capacity(m, k)
    # every valid route appears exactly once
    assert sorted(order) == sorted(set(order))
