"""Pins for the reference planner (oracle/plan.py).

It is checked against a hand-derived schedule (tests/golden), against the
special cases of the xllm-io review's "4.3 hardware-aware work distribution"
(G equal to the number of output tiles behaves like FlashAttention-2; G a
multiple of it like FlashDecoding) and against invariants that follow from
"3.4 stream-K style decomposition" and "3.5 execution flow".
"""
import json
import os

import numpy as np
import pytest

from oracle import plan as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
KIND = {"whole": P.WHOLE, "nonhost": P.NONHOST, "host": P.HOST, "partial": P.PARTIAL}


def cu_of(lengths):
    return [0] + np.cumsum(lengths).tolist()


def test_lean_tile_table_matches_the_review():
    g = json.load(open(os.path.join(GOLDEN, "lean_tile.json")))
    for d, t in g["lean_tile_tokens"].items():
        assert P.lean_tile(int(d)) == t
    with pytest.raises(ValueError):
        P.lean_tile(96)


def test_hand_derived_tiny_schedule():
    g = json.load(open(os.path.join(GOLDEN, "plan_tiny_g3.json")))
    s = g["shape"]
    p = P.plan_lean(s["batch"], s["hq"], s["hkv"], s["d"], cu_of(s["lengths"]), s["G"])
    assert p["T"] == g["T"] and p["I"] == g["I"]
    assert p["cta_iter"] == g["cta_iter"]
    assert p["unit_iter"] == g["unit_iter"]
    assert p["unit_host"] == g["unit_host"] and p["unit_fin"] == g["unit_fin"]
    for c, segs in enumerate(g["segments"]):
        got = p["segs"][p["cta_seg"][c]:p["cta_seg"][c + 1]]
        want = [(u, t0, t1, KIND[k], peer) for u, t0, t1, k, peer in segs]
        assert got == want


def check_lean_invariants(p, lengths, hkv, d):
    G, U, I, T = p["G"], p["U"], p["I"], p["T"]
    tiles = [-(-L // T) for L in lengths for _ in range(hkv)]
    assert U == len(tiles) and I == sum(tiles)
    # even split: every CTA has floor or ceil of I / G iterations, the larger ones first
    counts = np.diff(p["cta_iter"])
    assert set(counts.tolist()) <= {I // G, -(-I // G)}
    assert list(counts) == sorted(counts, reverse=True)
    cover = np.zeros(I, int)
    host_count = np.zeros(U, int)
    for g in range(G):
        segs = p["segs"][p["cta_seg"][g]:p["cta_seg"][g + 1]]
        pos = p["cta_iter"][g]
        for j, (u, t0, t1, kind, peer) in enumerate(segs):
            assert 0 <= t0 < t1 <= tiles[u]
            a = p["unit_iter"][u] + t0
            assert a == pos  # segments are contiguous and in order
            pos += t1 - t0
            cover[a:a + t1 - t0] += 1
            if kind == P.NONHOST:
                assert j == 0 and t0 > 0  # at most one, and it is the CTA's first work
            if kind in (P.HOST, P.WHOLE):
                assert t0 == 0
                host_count[u] += 1
                assert p["unit_host"][u] == g
            if kind == P.HOST:
                assert j == len(segs) - 1 and t1 < tiles[u] and peer == p["unit_fin"][u] > g
            if kind == P.WHOLE:
                assert t1 == tiles[u] and p["unit_fin"][u] == g
            if kind != P.HOST:
                assert peer == -1
        assert pos == p["cta_iter"][g + 1]
    assert np.all(cover == 1)  # every iteration exactly once
    assert np.all(host_count == 1)  # exactly one host per unit
    # every CTA between host and finisher works only on that unit
    for u in range(U):
        h, f = p["unit_host"][u], p["unit_fin"][u]
        for g in range(h + 1, f + 1):
            first = p["segs"][p["cta_seg"][g]]
            assert first[0] == u and first[3] == P.NONHOST


@pytest.mark.parametrize("seed", range(40))
def test_lean_invariants_random_shapes(seed):
    r = np.random.default_rng(seed)
    batch = int(r.integers(1, 6))
    hkv = int(r.integers(1, 5))
    grp = int(r.choice([1, 2, 4, 8]))
    d = int(r.choice([64, 128]))
    lengths = r.integers(1, 2000, size=batch).tolist()
    tiles = sum(-(-L // P.lean_tile(d)) for L in lengths) * hkv
    G = int(r.integers(1, tiles + 5))
    p = P.plan_lean(batch, hkv * grp, hkv, d, cu_of(lengths), G)
    check_lean_invariants(p, lengths, hkv, d)


def test_grid_equal_to_units_is_the_flashattention2_partition():
    lengths = [1000] * 3
    p = P.plan_lean(3, 8, 4, 128, cu_of(lengths), 12)
    for g in range(12):
        segs = p["segs"][p["cta_seg"][g]:p["cta_seg"][g + 1]]
        assert segs == [(g, 0, 8, P.WHOLE, -1)]


@pytest.mark.parametrize("k", [2, 3, 4, 8])
def test_grid_multiple_of_units_is_the_flashdecoding_split(k):
    tiles = 8 * 3  # divisible by every k above except where tested below
    if tiles % k:
        pytest.skip("needs tiles divisible by k")
    L = tiles * 256
    p = P.plan_lean(2, 4, 2, 64, cu_of([L, L]), 4 * k)
    for u in range(4):
        pieces = [s for s in p["segs"] if s[0] == u]
        assert len(pieces) == k
        assert all(s[2] - s[1] == tiles // k for s in pieces)
        assert pieces[0][3] == P.HOST and all(s[3] == P.NONHOST for s in pieces[1:])


def test_more_ctas_than_iterations_leaves_the_rest_idle():
    p = P.plan_lean(1, 2, 2, 64, cu_of([300]), 7)  # 2 tiles per head, I = 4
    assert p["cta_iter"] == [0, 1, 2, 3, 4, 4, 4, 4]
    assert p["cta_seg"][4:] == [4, 4, 4, 4]


def test_fixed_partition_planner():
    lengths = [5 * 128, 1 * 128 + 1, 3]
    p = P.plan_fixed(3, 2, 1, 128, cu_of(lengths), 1)
    assert p["G"] == 3 and all(s[3] == P.WHOLE for s in p["segs"])
    p = P.plan_fixed(3, 2, 1, 128, cu_of(lengths), 3)
    # unit 0 has 5 tiles -> 3 pieces (1, 2, 2 tiles); unit 1 has 2 tiles -> 2 pieces; unit 2 -> 1
    assert p["G"] == 6
    assert [s[:4] for s in p["segs"]] == [(0, 0, 1, P.PARTIAL), (0, 1, 3, P.PARTIAL),
                                          (0, 3, 5, P.PARTIAL), (1, 0, 1, P.PARTIAL),
                                          (1, 1, 2, P.PARTIAL), (2, 0, 1, P.WHOLE)]
    assert p["unit_host"] == [0, 3, 5] and p["unit_fin"] == [2, 4, 5]


def test_rejects_empty_context():
    with pytest.raises(ValueError):
        P.plan_lean(2, 4, 4, 64, [0, 10, 10], 4)
