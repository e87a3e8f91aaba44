"""Pins for the float64 oracle: it is checked against things other than itself.

Each test ties the oracle to a closed form, a library routine, a
high-precision brute force or an invariant of the attention definition
(xllm-io paper review of LeanAttention, "3.1 standard attention" and
"3.2 softmax rescaling as a reduction"). Together they are chosen so that a
dropped term, a wrong sign, a wrong index or a transposed operand in the
oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def rng(seed):
    return np.random.default_rng(seed)


# --- element decoding --------------------------------------------------------

def test_half_decode_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_matches_torch_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_double(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("tdt,code", [(torch.float16, oracle.F16), (torch.bfloat16, oracle.BF16)])
def test_half_inputs_equal_their_decoded_doubles(tdt, code):
    g = torch.Generator().manual_seed(3)
    L, d = 37, 16
    q = torch.randn(1, 1, d, generator=g).to(tdt)
    k = torch.randn(L * d, generator=g).to(tdt)
    v = torch.randn(L * d, generator=g).to(tdt)
    cu = np.array([0, L], np.int32)
    a = oracle.attend(q, k, v, cu, 1, 1, d, 0.25, code, threads=1)
    b = oracle.attend(q.double().numpy(), k.double().numpy(), v.double().numpy(), cu, 1, 1, d,
                      0.25, oracle.F64, threads=1)
    assert np.array_equal(a, b)


# --- closed forms and hand cases -------------------------------------------

def test_single_key_returns_its_value_exactly():
    r = rng(1)
    for d in (1, 8, 64):
        q, K, V = r.normal(size=d), r.normal(size=(1, d)), r.normal(size=(1, d))
        assert np.array_equal(oracle.attend_row(q, K, V, 0.7), V[0])


def test_two_keys_follow_the_logistic_closed_form():
    r = rng(2)
    d, scale = 16, 0.3
    for _ in range(20):
        q, K, V = r.normal(size=d), r.normal(size=(2, d)), r.normal(size=(2, d))
        s0 = scale * math.fsum(q * K[0])
        s1 = scale * math.fsum(q * K[1])
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        expect = w0 * V[0] + w1 * V[1]
        np.testing.assert_allclose(oracle.attend_row(q, K, V, scale), expect, rtol=1e-13, atol=1e-15)


def test_hand_checked_d1_case():
    # scores 0, ln 2, ln 3 -> weights 1:2:3 of 6; values 6, 12, 18 -> (6 + 24 + 54) / 6 = 14
    q = np.array([1.0])
    K = np.array([[0.0], [math.log(2.0)], [math.log(3.0)]])
    V = np.array([[6.0], [12.0], [18.0]])
    out = oracle.attend_row(q, K, V, 1.0)
    assert abs(out[0] - 14.0) < 1e-13
    # the scale multiplies the scores: scale 2 gives weights 1:4:9 of 14 -> (6+48+162)/14
    out2 = oracle.attend_row(q, K, V, 2.0)
    assert abs(out2[0] - 216.0 / 14.0) < 1e-13


def test_constant_scores_give_the_mean_of_v():
    r = rng(4)
    L, d = 57, 32
    K, V = r.normal(size=(L, d)), r.normal(size=(L, d))
    np.testing.assert_allclose(oracle.attend_row(np.zeros(d), K, V, 0.5), V.mean(axis=0),
                               rtol=1e-13, atol=1e-15)
    # scale 0 makes every score zero whatever q is
    np.testing.assert_allclose(oracle.attend_row(r.normal(size=d), K, V, 0.0), V.mean(axis=0),
                               rtol=1e-13, atol=1e-15)


def test_one_hot_scores_select_one_value_row():
    r = rng(5)
    L, d = 40, 16
    K, V = r.normal(size=(L, d)), r.normal(size=(L, d))
    for j in (0, 17, L - 1):
        q = 200.0 * K[j]
        s = K @ q
        assert s[j] - np.max(np.delete(s, j)) > 60  # the selected score dominates by > 60
        np.testing.assert_allclose(oracle.attend_row(q, K, V, 1.0), V[j], rtol=0, atol=1e-20 + 1e-12)


def test_shift_of_every_key_changes_nothing():
    r = rng(6)
    L, d = 33, 8
    K = r.integers(-8, 9, size=(L, d)).astype(np.float64)  # exact in float64
    V = r.normal(size=(L, d))
    q = r.integers(-3, 4, size=d).astype(np.float64)
    u = r.integers(-5, 6, size=d).astype(np.float64)
    a = oracle.attend_row(q, K, V, 0.125)
    b = oracle.attend_row(q, K + u, V, 0.125)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_joint_permutation_of_keys_and_values_changes_nothing():
    r = rng(7)
    L, d = 64, 16
    q, K, V = r.normal(size=d), r.normal(size=(L, d)), r.normal(size=(L, d))
    perm = r.permutation(L)
    np.testing.assert_allclose(oracle.attend_row(q, K, V, 0.25),
                               oracle.attend_row(q, K[perm], V[perm], 0.25), rtol=1e-12, atol=1e-14)


def test_matches_scipy_softmax():
    from scipy.special import softmax
    r = rng(8)
    for L, d in ((1, 4), (5, 64), (300, 128), (1000, 64)):
        q, K, V = r.normal(size=d), r.normal(size=(L, d)), r.normal(size=(L, d))
        scale = 1.0 / math.sqrt(d)
        expect = softmax(scale * (K @ q)) @ V
        np.testing.assert_allclose(oracle.attend_row(q, K, V, scale), expect, rtol=1e-12, atol=1e-14)


def test_brute_force_high_precision_tiny_inputs():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    r = rng(9)
    for L in range(1, 7):
        d = 3
        q, K, V = r.normal(size=d) * 2, r.normal(size=(L, d)) * 2, r.normal(size=(L, d))
        scale = 0.6
        s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[c]) * mpmath.mpf(K[t, c]) for c in range(d))
             for t in range(L)]
        e = [mpmath.exp(x) for x in s]
        tot = mpmath.fsum(e)
        expect = [float(mpmath.fsum(e[t] * mpmath.mpf(V[t, c]) for t in range(L)) / tot) for c in range(d)]
        np.testing.assert_allclose(oracle.attend_row(q, K, V, scale), expect, rtol=1e-14, atol=1e-15)
        # the partial triple of the whole row: m = max score, l = sum exp(s - m)
        tri = oracle.partial(q, K, V, 0, L, scale)
        m = max(s)
        assert abs(tri[0] - float(m)) <= 1e-14 * max(1.0, abs(float(m)))
        assert abs(tri[1] - float(mpmath.fsum(mpmath.exp(x - m) for x in s))) <= 1e-14 * tri[1]


# --- batched layout: ragged requests and grouped query heads ------------------

def test_batched_layout_reads_the_right_slab_and_kv_head():
    # Every value row of slab (b, kvh) is the marker vector (b, kvh, ...); attention
    # weights sum to one, so out[b, h] must equal the marker of (b, h // grp).
    r = rng(10)
    lens = [3, 1, 7, 5]
    batch, hq, hkv, d = len(lens), 6, 2, 4
    grp = hq // hkv
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = hkv * cu[-1] * d
    K = r.normal(size=n)
    V = np.zeros(n)
    for b in range(batch):
        for h in range(hkv):
            for t in range(lens[b]):
                off = (hkv * cu[b] + h * lens[b] + t) * d
                V[off:off + d] = [b, h, 10 * b + h, 1.0]
    q = r.normal(size=(batch, hq, d))
    out = oracle.attend(q, K, V, cu, hq, hkv, d, 0.5, oracle.F64, threads=3)
    for b in range(batch):
        for h in range(hq):
            np.testing.assert_allclose(out[b * hq + h], [b, h // grp, 10 * b + h // grp, 1.0],
                                       rtol=1e-14, atol=1e-14)


def test_batched_rows_match_single_rows_on_sliced_slabs():
    from scipy.special import softmax
    r = rng(11)
    lens = [300, 17, 129, 256]
    batch, hq, hkv, d = len(lens), 8, 2, 64
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    K = r.normal(size=hkv * cu[-1] * d)
    V = r.normal(size=hkv * cu[-1] * d)
    q = r.normal(size=(batch, hq, d))
    out = oracle.attend(q, K, V, cu, hq, hkv, d, 0.125, oracle.F64, threads=4)
    rows = np.array([5, 0, 31, 12], np.int64)
    sub = oracle.attend(q, K, V, cu, hq, hkv, d, 0.125, oracle.F64, rows=rows, threads=2)
    np.testing.assert_array_equal(sub, out[rows])
    for b in range(batch):
        slab_k = K[hkv * cu[b] * d:hkv * cu[b + 1] * d].reshape(hkv, lens[b], d)
        slab_v = V[hkv * cu[b] * d:hkv * cu[b + 1] * d].reshape(hkv, lens[b], d)
        for h in range(hq):
            kv = h // (hq // hkv)
            expect = softmax(0.125 * (slab_k[kv] @ q[b, h])) @ slab_v[kv]
            np.testing.assert_allclose(out[b * hq + h], expect, rtol=1e-12, atol=1e-14)


# --- the reduction f -----------------------------------------------------------

def _random_cuts(r, L, k):
    cuts = sorted(r.choice(np.arange(1, L), size=k - 1, replace=False).tolist())
    return [0] + cuts + [L]


def test_f_is_associative_on_random_unequal_splits_and_equals_the_unsplit_row():
    r = rng(12)
    for trial in range(30):
        L, d = int(r.integers(3, 400)), int(r.choice([1, 8, 64, 128]))
        q, K, V = r.normal(size=d), r.normal(size=(L, d)) * 1.5, r.normal(size=(L, d))
        scale = 1 / math.sqrt(d)
        c = _random_cuts(r, L, 3)
        x, y, z = (oracle.partial(q, K, V, c[i], c[i + 1], scale) for i in range(3))
        left = oracle.merge_f(oracle.merge_f(x, y), z)
        right = oracle.merge_f(x, oracle.merge_f(y, z))
        np.testing.assert_allclose(left, right, rtol=1e-12, atol=1e-14)
        full = oracle.attend_row(q, K, V, scale)
        np.testing.assert_allclose(oracle.normalise(left), full, rtol=1e-12, atol=1e-14)
        # the merged statistics equal those of the unsplit block
        whole = oracle.partial(q, K, V, 0, L, scale)
        np.testing.assert_allclose(left[:2], whole[:2], rtol=1e-12)


def test_f_k_way_folds_in_any_grouping_agree():
    r = rng(13)
    L, d = 500, 64
    q, K, V = r.normal(size=d), r.normal(size=(L, d)), r.normal(size=(L, d))
    scale = 0.125
    for k in (2, 5, 11):
        c = _random_cuts(r, L, k)
        parts = [oracle.partial(q, K, V, c[i], c[i + 1], scale) for i in range(k)]
        acc_l = parts[0]
        for p in parts[1:]:
            acc_l = oracle.merge_f(acc_l, p)
        acc_r = parts[-1]
        for p in reversed(parts[:-1]):
            acc_r = oracle.merge_f(p, acc_r)
        # a random tree
        pool = list(parts)
        while len(pool) > 1:
            i = int(r.integers(0, len(pool) - 1))
            pool[i:i + 2] = [oracle.merge_f(pool[i], pool[i + 1])]
        for other in (acc_r, pool[0]):
            np.testing.assert_allclose(acc_l, other, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(oracle.normalise(acc_l), oracle.attend_row(q, K, V, scale),
                                   rtol=1e-12, atol=1e-14)


def test_f_weights_each_side_by_its_own_maximum():
    # two single-key blocks: f must reproduce the logistic weights of the two scores
    d = 2
    x = np.array([3.0, 1.0, 10.0, 0.0])   # m = 3, l = 1, Obar = v0 = (10, 0)
    y = np.array([1.0, 1.0, 0.0, 20.0])   # m = 1, l = 1, Obar = v1 = (0, 20)
    out = oracle.normalise(oracle.merge_f(x, y))
    w0 = 1.0 / (1.0 + math.exp(1.0 - 3.0))
    np.testing.assert_allclose(out, [w0 * 10.0, (1 - w0) * 20.0], rtol=1e-14)
    # and it is symmetric in its operands
    np.testing.assert_allclose(oracle.merge_f(x, y), oracle.merge_f(y, x), rtol=1e-15)


def test_f_identity_element():
    r = rng(14)
    d = 16
    q, K, V = r.normal(size=d), r.normal(size=(9, d)), r.normal(size=(9, d))
    x = oracle.partial(q, K, V, 2, 9, 0.25)
    empty = oracle.partial(q, K, V, 4, 4, 0.25)
    assert empty[0] == -np.inf and empty[1] == 0 and not np.any(empty[2:])
    np.testing.assert_array_equal(oracle.merge_f(x, empty), x)
    np.testing.assert_array_equal(oracle.merge_f(empty, x), x)


# --- several query tokens per request (speculative-decoding verification) -----

def test_each_query_token_sees_exactly_its_causal_prefix():
    r = rng(15)
    lens, nq, hq, hkv, d = [9, 4, 30], 4, 4, 2, 8
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    K = r.normal(size=hkv * cu[-1] * d)
    V = r.normal(size=hkv * cu[-1] * d)
    q = r.normal(size=(len(lens), nq, hq, d))
    out = oracle.attend(q, K, V, cu, hq, hkv, d, 0.3, oracle.F64, nq=nq, threads=3)
    for b, L in enumerate(lens):
        slab_k = K[hkv * cu[b] * d:hkv * cu[b + 1] * d].reshape(hkv, L, d)
        slab_v = V[hkv * cu[b] * d:hkv * cu[b + 1] * d].reshape(hkv, L, d)
        for i in range(nq):
            vis = L - nq + i + 1  # keys 0 .. L - nq + i
            for h in range(hq):
                kv = h // (hq // hkv)
                want = oracle.attend_row(q[b, i, h], slab_k[kv, :vis], slab_v[kv, :vis], 0.3)
                np.testing.assert_array_equal(out[(b * nq + i) * hq + h], want)


def test_keys_after_a_query_token_do_not_change_it():
    r = rng(16)
    L, nq, d = 20, 3, 16
    cu = np.array([0, L], np.int32)
    K, V = r.normal(size=L * d), r.normal(size=L * d)
    q = r.normal(size=(1, nq, 1, d))
    base = oracle.attend(q, K, V, cu, 1, 1, d, 0.25, oracle.F64, nq=nq, threads=1)
    K2, V2 = K.copy(), V.copy()
    K2[(L - 1) * d:] += 5.0  # the last key: visible to the last query only
    V2[(L - 1) * d:] -= 3.0
    moved = oracle.attend(q, K2, V2, cu, 1, 1, d, 0.25, oracle.F64, nq=nq, threads=1)
    np.testing.assert_array_equal(moved[:nq - 1], base[:nq - 1])
    assert not np.allclose(moved[nq - 1], base[nq - 1])


def test_one_query_token_is_ordinary_decode():
    r = rng(17)
    cu = np.array([0, 50, 51], np.int32)
    K, V = r.normal(size=2 * 51 * 8), r.normal(size=2 * 51 * 8)
    q = r.normal(size=(2, 4, 8))
    a = oracle.attend(q, K, V, cu, 4, 2, 8, 0.5, oracle.F64)
    b = oracle.attend(q.reshape(2, 1, 4, 8), K, V, cu, 4, 2, 8, 0.5, oracle.F64, nq=1)
    np.testing.assert_array_equal(a, b)
