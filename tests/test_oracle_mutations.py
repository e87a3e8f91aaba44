"""The oracle's pins catch planted mistakes.

Each case copies oracle/lean_oracle.c, plants one plausible mistake (a
dropped term, a wrong sign, a wrong index, a transposed operand, a broken
reduction), compiles the copy and runs a battery of pin checks against it:
closed forms, library routines and invariants of the attention definition
(xllm-io review of LeanAttention, "3.1" and "3.2"). Every mutant must fail
at least one check, and the unmodified source must pass all of them.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "lean_oracle.c")

MUTATIONS = {
    "exponent sign": ("double p = exp(s[t] - m);", "double p = exp(m - s[t]);"),
    "dropped scale": ("s[t] = scale * acc;", "s[t] = acc;"),
    "dropped l term": ("    l += p;\n", "    l += 1.0;\n"),
    "K and V swapped in q.k": ("acc += elem(q, q_off + c, dtype) * elem(k, krow + c, dtype);",
                               "acc += elem(q, q_off + c, dtype) * elem(v, krow + c, dtype);"),
    "V row ignores the block start": ("long vrow = kv_off + (t0 + t) * (long)d;", "long vrow = kv_off + t * (long)d;"),
    "kv head mapping": ("kvh = h / grp;", "kvh = h % j->hkv;"),
    "slab offset drops the head": ("long kv_off = ((long)j->hkv * j->cu[b] + kvh * L) * (long)j->d;",
                                   "long kv_off = ((long)j->hkv * j->cu[b]) * (long)j->d;"),
    "f weights y with x's factor": ("double l = ax * x[1] + ay * y[1];", "double l = ax * x[1] + ax * y[1];"),
    "f keeps the wrong max": ("  out[0] = m;\n", "  out[0] = mx;\n"),
    "f drops the O rescale": ("out[2 + c] = ax * x[2 + c] + ay * y[2 + c];", "out[2 + c] = x[2 + c] + y[2 + c];"),
    "normalise multiplies": ("o[c] = x[2 + c] / x[1];", "o[c] = x[2 + c] * x[1];"),
    "fp16 exponent bias": ("mag = ldexp(1024.0 + (double)f, e - 25);", "mag = ldexp(1024.0 + (double)f, e - 24);"),
    "fp16 subnormal scale": ("mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);"),
    "bf16 exponent bias": ("mag = ldexp(128.0 + (double)f, e - 134);", "mag = ldexp(128.0 + (double)f, e - 133);"),
    "bf16 sign dropped": ("  return sign ? -mag : mag;\n}\n\nvoid oracle_decode_array",
                          "  return mag;\n}\n\nvoid oracle_decode_array"),
}


def battery():
    """Pin checks; returns the names of those that fail."""
    from scipy.special import softmax
    failed = []
    r = np.random.default_rng(77)

    def check(name, fn):
        try:
            ok = fn()
        except Exception:
            ok = False
        if not ok:
            failed.append(name)

    def two_keys():
        d, scale = 8, 0.3
        q, K, V = r.normal(size=d), r.normal(size=(2, d)), r.normal(size=(2, d))
        s0, s1 = scale * math.fsum(q * K[0]), scale * math.fsum(q * K[1])
        w0 = 1 / (1 + math.exp(s1 - s0))
        return np.allclose(oracle.attend_row(q, K, V, scale), w0 * V[0] + (1 - w0) * V[1], rtol=1e-12, atol=1e-14)

    def mean_of_v():
        K, V = r.normal(size=(33, 8)), r.normal(size=(33, 8))
        return np.allclose(oracle.attend_row(np.zeros(8), K, V, 0.5), V.mean(0), rtol=1e-12, atol=1e-14)

    def one_hot():
        K, V = r.normal(size=(20, 8)), r.normal(size=(20, 8))
        return np.allclose(oracle.attend_row(300 * K[5], K, V, 1.0), V[5], atol=1e-12)

    def scipy_ref():
        q, K, V = r.normal(size=16), r.normal(size=(50, 16)), r.normal(size=(50, 16))
        return np.allclose(oracle.attend_row(q, K, V, 0.25), softmax(0.25 * K @ q) @ V, rtol=1e-12, atol=1e-14)

    def markers():
        lens, hq, hkv, d = [3, 5], 4, 2, 4
        cu = np.array([0, 3, 8], np.int32)
        K = r.normal(size=hkv * 8 * d)
        V = np.zeros(hkv * 8 * d)
        for b in range(2):
            for h in range(hkv):
                for t in range(lens[b]):
                    off = (hkv * cu[b] + h * lens[b] + t) * d
                    V[off:off + d] = [b, h, 1, 2]
        out = oracle.attend(r.normal(size=(2, hq, d)), K, V, cu, hq, hkv, d, 0.5, oracle.F64, threads=2)
        want = np.array([[b, h // 2, 1, 2] for b in range(2) for h in range(hq)], float)
        return np.allclose(out, want, atol=1e-13)

    def split_merge():
        q, K, V = r.normal(size=8), r.normal(size=(40, 8)), r.normal(size=(40, 8))
        x, y, z = (oracle.partial(q, K, V, a, b, 0.4) for a, b in ((0, 7), (7, 8), (8, 40)))
        lft = oracle.merge_f(oracle.merge_f(x, y), z)
        rgt = oracle.merge_f(x, oracle.merge_f(y, z))
        return (np.allclose(lft, rgt, rtol=1e-12) and
                np.allclose(oracle.normalise(lft), oracle.attend_row(q, K, V, 0.4), rtol=1e-12, atol=1e-14))

    def fp16_decode():
        bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        ref = bits.view(np.float16).astype(np.float64)
        got = oracle.half_to_double(bits)
        fin = np.isfinite(ref)
        return np.array_equal(got[fin], ref[fin])

    def bf16_decode():
        bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
        got = oracle.bf16_to_double(bits)
        fin = np.isfinite(ref)
        return np.array_equal(got[fin], ref[fin])

    for name, fn in (("two keys", two_keys), ("mean", mean_of_v), ("one hot", one_hot), ("scipy", scipy_ref),
                     ("markers", markers), ("split/merge", split_merge), ("fp16 decode", fp16_decode),
                     ("bf16 decode", bf16_decode)):
        check(name, fn)
    return failed


def _compile(src_text, tmp_path, name):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src_text)
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(c),
                    "-lm", "-lpthread"], check=True)
    return str(so)


def _with_library(path):
    saved = oracle._lib
    oracle._lib = oracle._open(path)
    try:
        return battery()
    finally:
        oracle._lib = saved


def test_unmodified_oracle_passes_the_battery(tmp_path):
    assert _with_library(_compile(open(SRC).read(), tmp_path, "orig")) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    failed = _with_library(_compile(src.replace(old, new), tmp_path, "mut"))
    assert failed, f"no pin caught the mutation '{name}'"
