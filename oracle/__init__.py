"""Float64 CPU oracle for LeanAttention decode-phase attention.

TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the library and its Python binding
never do, and nothing here is a fallback for the GPU path. The oracle shares
no code with the CUDA library.

Contents:
  * lean_oracle.c (built into liboracle.so with gcc): the definition of
    decode attention in float64, the partial triple of a block of keys and
    the rescaling reduction f (xllm-io paper review, sections 3.1 and 3.2);
  * plan.py: the stream-K planner written the slow, direct way (same
    review, sections 3.3 to 3.5 and 4.3).

Parity status: every function here is pinned by tests/test_oracle_pins.py
and tests/test_planner_oracle.py against closed forms, library routines,
high-precision brute force and invariants; none is "parity unpinned".
"""
import ctypes
import os
import subprocess

import numpy as np

from . import plan  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lean_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F16, BF16, F64 = 0, 1, 2
_lib = None


def build(force=False):
    """Compile liboracle.so with gcc (plain C, IEEE double, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _open(path):
    """Load an oracle library file and declare its C signatures."""
    lib = ctypes.CDLL(path)
    vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_double
    lib.oracle_half_to_double.restype = dbl
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = dbl
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_array.restype = None
    lib.oracle_decode_array.argtypes = [i32, vp, vp, i64]
    lib.oracle_merge_f.restype = None
    lib.oracle_merge_f.argtypes = [i32, vp, vp, vp]
    lib.oracle_normalise.restype = None
    lib.oracle_normalise.argtypes = [i32, vp, vp]
    lib.oracle_partial.restype = i32
    lib.oracle_partial.argtypes = [i32, i32, vp, vp, vp, i64, i64, dbl, vp]
    lib.oracle_attend.restype = i32
    lib.oracle_attend.argtypes = [i32, i32, i32, i32, vp, i32, vp, vp, vp, dbl, i64, vp, vp, i32]
    lib.oracle_attend_spec.restype = i32
    lib.oracle_attend_spec.argtypes = [i32, i32, i32, i32, i32, vp, i32, vp, vp, vp, dbl, i64, vp, vp, i32]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _open(_LIB)
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_input(a, dtype):
    """Contiguous numpy view of an input: uint16 bit patterns for fp16/bf16, float64 otherwise."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().contiguous().cpu()
            if a.dtype in (torch.float16, torch.bfloat16):
                a = a.view(torch.int16).numpy().view(np.uint16)
            else:
                a = a.to(torch.float64).numpy()
    except ImportError:
        pass
    a = np.ascontiguousarray(a)
    if dtype in (F16, BF16):
        if a.dtype == np.float16:
            a = a.view(np.uint16)
        if a.dtype != np.uint16:
            raise TypeError("fp16/bf16 inputs are passed as their uint16 bit patterns")
    else:
        a = np.ascontiguousarray(a, dtype=np.float64)
    return a


def dtype_code(torch_dtype):
    import torch
    return {torch.float16: F16, torch.bfloat16: BF16, torch.float64: F64}[torch_dtype]


def half_to_double(bits):
    lib = _load()
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib.oracle_decode_array(F16, _ptr(bits), _ptr(out), bits.size)
    return out


def bf16_to_double(bits):
    lib = _load()
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib.oracle_decode_array(BF16, _ptr(bits), _ptr(out), bits.size)
    return out


def attend(q, k, v, cu, hq, hkv, d, scale, dtype, rows=None, threads=None, nq=1):
    """Decode attention for every (request, query token, query head) row, or the listed rows.

    q: [batch, nq, hq, d]; k, v: per request b a [hkv, L_b, d] slab at element
    offset hkv*cu[b]*d (L_b = cu[b+1]-cu[b]); query head h reads kv head
    h // (hq // hkv); with nq > 1 query i of request b sees keys
    0 .. L_b - nq + i. Returns float64 [nrows, d] (rows are (b*nq + i)*hq + h).
    """
    lib = _load()
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    batch = cu.size - 1
    qa, ka, va = _as_input(q, dtype), _as_input(k, dtype), _as_input(v, dtype)
    need_kv = int(cu[-1]) * hkv * d
    if qa.size < batch * nq * hq * d or ka.size < need_kv or va.size < need_kv:
        raise ValueError("input arrays are smaller than the shape implies")
    if rows is None:
        nrows, rows_ptr = batch * nq * hq, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rows_ptr = rows.size, _ptr(rows)
    out = np.zeros((nrows, d), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = lib.oracle_attend_spec(batch, int(nq), hq, hkv, d, _ptr(cu), dtype, _ptr(qa), _ptr(ka), _ptr(va),
                                float(scale), nrows, rows_ptr, _ptr(out), int(threads))
    if rc != 0:
        raise ValueError("oracle_attend rejected its arguments")
    return out


def attend_row(q, K, V, scale):
    """One row on float64 arrays: q [d], K [L, d], V [L, d] -> out [d]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    L, d = K.shape
    cu = np.array([0, L], dtype=np.int32)
    return attend(q.reshape(1, 1, d), K, V, cu, 1, 1, d, scale, F64, threads=1)[0]


def partial(q, K, V, t0, t1, scale):
    """Partial triple [m, l, Obar[d]] of one row over keys [t0, t1) (float64 inputs)."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    d = q.size
    if not (0 <= t0 <= t1 <= K.shape[0]):
        raise ValueError("bad key range")
    out = np.zeros(d + 2, dtype=np.float64)
    rc = lib.oracle_partial(d, F64, _ptr(q), _ptr(K), _ptr(V), int(t0), int(t1), float(scale),
                            _ptr(out))
    if rc != 0:
        raise MemoryError("oracle_partial")
    return out


def merge_f(x, y):
    """The rescaling reduction f on triples [m, l, Obar[d]]."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.ascontiguousarray(y, dtype=np.float64)
    out = np.zeros_like(x)
    lib.oracle_merge_f(x.size - 2, _ptr(x), _ptr(y), _ptr(out))
    return out


def normalise(x):
    """O = Obar / l."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(x.size - 2, dtype=np.float64)
    lib.oracle_normalise(x.size - 2, _ptr(x), _ptr(out))
    return out
