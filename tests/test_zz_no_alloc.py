"""la_decode_static: the decode call for callers that cannot allocate device
memory (a plugin that cannot reach its host program's allocator, or a
serving loop that keeps all of HBM for its KV cache and must not call
cudaMalloc mid-decode). It keeps its scratch in a fixed 4 MiB array inside
the library instead of a caller workspace.

This file is collected last on purpose: if its GPU test fails, a run that
stops at the first failure has already run every other test. The GPU test
calls the entry point through the C ABI and checks it against la_decode on
two calls in a row (the array keeps the previous call's contents)."""
import ctypes

import numpy as np
import pytest
import torch

import decode_phase_attention_gb300 as la
import workloads
from _parity import MAX_ABS, REL_L2


def _static_call(q, k, v, cu, sched, out, scale):
    dt = la.LA_BF16 if q.dtype == torch.bfloat16 else la.LA_F16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return la._lib.la_decode_static(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                    ctypes.c_void_p(v.data_ptr()), dt, ctypes.c_void_p(cu.data_ptr()),
                                    sched.handle, ctypes.c_void_p(out.data_ptr()), ctypes.c_float(scale),
                                    stream)


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    assert np.all(np.isfinite(a))
    err = np.abs(a - b).max()
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)


def test_schedule_too_large_for_the_fixed_array_is_rejected_before_any_launch():
    # 8000 one-CTA units of 128 tokens at d = 128: 8000 records of 520 bytes > 4 MiB
    lengths = [128] * 250
    s = la.la_plan_fixed(250, 32, 32, 128, [0] + np.cumsum(lengths).tolist(), 1)
    assert s.grid == 8000
    p = ctypes.c_void_p(0x100000)  # never dereferenced: the size check comes first
    assert la._lib.la_decode_static(p, p, p, la.LA_BF16, p, s.handle, p, ctypes.c_float(0.1), None) \
        == la.LA_ERR_WORKSPACE


def test_wide_unit_records_fill_the_fixed_array_sooner():
    # units of more than 16 rows keep 128-row records (65 KiB each at
    # d = 128): 152 CTAs need 9.9 MiB, 48 fit in the 4 MiB array
    p = ctypes.c_void_p(0x100000)  # never dereferenced: the size check comes first
    big = la.la_plan(1, 64, 1, 128, [0, 100000], 152)
    assert la.la_workspace_size(big) > 4 << 20
    assert la._lib.la_decode_static(p, p, p, la.LA_BF16, p, big.handle, p, ctypes.c_float(0.1), None) \
        == la.LA_ERR_WORKSPACE


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["tiny", "ragged_gqa", "fixed_split", "three_query_tokens"])
def test_static_scratch_matches_la_decode_on_two_calls_in_a_row(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    if case == "tiny":
        w = workloads.named("tiny")
        make = lambda: la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, w.grid)  # noqa: E731
    elif case == "ragged_gqa":
        w = workloads.custom(5, 32, 4, 64, "bf16", [3000, 17, 20000, 257, 9000])
        make = lambda: la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, 0)  # noqa: E731
    elif case == "fixed_split":
        w = workloads.custom(3, 8, 8, 128, "f16", [5000, 300, 12000])
        make = lambda: la.la_plan_fixed(w.batch, w.hq, w.hkv, w.d, w.cu, 6)  # noqa: E731
    else:
        w = workloads.custom(3, 4, 2, 128, "bf16", [700, 3, 4000], nq=3)
        make = lambda: la.la_plan_spec(w.batch, w.hq, w.hkv, w.d, 3, w.cu)  # noqa: E731
    q, k, v, _ = workloads.make_inputs(w, seed=11, device="cuda")
    cu = torch.as_tensor(w.cu, dtype=torch.int32, device="cuda")
    sched = make()
    ref = torch.empty(*q.shape, device="cuda")
    ws = la.new_workspace(sched)
    la.la_decode(q, k, v, cu, sched, ws, ref, w.scale)
    assert la.la_get_status(ws) == la.LA_OK
    for _ in range(2):
        out = torch.full(tuple(q.shape), float("nan"), device="cuda")
        assert _static_call(q, k, v, cu, sched, out, w.scale) == la.LA_OK
        torch.cuda.synchronize()
        _close(out, ref)
