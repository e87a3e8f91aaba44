"""la_decode_static: the decode call for callers that cannot allocate device
memory (a plugin that cannot reach its host program's allocator, or a
serving loop that keeps all of HBM for its KV cache and must not call
cudaMalloc mid-decode). It keeps its scratch in a fixed 4 MiB array inside
the library instead of a caller workspace.

This file is collected last on purpose: if its GPU test fails, a run that
stops at the first failure has already run every other test. The GPU tests
call the entry point through the C ABI and check it against la_decode and
against the float64 oracle on two calls in a row (the array keeps the
previous call's contents), after a larger schedule has left its flags,
records and tables in the array, where the second record slot per CTA of
the shared merge does not fit (every split unit is then merged at its
host), and when a bounded wait runs out."""
import ctypes

import numpy as np
import pytest
import torch

import decode_phase_attention_gb300 as la
import workloads
from _parity import MAX_ABS, REL_L2, compare, reference


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
    exact = reference(w, q, k, v)
    for _ in range(2):
        out = torch.full(tuple(q.shape), float("nan"), device="cuda")
        assert _static_call(q, k, v, cu, sched, out, w.scale) == la.LA_OK
        torch.cuda.synchronize()
        _close(out, ref)
        compare(out.cpu(), exact)


def _decode_both(w, q, k, v, cu, sched):
    ref = torch.empty(*q.shape, device="cuda")
    ws = la.new_workspace(sched)
    la.la_decode(q, k, v, cu, sched, ws, ref, w.scale)
    assert la.la_get_status(ws) == la.LA_OK
    out = torch.full(tuple(q.shape), float("nan"), device="cuda")
    assert _static_call(q, k, v, cu, sched, out, w.scale) == la.LA_OK
    torch.cuda.synchronize()
    return out, ref


@pytest.mark.gpu
def test_static_scratch_merges_at_the_host_when_two_record_slots_do_not_fit():
    # d 256, group 16, every SM: two record slots per CTA (the shared merge
    # of split units) need 5.1 MB, one slot fits; the call merges every
    # split unit at its host instead and matches the oracle
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    w = workloads.custom(1, 32, 2, 256, "bf16", [20000])
    q, k, v, _ = workloads.make_inputs(w, seed=17, device="cuda")
    cu = torch.as_tensor(w.cu, dtype=torch.int32, device="cuda")
    sched = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, 0)
    assert la.la_workspace_size(sched) > 4 << 20
    out, ref = _decode_both(w, q, k, v, cu, sched)
    _close(out, ref)
    compare(out.cpu(), reference(w, q, k, v))


@pytest.mark.gpu
def test_static_scratch_after_a_larger_schedule_and_back():
    # A stream-K schedule over every SM with many split units leaves flags,
    # records and tables in the array; a smaller, different schedule follows,
    # then the first one again (its tables must be copied back in).
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    big = workloads.custom(6, 16, 4, 128, "bf16", [9000, 40000, 3, 700, 21000, 12345])
    small = workloads.custom(2, 8, 8, 64, "f16", [1500, 300])
    runs = []
    for w, grid in ((big, 0), (small, 5), (big, 0)):
        q, k, v, _ = workloads.make_inputs(w, seed=13, device="cuda")
        cu = torch.as_tensor(w.cu, dtype=torch.int32, device="cuda")
        sched = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, grid)
        out, ref = _decode_both(w, q, k, v, cu, sched)
        _close(out, ref)
        compare(out.cpu(), reference(w, q, k, v))
        runs.append(sched.grid)
    assert runs[0] > runs[1]


@pytest.mark.gpu
def test_static_scratch_wait_that_runs_out_gives_nan_for_that_unit_only():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    w = workloads.custom(1, 4, 4, 64, "f16", [4096])  # 16 tiles per head, I = 64
    q, k, v, _ = workloads.make_inputs(w, seed=4, device="cuda")
    cu = torch.as_tensor(w.cu, dtype=torch.int32, device="cuda")
    exact = reference(w, q, k, v)
    sched = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, 5)
    exp = la.la_schedule_export(sched)
    G, U, nseg = exp[1], exp[2], exp[5]
    base = 8 + 2 * (G + 1) + (U + 1)
    segs = [exp[base + 5 * i: base + 5 * i + 5] for i in range(nseg)]
    host = next(s for s in segs if s[3] == la.SEG_HOST)
    unit, fin = host[0], host[4]
    la.la_schedule_set_debug(sched, skip_signal_cta=fin, spin_timeout_ns=50_000_000)
    out = torch.zeros(tuple(q.shape), device="cuda")
    assert _static_call(q, k, v, cu, sched, out, w.scale) == la.LA_OK
    torch.cuda.synchronize()
    got = out.cpu().double().numpy().reshape(exact.shape)
    bad = np.isnan(got).any(axis=1)
    assert bad[unit] and bad.sum() == 1  # kv head == query head here
    compare(np.delete(got, unit, axis=0), np.delete(exact, unit, axis=0))
    # the next clean call on the same array is correct
    la.la_schedule_set_debug(sched, skip_signal_cta=-1, spin_timeout_ns=2_000_000_000)
    out = torch.full(tuple(q.shape), float("nan"), device="cuda")
    assert _static_call(q, k, v, cu, sched, out, w.scale) == la.LA_OK
    torch.cuda.synchronize()
    compare(out.cpu(), exact)
