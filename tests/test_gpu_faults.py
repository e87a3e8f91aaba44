"""Failure detection on the GPU without faulting it: a bounded wait that is
made to run out (a ready flag that is never set), and device offsets that
disagree with the schedule. Both must come back as a status the host reads,
with the GPU context still usable afterwards."""
import numpy as np
import pytest
import torch

import decode_phase_attention_gb300 as la
import workloads
from _parity import compare, reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def test_missing_ready_flag_times_out_and_poisons_only_that_unit():
    w = workloads.custom(1, 4, 4, 64, "f16", [4096])  # 16 tiles per head, I = 64
    q, k, v, _ = workloads.make_inputs(w, seed=4, device="cuda")
    ref = reference(w, q, k, v)
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=5)
    exp = la.la_schedule_export(dec.sched)
    G, U, nseg = exp[1], exp[2], exp[5]
    base = 8 + 2 * (G + 1) + (U + 1)
    segs = [exp[base + 5 * i: base + 5 * i + 5] for i in range(nseg)]
    host = next(s for s in segs if s[3] == la.SEG_HOST)
    unit, fin = host[0], host[4]
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=fin, spin_timeout_ns=50_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_ERR_TIMEOUT
    got = out.cpu().double().numpy().reshape(ref.shape)
    bad = np.isnan(got).any(axis=1)
    assert bad[unit] and bad.sum() == 1  # kv head == query head here
    compare(np.delete(got, unit, axis=0), np.delete(ref, unit, axis=0))
    # the context and the workspace stay usable
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=-1, spin_timeout_ns=2_000_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), ref)


def test_device_offsets_that_disagree_with_the_schedule_are_reported():
    w = workloads.custom(2, 4, 2, 128, "bf16", [1000, 3000])
    q, k, v, _ = workloads.make_inputs(w, seed=6, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=4)
    wrong = torch.tensor([0, 3000, 4000], dtype=torch.int32, device="cuda")  # same total, other split
    out = torch.empty(w.batch, w.hq, w.d, device="cuda")
    la.la_decode(q, k, v, wrong, dec.sched, dec.workspace, out, w.scale)
    assert dec.status() == la.LA_ERR_INVALID
    assert torch.isnan(out).all()
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), reference(w, q, k, v))


def test_trace_records_the_planned_work_of_every_cta():
    w = workloads.custom(3, 16, 2, 64, "bf16", [5000, 300, 12000])
    q, k, v, _ = workloads.make_inputs(w, seed=8, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=23)
    G = dec.sched.grid
    trace = torch.zeros(G * la.TRACE_WORDS, dtype=torch.int64, device="cuda")
    la.la_schedule_set_trace(dec.sched, trace)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    la.la_schedule_set_trace(dec.sched, None)
    compare(out.cpu(), reference(w, q, k, v))
    tr = trace.view(G, la.TRACE_WORDS).cpu().numpy()
    exp = la.la_schedule_export(dec.sched)
    cta_iter = np.array(exp[8:8 + G + 1])
    cta_seg = np.array(exp[8 + G + 1 + w.batch * w.hkv + 1:][:G + 1])
    assert np.array_equal(tr[:, 6], np.diff(cta_iter))  # tiles per CTA as planned
    assert np.array_equal(tr[:, 7], np.diff(cta_seg))   # segments per CTA as planned
    assert np.all(tr[:, 1] <= tr[:, 2]) and np.all(tr[:, 2] <= tr[:, 3]) and np.all(tr[:, 3] <= tr[:, 5])
    assert np.all(tr[:, 4] >= 0) and np.all(tr[:, 4] <= tr[:, 5] - tr[:, 1])
