"""The tcgen05 kernel (units of 17-128 query rows at d = 64, 96 and 128) under
the same checks as the 16-row kernel: a bounded wait made to run out and
device offsets that disagree with the schedule come back as a status with
the context still usable; the trace records the planned work; the ring
depth, 16-bit outputs and CUDA-graph replay leave results unchanged."""
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


def segments(sched):
    exp = la.la_schedule_export(sched)
    G, U, nseg = exp[1], exp[2], exp[5]
    base = 8 + 2 * (G + 1) + (U + 1)
    return [exp[base + 5 * i: base + 5 * i + 5] for i in range(nseg)]


def test_missing_ready_flag_times_out_and_poisons_only_that_unit():
    w = workloads.custom(1, 64, 2, 128, "bf16", [4096])  # two units of 32 rows, 32 tiles each
    q, k, v, _ = workloads.make_inputs(w, seed=4, device="cuda")
    ref = reference(w, q, k, v).reshape(w.hq, w.d)
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=5)
    host = next(s for s in segments(dec.sched) if s[3] == la.SEG_HOST)
    unit, fin = host[0], host[4]
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=fin, spin_timeout_ns=50_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_ERR_TIMEOUT
    got = out.cpu().double().numpy().reshape(w.hq, w.d)
    bad = np.isnan(got).any(axis=1)
    rows = np.arange(unit * 32, unit * 32 + 32)  # the unit's query heads
    assert bad[rows].all() and bad.sum() == 32
    keep = np.setdiff1d(np.arange(w.hq), rows)
    compare(got[keep], ref[keep])
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=-1, spin_timeout_ns=2_000_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), ref)


def test_device_offsets_that_disagree_with_the_schedule_are_reported():
    w = workloads.custom(2, 32, 1, 64, "bf16", [1000, 3000])
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
    w = workloads.custom(3, 48, 2, 128, "bf16", [5000, 300, 12000])
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


@pytest.mark.parametrize("d", [64, 80, 96, 128, 256])
def test_ring_depth_does_not_change_the_result(d):
    w = workloads.custom(2, 64, 2, d, "bf16", [3000, 777])
    q, k, v, cu = workloads.make_inputs(w, seed=d, device="cuda")
    outs = []
    for stages in (0, 2, 3):
        s = la.la_plan(w.batch, w.hq, w.hkv, w.d, cu, 0)
        la.la_schedule_set_stages(s, stages)
        ws = la.new_workspace(s)
        out = torch.empty(w.batch, w.hq, w.d, device="cuda")
        la.la_decode(q, k, v, torch.as_tensor(cu, device="cuda"), s, ws, out, w.scale)
        assert la.la_get_status(ws) == la.LA_OK
        outs.append(out)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    compare(outs[0].cpu(), reference(w, q, k, v))


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d,hq", [(128, 32), (80, 32), (80, 96), (256, 48)])
def test_sixteen_bit_outputs_are_the_fp32_outputs_rounded(out_dtype, d, hq):
    # 32 rows: lane replicas; 96 rows at d = 80: one replica (20-dim O quarters)
    w = workloads.custom(2, hq, 1, d, "f16", [2000, 513])
    q, k, v, cu = workloads.make_inputs(w, seed=3, device="cuda")
    s = la.la_plan(w.batch, w.hq, w.hkv, w.d, cu, 0)
    ws = la.new_workspace(s)
    cu_dev = torch.as_tensor(cu, device="cuda")
    o32 = torch.empty(w.batch, w.hq, w.d, device="cuda")
    la.la_decode(q, k, v, cu_dev, s, ws, o32, w.scale)
    o16 = torch.empty(w.batch, w.hq, w.d, device="cuda", dtype=out_dtype)
    la.la_decode(q, k, v, cu_dev, s, ws, o16, w.scale)
    assert la.la_get_status(ws) == la.LA_OK
    assert torch.equal(o16, o32.to(out_dtype))


def test_graph_replay_matches_eager_calls():
    w = workloads.custom(4, 64, 1, 128, "bf16", [1500, 4000, 129, 2048])
    q, k, v, _ = workloads.make_inputs(w, seed=12, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu)
    eager = dec(q, k, v, w.scale).clone()  # the first call uploads the schedule: before any capture
    out = torch.empty_like(eager)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dec(q, k, v, w.scale, out=out)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert dec.status() == la.LA_OK
    compare(eager.cpu(), reference(w, q, k, v))
