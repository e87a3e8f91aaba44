"""The decode call inside CUDA graphs and on concurrent streams: a captured
call replays with new query contents (the workspace epochs keep advancing
across replays), paged caches and fixed-split plans capture too, and two
schedules with their own workspaces run on two streams at once. Every output
is checked against the float64 oracle."""
import numpy as np
import pytest
import torch

import decode_phase_attention_gb300 as la
import oracle
import workloads
from _parity import compare, reference
from oracle import layouts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def fresh_q(q, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q.copy_(torch.randn(q.shape, generator=g, device="cuda", dtype=torch.float32).to(q.dtype))


@pytest.mark.parametrize("fixed_splits", [None, 1, 3])
def test_decode_replays_in_a_cuda_graph(fixed_splits):
    w = workloads.custom(3, 8, 4, 128, "bf16", [3000, 700, 129])
    q, k, v, _ = workloads.make_inputs(w, seed=1, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, fixed_splits=fixed_splits)
    out = torch.empty(w.batch, w.hq, w.d, device="cuda")
    dec(q, k, v, w.scale, out=out)  # the first call uploads the schedule: before any capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dec(q, k, v, w.scale, out=out)
    for rep in range(4):
        fresh_q(q, 100 + rep)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        compare(out.cpu(), reference(w, q, k, v))
    # eager calls and replays interleave on the same workspace
    dec(q, k, v, w.scale, out=out)
    graph.replay()
    torch.cuda.synchronize()
    compare(out.cpu(), reference(w, q, k, v))
    assert dec.status() == la.LA_OK


def test_paged_decode_with_multi_head_units_in_a_cuda_graph():
    w = workloads.custom(2, 16, 8, 64, "bf16", [2000, 333])
    q, k, v, cu = workloads.make_inputs(w, seed=2, device="cuda")
    kc, vc, table, npages = workloads.to_paged(w, k, v, 16, seed=2)
    table = table.cuda()
    s = la.la_plan_kv(w.batch, w.hq, w.hkv, w.d, cu)
    assert s.heads_per_unit == 2
    ws = la.new_workspace(s)
    cu_dev = torch.as_tensor(cu, device="cuda")
    out = torch.empty(w.batch, w.hq, w.d, device="cuda")

    def call():
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="paged", block_table=table,
                        page_size=16, num_pages=npages)

    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    kk = layouts.gather_paged(kc.cpu().view(torch.int16).numpy(), table.cpu().numpy(), cu, 16, w.hkv, w.d)
    vv = layouts.gather_paged(vc.cpu().view(torch.int16).numpy(), table.cpu().numpy(), cu, 16, w.hkv, w.d)
    kk, vv = kk.astype(np.int16).view(np.uint16), vv.astype(np.int16).view(np.uint16)
    for rep in range(3):
        fresh_q(q, 200 + rep)
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.attend(q.cpu(), kk, vv, cu, w.hq, w.hkv, w.d, w.scale, oracle.BF16)
        compare(out.cpu(), ref)
    assert la.la_get_status(ws) == la.LA_OK


def test_two_schedules_on_two_streams_at_once():
    wa = workloads.custom(2, 32, 32, 128, "bf16", [8192, 3000])
    wb = workloads.custom(4, 16, 2, 64, "f16", [5000, 1, 700, 129])
    qa, ka, va, _ = workloads.make_inputs(wa, seed=3, device="cuda")
    qb, kb, vb, _ = workloads.make_inputs(wb, seed=4, device="cuda")
    # well under half the SMs each, so both grids are resident together
    per_sm, sms = la.la_device_capacity(128, 1)
    grid = max(1, sms // 2 - 12)
    da = la.LeanDecoder(wa.batch, wa.hq, wa.hkv, wa.d, wa.cu, num_sms=grid)
    db = la.LeanDecoder(wb.batch, wb.hq, wb.hkv, wb.d, wb.cu, num_sms=grid)
    oa = torch.empty(wa.batch, wa.hq, wa.d, device="cuda")
    ob = torch.empty(wb.batch, wb.hq, wb.d, device="cuda")
    da(qa, ka, va, wa.scale, out=oa)
    db(qb, kb, vb, wb.scale, out=ob)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(10):
        with torch.cuda.stream(sa):
            da(qa, ka, va, wa.scale, out=oa, stream=sa)
        with torch.cuda.stream(sb):
            db(qb, kb, vb, wb.scale, out=ob, stream=sb)
    torch.cuda.synchronize()
    assert da.status(sa) == la.LA_OK and db.status(sb) == la.LA_OK
    compare(oa.cpu(), reference(wa, qa, ka, va))
    compare(ob.cpu(), reference(wb, qb, kb, vb))
