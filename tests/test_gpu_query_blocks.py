"""GPU parity for kv heads with more than 16 query rows (grouped-query groups
above 16, multi-query attention, or group x query tokens above 16). At
d = 64, 80, 96 and 128 a unit of up to 128 rows (64 at d = 256) runs on the
tcgen05 kernel; above that the query heads of a kv head
are split into equal blocks, each a stream-K unit of its own over the kv
head's K/V. The float64 oracle computes every row from the plain definition,
unaware of units and blocks."""
import numpy as np
import pytest
import torch

import decode_phase_attention_gb300 as la
import oracle
import workloads
from _parity import compare, reference, run_lean

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


# (d, hq, hkv, query blocks per kv head)
SLAB = [(128, 32, 1, 1), (128, 64, 1, 1), (64, 48, 2, 1), (96, 34, 2, 1), (80, 34, 2, 1), (80, 48, 2, 1),
        (256, 64, 2, 1), (128, 40, 2, 1), (64, 128, 1, 1), (128, 256, 1, 2), (64, 17, 1, 1), (128, 130, 1, 2),
        (96, 64, 1, 1), (96, 128, 1, 1), (80, 64, 1, 1), (96, 256, 1, 2), (80, 128, 1, 1), (80, 17, 1, 1),
        (80, 256, 1, 2), (256, 34, 2, 1), (256, 48, 2, 1), (256, 128, 1, 2), (256, 17, 1, 1), (256, 200, 2, 2)]


@pytest.mark.parametrize("d,hq,hkv,qb", SLAB)
@pytest.mark.parametrize("grid", [7, 0])
def test_query_blocks_slab(d, hq, hkv, qb, grid):
    lengths = [1000, 129, 2500, 64 * 5 + 1]
    dt = "bf16" if (d + hq) % 2 == 0 else "f16"
    w = workloads.custom(len(lengths), hq, hkv, d, dt, lengths)
    q, k, v, _ = workloads.make_inputs(w, seed=d + hq, device="cuda")
    out, dec = run_lean(w, q, k, v, num_sms=grid)
    assert dec.sched.query_blocks == qb
    compare(out.cpu(), reference(w, q, k, v))


def ref_spec(w, q, k, v):
    code = oracle.F16 if q.dtype == torch.float16 else oracle.BF16
    return oracle.attend(q.cpu(), k.cpu(), v.cpu(), w.cu, w.hq, w.hkv, w.d, w.scale, code, nq=w.nq)


# (d, grp, nq, query blocks): group x query tokens above 16
SPEC = [(128, 8, 4, 1), (64, 16, 2, 1), (64, 4, 5, 1), (128, 32, 2, 1), (96, 3, 7, 1), (80, 3, 7, 1),
        (128, 2, 16, 1), (128, 16, 9, 2), (64, 1, 100, 1), (96, 8, 4, 1), (80, 8, 4, 1), (128, 3, 40, 1),
        (80, 1, 100, 1), (256, 3, 7, 1), (256, 8, 4, 1), (256, 8, 9, 2), (256, 1, 40, 1)]


@pytest.mark.parametrize("d,grp,nq,qb", SPEC)
def test_query_blocks_with_several_query_tokens(d, grp, nq, qb):
    lengths = [nq, 300, 1000, 64 * 7 + 3, nq + 129]
    w = workloads.custom(len(lengths), 2 * grp, 2, d, "bf16", lengths, nq=nq)
    q, k, v, _ = workloads.make_inputs(w, seed=d + grp + nq, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=0, nq=nq)
    assert dec.sched.query_blocks == qb
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), ref_spec(w, q, k, v))


@pytest.mark.parametrize("layout", ["token_major", "paged"])
@pytest.mark.parametrize("d,hq,hkv,nq,qb", [(128, 32, 1, 1, 1), (64, 48, 2, 1, 1), (80, 64, 2, 1, 1),
                                            (128, 16, 2, 3, 1), (96, 40, 2, 1, 1), (80, 40, 2, 1, 1),
                                            (64, 256, 1, 1, 2), (256, 64, 2, 1, 1), (80, 20, 2, 2, 1),
                                            (256, 256, 2, 1, 2)])
def test_query_blocks_on_caches(layout, d, hq, hkv, nq, qb):
    from oracle import layouts
    lengths = [700, 64, 2000]
    w = workloads.custom(len(lengths), hq, hkv, d, "bf16", lengths, nq=nq)
    q, k, v, cu = workloads.make_inputs(w, seed=hq + d, device="cuda")
    cu_dev = torch.as_tensor(cu, device="cuda")
    s = la.la_plan_kv(w.batch, w.hq, w.hkv, w.d, cu, nq=nq, num_sms=0)
    assert s.query_blocks == qb and s.heads_per_unit == 1
    ws = la.new_workspace(s)
    out = torch.empty(w.batch, nq, w.hq, w.d, device="cuda")
    if layout == "token_major":
        kc, vc = workloads.to_token_major(w, k, v)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="token_major")
        kk = layouts.gather_token_major(kc.cpu().view(torch.int16).numpy(), cu, w.hkv, w.d)
        vv = layouts.gather_token_major(vc.cpu().view(torch.int16).numpy(), cu, w.hkv, w.d)
    else:
        kc, vc, table, npages = workloads.to_paged(w, k, v, 32, seed=hq)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="paged", block_table=table.cuda(),
                        page_size=32, num_pages=npages)
        kk = layouts.gather_paged(kc.cpu().view(torch.int16).numpy(), table.numpy(), cu, 32, w.hkv, w.d)
        vv = layouts.gather_paged(vc.cpu().view(torch.int16).numpy(), table.numpy(), cu, 32, w.hkv, w.d)
    assert la.la_get_status(ws) == la.LA_OK
    ref = oracle.attend(q.cpu(), kk.astype(np.int16).view(np.uint16), vv.astype(np.int16).view(np.uint16),
                        cu, w.hq, w.hkv, w.d, w.scale, oracle.BF16, nq=nq)
    compare(out.cpu(), ref)


@pytest.mark.parametrize("splits", [1, 4])
def test_query_blocks_with_fixed_partitions(splits):
    w = workloads.custom(3, 64, 2, 128, "bf16", [3000, 257, 900])
    q, k, v, _ = workloads.make_inputs(w, seed=64 + splits, device="cuda")
    out, dec = run_lean(w, q, k, v, fixed_splits=splits)
    assert dec.sched.query_blocks == 1
    compare(out.cpu(), reference(w, q, k, v))


def test_query_blocks_through_the_partition_choice():
    w = workloads.custom(2, 64, 1, 128, "bf16", [5000, 300])
    q, k, v, _ = workloads.make_inputs(w, seed=3, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, auto=True)
    assert dec.sched.query_blocks == 1
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), reference(w, q, k, v))


def test_query_blocks_through_the_allocation_free_entry():
    w = workloads.custom(3, 32, 1, 128, "bf16", [3000, 257, 900])
    q, k, v, cu = workloads.make_inputs(w, seed=11, device="cuda")
    s = la.la_plan(w.batch, w.hq, w.hkv, w.d, cu, 24)  # 24 records of 128 rows fit the fixed scratch
    out = torch.empty(w.batch, w.hq, w.d, device="cuda")
    la.la_decode_static(q, k, v, torch.as_tensor(cu, device="cuda"), s, out, w.scale)
    torch.cuda.synchronize()
    compare(out.cpu(), reference(w, q, k, v))


def test_multi_query_attention_at_scale():
    # 64 query heads on one kv head, 16 requests of 32k tokens (one unit of
    # 64 rows per request, every SM busy); rows sampled for the oracle
    w = workloads.custom(16, 64, 1, 128, "bf16", [32768] * 16)
    q, k, v, _ = workloads.make_inputs(w, seed=64, device="cuda")
    out, dec = run_lean(w, q, k, v)
    assert dec.sched.query_blocks == 1
    rows = np.array([0, 15, 16, 31, 47, 63, 64 * 7 + 20, 64 * 15 + 63], np.int64)
    compare(out.view(-1, 128)[rows].cpu(), reference(w, q, k, v, rows=rows))
