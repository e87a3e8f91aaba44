"""GPU parity for several query tokens per request (speculative-decoding
verification): query i of request b sits at position L_b - nq + i and sees
keys 0 .. L_b - nq + i; the float64 oracle computes the same rows."""
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


def ref_spec(w, q, k, v):
    import oracle
    code = oracle.F16 if q.dtype == torch.float16 else oracle.BF16
    return oracle.attend(q.cpu(), k.cpu(), v.cpu(), w.cu, w.hq, w.hkv, w.d, w.scale, code, nq=w.nq)


CASES = [(d, grp, nq) for d in (64, 128) for grp, nq in ((1, 2), (1, 3), (1, 4), (1, 8), (2, 2), (2, 3),
                                                          (2, 4), (4, 2))]
CASES += [(80, 1, 4), (96, 2, 2), (256, 1, 5)]
# 9-16 query rows per kv head (two blocks of 8 on the tensor-core path)
CASES += [(64, 8, 2), (128, 8, 2), (128, 4, 4), (64, 2, 8), (128, 1, 16), (96, 4, 3), (256, 2, 6), (80, 8, 2)]
# groups that are not powers of two, times several query tokens
CASES += [(128, 3, 2), (64, 5, 3), (128, 7, 2)]


@pytest.mark.parametrize("d,grp,nq", CASES)
@pytest.mark.parametrize("grid", [5, 0])
def test_spec_decoding_rows(d, grp, nq, grid):
    # lengths put the draft tokens across tile boundaries (T = 256 / 128 / 64)
    lengths = [nq, 130, 257, 1000, 64 * 7 + 3]
    dt = "bf16" if (d + grp + nq) % 2 else "f16"
    w = workloads.custom(len(lengths), 2 * grp, 2, d, dt, lengths, nq=nq)
    q, k, v, _ = workloads.make_inputs(w, seed=d + 10 * nq + grp, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=grid, nq=nq)
    out = dec(q, k, v, w.scale)
    assert out.shape == (w.batch, nq, w.hq, w.d)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), ref_spec(w, q, k, v))


def test_spec_with_one_query_token_equals_plain_decode():
    w = workloads.custom(3, 8, 4, 128, "bf16", [500, 3000, 129])
    q, k, v, _ = workloads.make_inputs(w, seed=3, device="cuda")
    a = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu)(q, k, v, w.scale)
    s = la.la_plan_spec(w.batch, w.hq, w.hkv, w.d, 1, w.cu)
    ws = la.new_workspace(s)
    out = torch.empty_like(a)
    la.la_decode(q, k, v, torch.as_tensor(w.cu, device="cuda"), s, ws, out, w.scale)
    assert torch.equal(out, a)


@pytest.mark.parametrize("layout", ["token_major", "paged"])
def test_spec_on_a_paged_cache(layout):
    w = workloads.custom(3, 4, 2, 128, "bf16", [700, 64, 2001], nq=4)
    q, k, v, _ = workloads.make_inputs(w, seed=5, device="cuda")
    s = la.la_plan_spec(w.batch, w.hq, w.hkv, w.d, w.nq, w.cu)
    ws = la.new_workspace(s)
    out = torch.empty(w.batch, w.nq, w.hq, w.d, device="cuda")
    if layout == "paged":
        kc, vc, table, npages = workloads.to_paged(w, k, v, 32, seed=5)
        la.la_decode_kv(q, kc, vc, torch.as_tensor(w.cu, device="cuda"), s, ws, out, w.scale, layout="paged",
                        block_table=table.cuda(), page_size=32, num_pages=npages)
    else:
        kc, vc = workloads.to_token_major(w, k, v)
        la.la_decode_kv(q, kc, vc, torch.as_tensor(w.cu, device="cuda"), s, ws, out, w.scale, layout="token_major")
    assert la.la_get_status(ws) == la.LA_OK
    compare(out.cpu(), ref_spec(w, q, k, v))


def test_spec_workload_full_output():
    w = workloads.named("spec4")
    q, k, v, _ = workloads.make_inputs(w, seed=0, device="cuda")
    out = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, nq=w.nq)(q, k, v, w.scale)
    compare(out.cpu(), ref_spec(w, q, k, v))


@pytest.mark.parametrize("name", ["spec16", "spec32", "spec64"])
def test_long_drafts_at_bench_size(name):
    # batch 8, 32/32 heads, d 128, 8192-token contexts with 16, 32 or 64 draft
    # tokens per request (16 rows per kv head on the 16-row kernel, 32 and 64
    # on the tcgen05 kernel), in the launch configuration the bench times;
    # rows sampled for the oracle, the causal last tokens included
    import numpy as np
    import oracle
    w = workloads.named(name)
    q, k, v, _ = workloads.make_inputs(w, seed=7, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, nq=w.nq)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    rows = []
    for b in (0, 3, 7):
        for i in (0, w.nq // 2, w.nq - 1):
            for h in (0, 17, 31):
                rows.append((b * w.nq + i) * w.hq + h)
    rows = np.array(rows, np.int64)
    code = oracle.F16 if q.dtype == torch.float16 else oracle.BF16
    ref = oracle.attend(q.cpu(), k.cpu(), v.cpu(), w.cu, w.hq, w.hkv, w.d, w.scale, code, rows=rows, nq=w.nq)
    compare(out.view(-1, w.d)[rows].cpu(), ref)
