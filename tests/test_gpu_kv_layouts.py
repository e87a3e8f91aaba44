"""GPU parity for token-major and paged K/V caches (la_decode_kv): the
oracle gathers K and V from the same caches the kernel reads. Paged caches
put their pages in a seeded random order and fill unused slots with NaN,
so reading past a context shows up."""
import numpy as np
import pytest
import torch

import decode_phase_attention_gb300 as la
import oracle
import workloads
from _parity import compare
from oracle import layouts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def oracle_from_cache(w, q, kc, vc, gather):
    code = oracle.F16 if q.dtype == torch.float16 else oracle.BF16
    k = gather(kc.cpu().view(torch.int16).numpy().view(np.uint16))
    v = gather(vc.cpu().view(torch.int16).numpy().view(np.uint16))
    return oracle.attend(q.cpu(), k.astype(np.uint16), v.astype(np.uint16), w.cu, w.hq, w.hkv, w.d, w.scale, code)


def run(w, q, kc, vc, layout, grid=0, table=None, P=0, npages=0, out_dtype=torch.float32):
    s = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, grid)
    ws = la.new_workspace(s)
    out = torch.empty(w.batch, w.hq, w.d, dtype=out_dtype, device="cuda")
    la.la_decode_kv(q, kc, vc, torch.as_tensor(w.cu, device="cuda"), s, ws, out, w.scale, layout=layout,
                    block_table=table, page_size=P, num_pages=npages)
    assert la.la_get_status(ws) == la.LA_OK
    return out


CASES = [(64, 1, "f16"), (64, 8, "bf16"), (80, 1, "bf16"), (96, 4, "f16"), (128, 1, "bf16"), (128, 2, "f16"),
         (128, 8, "bf16"), (256, 1, "bf16"), (256, 4, "bf16")]
CASES += [(64, 16, "bf16"), (128, 16, "f16")]


@pytest.mark.parametrize("d,grp,dt", CASES)
def test_token_major_cache(d, grp, dt):
    w = workloads.custom(4, 2 * grp, 2, d, dt, [1, 700, 129, 3000])
    q, k, v, cu = workloads.make_inputs(w, seed=31, device="cuda")
    kc, vc = workloads.to_token_major(w, k, v)
    out = run(w, q, kc, vc, "token_major", grid=7)
    ref = oracle_from_cache(w, q, kc, vc, lambda c: layouts.gather_token_major(c, cu, w.hkv, w.d))
    compare(out.cpu(), ref)


@pytest.mark.parametrize("d,grp,dt", CASES)
@pytest.mark.parametrize("P", [32, 64, 256])
def test_paged_cache(d, grp, dt, P):
    w = workloads.custom(4, 2 * grp, 2, d, dt, [1, 700, 129, 3000])
    q, k, v, cu = workloads.make_inputs(w, seed=37, device="cuda")
    kc, vc, table, npages = workloads.to_paged(w, k, v, P, seed=P)
    out = run(w, q, kc, vc, "paged", grid=0, table=table.cuda(), P=P, npages=npages)
    ref = oracle_from_cache(w, q, kc, vc, lambda c: layouts.gather_paged(c, table.numpy(), cu, P, w.hkv, w.d))
    compare(out.cpu(), ref)


def test_paged_cache_with_16_token_pages_and_16_bit_output():
    w = workloads.custom(3, 16, 2, 128, "bf16", [2000, 33, 900])
    q, k, v, cu = workloads.make_inputs(w, seed=41, device="cuda")
    kc, vc, table, npages = workloads.to_paged(w, k, v, 16, seed=16)
    out = run(w, q, kc, vc, "paged", grid=11, table=table.cuda(), P=16, npages=npages, out_dtype=torch.bfloat16)
    ref = oracle_from_cache(w, q, kc, vc, lambda c: layouts.gather_paged(c, table.numpy(), cu, 16, w.hkv, w.d))
    got = out.double().cpu().numpy().reshape(ref.shape)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    assert np.all(np.abs(got - ref) <= 2e-3 + ulp)


@pytest.mark.parametrize("name", ["uniform", "ragged", "gqa"])
def test_named_workloads_in_a_paged_cache(name):
    w = workloads.named(name)
    q, k, v, cu = workloads.make_inputs(w, seed=0, device="cuda")
    kc, vc, table, npages = workloads.to_paged(w, k, v, 64, seed=0)
    del k, v
    out = run(w, q, kc, vc, "paged", table=table.cuda(), P=64, npages=npages)
    ref = oracle_from_cache(w, q, kc, vc, lambda c: layouts.gather_paged(c, table.numpy(), cu, 64, w.hkv, w.d))
    compare(out.cpu(), ref)
