"""GPU parity for units of several kv heads (la_plan_kv) on token-major and
paged caches: every output row against the float64 oracle, which gathers K
and V from the same caches by plain per-token indexing. Paged caches put
their pages in a seeded random order and fill unused slots with NaN."""
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
    return oracle.attend(q.cpu(), k.astype(np.uint16), v.astype(np.uint16), w.cu, w.hq, w.hkv, w.d, w.scale, code,
                         nq=w.nq)


def caches(w, k, v, layout, P):
    if layout == "token_major":
        kc, vc = workloads.to_token_major(w, k, v)
        return kc, vc, None, 0, lambda c: layouts.gather_token_major(c, w.cu, w.hkv, w.d)
    kc, vc, table, npages = workloads.to_paged(w, k, v, P, seed=P)
    return kc, vc, table, npages, lambda c: layouts.gather_paged(c, table.numpy(), w.cu, P, w.hkv, w.d)


def run(w, q, kc, vc, layout, grid=0, table=None, P=0, npages=0, out_dtype=torch.float32, heads_per_unit=0):
    s = la.la_plan_kv(w.batch, w.hq, w.hkv, w.d, w.cu, nq=w.nq, heads_per_unit=heads_per_unit, num_sms=grid)
    ws = la.new_workspace(s)
    shape = (w.batch, w.hq, w.d) if w.nq == 1 else (w.batch, w.nq, w.hq, w.d)
    out = torch.empty(*shape, dtype=out_dtype, device="cuda")
    la.la_decode_kv(q, kc, vc, torch.as_tensor(w.cu, device="cuda"), s, ws, out, w.scale, layout=layout,
                    block_table=None if table is None else table.cuda(), page_size=P, num_pages=npages)
    assert la.la_get_status(ws) == la.LA_OK
    return out, s


MULTI_HEAD = [(64, 2), (80, 2), (80, 8), (96, 2), (96, 4)]
CASES = [(d, hp, grp, dt) for d, hp in MULTI_HEAD
         for grp, dt in ((1, "f16"), (2, "bf16"), (4, "bf16"), (8, "f16"))]


@pytest.mark.parametrize("d,hp,grp,dt", CASES)
@pytest.mark.parametrize("layout,P", [("token_major", 0), ("paged", 16), ("paged", 64), ("paged", 256)])
def test_multi_head_units(d, hp, grp, dt, layout, P):
    # ragged lengths: a 1-token request, tails inside a page and across tiles;
    # two units per request
    hkv = 2 * hp
    w = workloads.custom(4, hkv * grp, hkv, d, dt, [1, 700, 129, 3000])
    q, k, v, _ = workloads.make_inputs(w, seed=d + hp + grp + P, device="cuda")
    kc, vc, table, npages, gather = caches(w, k, v, layout, P)
    out, s = run(w, q, kc, vc, layout, grid=7, table=table, P=P, npages=npages, heads_per_unit=hp)
    assert s.heads_per_unit == hp
    compare(out.cpu(), oracle_from_cache(w, q, kc, vc, gather))


@pytest.mark.parametrize("grid", [0, 1, 2, 5, 33, 150, 304])
def test_multi_head_units_over_grid_sizes(grid):
    w = workloads.custom(3, 48, 6, 64, "bf16", [2000, 37, 900])
    q, k, v, _ = workloads.make_inputs(w, seed=grid, device="cuda")
    kc, vc, table, npages, gather = caches(w, k, v, "paged", 32)
    per_sm, sms = la.la_device_capacity(64, 8)
    if grid > per_sm * sms:
        pytest.skip("grid larger than the device holds at once")
    out, _ = run(w, q, kc, vc, "paged", grid=grid, table=table, P=32, npages=npages)
    compare(out.cpu(), oracle_from_cache(w, q, kc, vc, gather))


@pytest.mark.parametrize("d,hp,grp,nq", [(64, 2, 1, 3), (64, 2, 2, 4), (64, 2, 4, 2), (80, 2, 1, 8), (80, 8, 2, 3),
                                         (96, 2, 2, 2), (96, 4, 1, 5)])
@pytest.mark.parametrize("layout,P", [("token_major", 0), ("paged", 16)])
def test_multi_head_units_with_several_query_tokens(d, hp, grp, nq, layout, P):
    lengths = [nq, 130, 257, 1000, 64 * 7 + 3]
    w = workloads.custom(len(lengths), hp * grp, hp, d, "bf16", lengths, nq=nq)
    q, k, v, _ = workloads.make_inputs(w, seed=d * nq + grp, device="cuda")
    kc, vc, table, npages, gather = caches(w, k, v, layout, P)
    out, s = run(w, q, kc, vc, layout, grid=5, table=table, P=P, npages=npages, heads_per_unit=hp)
    assert s.heads_per_unit == hp and out.shape == (w.batch, nq, w.hq, w.d)
    compare(out.cpu(), oracle_from_cache(w, q, kc, vc, gather))


def test_one_and_two_head_units_agree_and_16_bit_outputs_round_the_fp32_result():
    w = workloads.custom(2, 16, 2, 64, "bf16", [5000, 333])
    q, k, v, _ = workloads.make_inputs(w, seed=5, device="cuda")
    kc, vc, table, npages, gather = caches(w, k, v, "paged", 16)
    one, s1 = run(w, q, kc, vc, "paged", table=table, P=16, npages=npages, heads_per_unit=1)
    two, s2 = run(w, q, kc, vc, "paged", table=table, P=16, npages=npages, heads_per_unit=2)
    assert (s1.heads_per_unit, s2.heads_per_unit) == (1, 2)
    ref = oracle_from_cache(w, q, kc, vc, gather)
    compare(one.cpu(), ref)
    compare(two.cpu(), ref)
    b16, _ = run(w, q, kc, vc, "paged", table=table, P=16, npages=npages, out_dtype=torch.bfloat16)
    assert torch.equal(b16, two.to(torch.bfloat16))


@pytest.mark.parametrize("name,hp", [("gqa", 2), ("mha_h32_b8_c8192_d64", 2), ("hd80", 8), ("hd96", 4)])
@pytest.mark.parametrize("layout,P", [("token_major", 0), ("paged", 16)])
def test_named_workloads_with_multi_head_units(name, hp, layout, P):
    w = workloads.named(name)
    q, k, v, _ = workloads.make_inputs(w, seed=0, device="cuda")
    kc, vc, table, npages, gather = caches(w, k, v, layout, P)
    del k, v
    out, s = run(w, q, kc, vc, layout, table=table, P=P, npages=npages)
    assert s.heads_per_unit == hp  # the default choice
    compare(out.cpu(), oracle_from_cache(w, q, kc, vc, gather))


def test_slab_layout_is_refused_for_two_head_units():
    w = workloads.custom(1, 4, 4, 64, "f16", [1024])
    q, k, v, _ = workloads.make_inputs(w, seed=1, device="cuda")
    s = la.la_plan_kv(1, 4, 4, 64, w.cu, num_sms=3)
    ws = la.new_workspace(s)
    out = torch.empty(1, 4, 64, device="cuda")
    with pytest.raises(la.LeanAttentionError) as e:
        la.la_decode_kv(q, k, v, torch.as_tensor(w.cu, device="cuda"), s, ws, out, w.scale, layout="slab")
    assert e.value.status == la.LA_ERR_UNSUPPORTED
