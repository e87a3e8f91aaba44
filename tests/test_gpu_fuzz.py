"""Seeded random configurations through every decode entry point, each
checked against the float64 oracle: head dims, groups, query tokens, grids,
cache layouts, page sizes, output types and ragged lengths drawn at random."""
import numpy as np
import pytest
import torch

import decode_phase_attention_gb300 as la
import oracle
import workloads
from _parity import MAX_ABS, REL_L2
from oracle import layouts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def draw(seed):
    r = np.random.default_rng(1000 + seed)
    d = int(r.choice(la.HEAD_DIMS))
    hkv = int(r.integers(1, 4))
    grp = int(r.choice([1, 2, 4, 8]))
    nq = int(r.choice([1, 1, 1, 2, 3, 4])) if grp * 2 <= 8 else 1
    while grp * nq > 8:
        nq -= 1
    batch = int(r.integers(1, 6))
    lengths = [int(x) for x in np.maximum(nq, np.exp(r.uniform(0, np.log(6000), size=batch)).astype(int))]
    dt = str(r.choice(["f16", "bf16"]))
    layout = str(r.choice(["slab", "slab", "token_major", "paged"]))
    page = int(r.choice([16, 32, 64, 128, 256]))
    if layout == "paged" and d == 80 and grp * nq > 2 and page < 32:
        page = 32  # 32-byte swizzled boxes need pieces of >= 1 KiB
    grid = int(r.choice([0, 0, 1, 3, 17, 64]))
    out_dt = r.choice([torch.float32, torch.float32, torch.float16, torch.bfloat16])
    return d, hkv, grp, nq, lengths, dt, layout, page, grid, out_dt


@pytest.mark.parametrize("seed", range(120))
def test_random_configuration(seed):
    d, hkv, grp, nq, lengths, dt, layout, page, grid, out_dt = draw(seed)
    w = workloads.custom(len(lengths), hkv * grp, hkv, d, dt, lengths, nq=nq)
    q, k, v, cu = workloads.make_inputs(w, seed=seed, device="cuda")
    s = (la.la_plan_spec(w.batch, w.hq, w.hkv, d, nq, cu, grid) if nq > 1
         else la.la_plan(w.batch, w.hq, w.hkv, d, cu, grid))
    ws = la.new_workspace(s)
    out = torch.empty(*q.shape, dtype=out_dt, device="cuda")
    cu_dev = torch.as_tensor(cu, device="cuda")
    if layout == "slab":
        la.la_decode(q, k, v, cu_dev, s, ws, out, w.scale)
        kk, vv = k, v
    elif layout == "token_major":
        kc, vc = workloads.to_token_major(w, k, v)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="token_major")
        kk = layouts.gather_token_major(kc.cpu().view(torch.int16).numpy(), cu, w.hkv, d)
        vv = layouts.gather_token_major(vc.cpu().view(torch.int16).numpy(), cu, w.hkv, d)
    else:
        kc, vc, table, npages = workloads.to_paged(w, k, v, page, seed=seed)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="paged", block_table=table.cuda(),
                        page_size=page, num_pages=npages)
        kk = layouts.gather_paged(kc.cpu().view(torch.int16).numpy(), table.numpy(), cu, page, w.hkv, d)
        vv = layouts.gather_paged(vc.cpu().view(torch.int16).numpy(), table.numpy(), cu, page, w.hkv, d)
    assert la.la_get_status(ws) == la.LA_OK
    if isinstance(kk, torch.Tensor):
        kk, vv = kk.cpu(), vv.cpu()
    else:
        kk, vv = kk.astype(np.int16).view(np.uint16), vv.astype(np.int16).view(np.uint16)
    code = oracle.F16 if dt == "f16" else oracle.BF16
    ref = oracle.attend(q.cpu(), kk, vv, cu, w.hq, w.hkv, d, w.scale, code, nq=nq)
    got = out.double().cpu().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(got))
    if out_dt == torch.float32:
        err = np.abs(got - ref).max()
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert err <= MAX_ABS and rel <= REL_L2, (err, rel)
    else:
        mant = 10 if out_dt == torch.float16 else 7
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - mant)
        assert np.all(np.abs(got - ref) <= MAX_ABS + ulp)


BUILT_HP = {64: [1, 2], 80: [1, 2, 8], 96: [1, 2, 4], 128: [1], 256: [1]}


@pytest.mark.parametrize("seed", range(60))
def test_random_configuration_through_la_plan_kv(seed):
    """Token-major and paged caches through la_plan_kv: a random built count
    of kv heads per unit (or the default), hkv a multiple of it."""
    r = np.random.default_rng(5000 + seed)
    d = int(r.choice(la.HEAD_DIMS))
    hp = int(r.choice(BUILT_HP[d]))
    hkv = hp * int(r.integers(1, 3))
    grp = int(r.choice([1, 2, 4, 8]))
    nq = int(r.choice([1, 1, 2, 3])) if grp * 2 <= 8 else 1
    while grp * nq > 8:
        nq -= 1
    batch = int(r.integers(1, 5))
    lengths = [int(x) for x in np.maximum(nq, np.exp(r.uniform(0, np.log(5000), size=batch)).astype(int))]
    dt = str(r.choice(["f16", "bf16"]))
    layout = str(r.choice(["token_major", "paged"]))
    page = int(r.choice([16, 32, 64, 128, 256]))
    if layout == "paged" and d == 80 and grp * nq > 2 and hp == 1 and page < 32:
        page = 32  # 32-byte swizzled boxes need pieces of >= 1 KiB
    grid = int(r.choice([0, 0, 1, 5, 40]))
    heads = int(r.choice([0, hp]))  # 0: la_plan_kv's default for this shape
    w = workloads.custom(batch, hkv * grp, hkv, d, dt, lengths, nq=nq)
    q, k, v, cu = workloads.make_inputs(w, seed=seed, device="cuda")
    s = la.la_plan_kv(batch, w.hq, hkv, d, cu, nq=nq, heads_per_unit=heads, num_sms=grid)
    if heads:
        assert s.heads_per_unit == hp
    ws = la.new_workspace(s)
    out = torch.empty(*q.shape, dtype=torch.float32, device="cuda")
    cu_dev = torch.as_tensor(cu, device="cuda")
    if layout == "token_major":
        kc, vc = workloads.to_token_major(w, k, v)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="token_major")
        kk = layouts.gather_token_major(kc.cpu().view(torch.int16).numpy(), cu, hkv, d)
        vv = layouts.gather_token_major(vc.cpu().view(torch.int16).numpy(), cu, hkv, d)
    else:
        kc, vc, table, npages = workloads.to_paged(w, k, v, page, seed=seed)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="paged", block_table=table.cuda(),
                        page_size=page, num_pages=npages)
        kk = layouts.gather_paged(kc.cpu().view(torch.int16).numpy(), table.numpy(), cu, page, hkv, d)
        vv = layouts.gather_paged(vc.cpu().view(torch.int16).numpy(), table.numpy(), cu, page, hkv, d)
    assert la.la_get_status(ws) == la.LA_OK
    kk, vv = kk.astype(np.int16).view(np.uint16), vv.astype(np.int16).view(np.uint16)
    code = oracle.F16 if dt == "f16" else oracle.BF16
    ref = oracle.attend(q.cpu(), kk, vv, cu, w.hq, hkv, d, w.scale, code, nq=nq)
    got = out.double().cpu().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)


@pytest.mark.parametrize("seed", range(30))
def test_random_configuration_with_9_to_16_rows(seed):
    """9-16 query rows per kv head (group 16, or a group times several query
    tokens) through la_plan / la_plan_spec / la_plan_kv on every layout."""
    r = np.random.default_rng(9000 + seed)
    d = int(r.choice(la.HEAD_DIMS))
    grp, nq = [(16, 1), (8, 2), (4, 3), (4, 4), (2, 5), (2, 8), (1, 12), (1, 16)][int(r.integers(0, 8))]
    hkv = int(r.integers(1, 3))
    batch = int(r.integers(1, 4))
    lengths = [int(x) for x in np.maximum(nq, np.exp(r.uniform(0, np.log(4000), size=batch)).astype(int))]
    dt = str(r.choice(["f16", "bf16"]))
    layout = str(r.choice(["slab", "token_major", "paged"]))
    page = int(r.choice([32, 64, 128]))
    grid = int(r.choice([0, 0, 3, 29]))
    w = workloads.custom(batch, hkv * grp, hkv, d, dt, lengths, nq=nq)
    q, k, v, cu = workloads.make_inputs(w, seed=seed, device="cuda")
    if layout == "slab":
        s = (la.la_plan_spec(batch, w.hq, hkv, d, nq, cu, grid) if nq > 1
             else la.la_plan(batch, w.hq, hkv, d, cu, grid))
    else:
        s = la.la_plan_kv(batch, w.hq, hkv, d, cu, nq=nq, num_sms=grid)
        assert s.heads_per_unit == 1
    ws = la.new_workspace(s)
    out = torch.empty(*q.shape, dtype=torch.float32, device="cuda")
    cu_dev = torch.as_tensor(cu, device="cuda")
    if layout == "slab":
        la.la_decode(q, k, v, cu_dev, s, ws, out, w.scale)
        kk, vv = k.cpu(), v.cpu()
    elif layout == "token_major":
        kc, vc = workloads.to_token_major(w, k, v)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="token_major")
        kk = layouts.gather_token_major(kc.cpu().view(torch.int16).numpy(), cu, hkv, d)
        vv = layouts.gather_token_major(vc.cpu().view(torch.int16).numpy(), cu, hkv, d)
        kk, vv = kk.astype(np.int16).view(np.uint16), vv.astype(np.int16).view(np.uint16)
    else:
        kc, vc, table, npages = workloads.to_paged(w, k, v, page, seed=seed)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="paged", block_table=table.cuda(),
                        page_size=page, num_pages=npages)
        kk = layouts.gather_paged(kc.cpu().view(torch.int16).numpy(), table.numpy(), cu, page, hkv, d)
        vv = layouts.gather_paged(vc.cpu().view(torch.int16).numpy(), table.numpy(), cu, page, hkv, d)
        kk, vv = kk.astype(np.int16).view(np.uint16), vv.astype(np.int16).view(np.uint16)
    assert la.la_get_status(ws) == la.LA_OK
    code = oracle.F16 if dt == "f16" else oracle.BF16
    ref = oracle.attend(q.cpu(), kk, vv, cu, w.hq, hkv, d, w.scale, code, nq=nq)
    got = out.double().cpu().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)


WIDE = [(17, 1), (20, 1), (24, 1), (32, 1), (40, 1), (48, 1), (64, 1), (96, 1), (128, 1), (130, 1), (256, 1),
        (8, 3), (16, 2), (4, 5), (2, 16), (6, 7), (3, 11)]


@pytest.mark.parametrize("seed", range(40))
def test_random_configuration_with_more_than_16_rows(seed):
    """More than 16 query rows per kv head: units of up to 128 rows on the
    tcgen05 kernel (d = 64, 128) or query blocks, through la_plan,
    la_plan_spec, la_plan_fixed, la_plan_auto and la_plan_kv on every layout."""
    r = np.random.default_rng(13000 + seed)
    d = int(r.choice(la.HEAD_DIMS))
    grp, nq = WIDE[int(r.integers(0, len(WIDE)))]
    hkv = int(r.integers(1, 3))
    batch = int(r.integers(1, 4))
    lengths = [int(x) for x in np.maximum(nq, np.exp(r.uniform(0, np.log(4000), size=batch)).astype(int))]
    dt = str(r.choice(["f16", "bf16"]))
    layout = str(r.choice(["slab", "slab", "token_major", "paged"]))
    page = int(r.choice([16, 32, 64, 128])) if d != 80 else int(r.choice([32, 64, 128]))
    grid = int(r.choice([0, 0, 3, 29]))
    entry = str(r.choice(["plan", "fixed", "auto"])) if (layout == "slab" and nq == 1) else "plan"
    w = workloads.custom(batch, hkv * grp, hkv, d, dt, lengths, nq=nq)
    q, k, v, cu = workloads.make_inputs(w, seed=seed, device="cuda")
    if layout != "slab":
        s = la.la_plan_kv(batch, w.hq, hkv, d, cu, nq=nq, num_sms=grid)
        assert s.heads_per_unit == 1
    elif nq > 1:
        s = la.la_plan_spec(batch, w.hq, hkv, d, nq, cu, grid)
    elif entry == "fixed":
        s = la.la_plan_fixed(batch, w.hq, hkv, d, cu, int(r.integers(1, 5)))
    elif entry == "auto":
        s, _, _ = la.la_plan_auto(batch, w.hq, hkv, d, cu, grid)
    else:
        s = la.la_plan(batch, w.hq, hkv, d, cu, grid)
    ws = la.new_workspace(s)
    out = torch.empty(*q.shape, dtype=torch.float32, device="cuda")
    cu_dev = torch.as_tensor(cu, device="cuda")
    if layout == "slab":
        la.la_decode(q, k, v, cu_dev, s, ws, out, w.scale)
        kk, vv = k.cpu(), v.cpu()
    elif layout == "token_major":
        kc, vc = workloads.to_token_major(w, k, v)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="token_major")
        kk = layouts.gather_token_major(kc.cpu().view(torch.int16).numpy(), cu, hkv, d)
        vv = layouts.gather_token_major(vc.cpu().view(torch.int16).numpy(), cu, hkv, d)
        kk, vv = kk.astype(np.int16).view(np.uint16), vv.astype(np.int16).view(np.uint16)
    else:
        kc, vc, table, npages = workloads.to_paged(w, k, v, page, seed=seed)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="paged", block_table=table.cuda(),
                        page_size=page, num_pages=npages)
        kk = layouts.gather_paged(kc.cpu().view(torch.int16).numpy(), table.numpy(), cu, page, hkv, d)
        vv = layouts.gather_paged(vc.cpu().view(torch.int16).numpy(), table.numpy(), cu, page, hkv, d)
        kk, vv = kk.astype(np.int16).view(np.uint16), vv.astype(np.int16).view(np.uint16)
    assert la.la_get_status(ws) == la.LA_OK
    code = oracle.F16 if dt == "f16" else oracle.BF16
    ref = oracle.attend(q.cpu(), kk, vv, cu, w.hq, hkv, d, w.scale, code, nq=nq)
    got = out.double().cpu().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)
