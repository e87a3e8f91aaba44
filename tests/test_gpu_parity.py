"""GPU parity: the CUDA library against the float64 oracle on the same
seeded bytes, through the C ABI (tolerances: max-abs 2e-3, rel-L2 1e-3)."""
import numpy as np
import pytest
import torch

import decode_phase_attention_gb300 as la
import workloads
from _parity import compare, reference, run_lean

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def capacity(d, grp):
    per_sm, sms = la.la_device_capacity(d, grp)
    return per_sm * sms


def test_tiny_exact_check_three_ctas_cross_head_boundaries():
    w = workloads.named("tiny")
    q, k, v, _ = workloads.make_inputs(w, seed=0, device="cuda")
    out, dec = run_lean(w, q, k, v, num_sms=3)
    compare(out.cpu(), reference(w, q, k, v))
    exp = la.la_schedule_export(dec.sched)
    assert exp[1] == 3 and exp[3] == 16  # G = 3, I = 16 LeanTiles


SMALL = []
for d in (64, 128):
    for grp in (1, 2, 4, 8):
        for dt in ("f16", "bf16"):
            SMALL.append((d, grp, dt))


@pytest.mark.parametrize("d,grp,dt", SMALL)
@pytest.mark.parametrize("grid", [1, 2, 7, 0])
def test_small_shapes_ragged_tails(d, grp, dt, grid):
    lengths = [1, 255, 257, 1000, 128, 129]
    hkv = 2
    w = workloads.custom(len(lengths), hkv * grp, hkv, d, dt, lengths)
    q, k, v, _ = workloads.make_inputs(w, seed=d + grp, device="cuda")
    out, _ = run_lean(w, q, k, v, num_sms=grid)
    compare(out.cpu(), reference(w, q, k, v))


def test_grid_sweep_up_to_device_capacity():
    w = workloads.custom(3, 8, 4, 128, "bf16", [700, 3000, 129])
    q, k, v, _ = workloads.make_inputs(w, seed=5, device="cuda")
    ref = reference(w, q, k, v)
    cap = capacity(128, 2)
    for G in list(range(1, 40)) + [cap // 2, cap - 1, cap]:
        out, _ = run_lean(w, q, k, v, num_sms=G)
        compare(out.cpu(), ref)


def test_grid_beyond_residency_is_rejected():
    w = workloads.custom(1, 4, 4, 64, "f16", [4096])
    cap = capacity(64, 1)
    s = la.la_plan(1, 4, 4, 64, w.cu, cap + 1)
    q, k, v, _ = workloads.make_inputs(w, device="cuda")
    ws = la.new_workspace(s)
    out = torch.empty(1, 4, 64, device="cuda")
    cu = torch.as_tensor(w.cu, device="cuda")
    with pytest.raises(la.LeanAttentionError) as e:
        la.la_decode(q, k, v, cu, s, ws, out, w.scale)
    assert e.value.status == la.LA_ERR_INVALID


def test_zero_query_gives_the_mean_of_v():
    w = workloads.custom(2, 8, 8, 128, "bf16", [5000, 777])
    q, k, v, _ = workloads.make_inputs(w, seed=1, device="cuda")
    q.zero_()
    out, _ = run_lean(w, q, k, v)
    for b in range(w.batch):
        L, off0 = w.lengths[b], int(w.cu[b]) * w.hkv * w.d
        slab = v[off0:off0 + w.hkv * L * w.d].double().reshape(w.hkv, L, w.d)
        np.testing.assert_allclose(out[b].double().cpu().numpy(), slab.mean(dim=1).cpu().numpy(),
                                   atol=2e-3, rtol=0)


def test_one_hot_scores_select_one_value_row():
    w = workloads.custom(1, 4, 4, 64, "f16", [3000])
    q, k, v, _ = workloads.make_inputs(w, seed=2, device="cuda")
    j = 2345
    kk = k.view(w.hkv, 3000, w.d)
    q.copy_((kk[:, j, :].float() * 4.0).to(q.dtype).view(1, w.hkv, w.d))
    out, _ = run_lean(w, q, k, v, scale=1.0)
    vv = v.view(w.hkv, 3000, w.d)[:, j, :].float()
    torch.testing.assert_close(out[0], vv, atol=2e-3, rtol=0)


@pytest.mark.parametrize("splits", [1, 3, 16])
def test_fixed_partition_baselines(splits):
    w = workloads.custom(4, 16, 4, 128, "bf16", [10000, 300, 4097, 128])
    q, k, v, _ = workloads.make_inputs(w, seed=9, device="cuda")
    out, _ = run_lean(w, q, k, v, fixed_splits=splits)
    compare(out.cpu(), reference(w, q, k, v))


def test_repeated_calls_and_two_schedules_sharing_one_workspace():
    w = workloads.custom(2, 8, 8, 64, "f16", [3000, 5000])
    q, k, v, _ = workloads.make_inputs(w, seed=3, device="cuda")
    ref = reference(w, q, k, v)
    s1 = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, 13)
    s2 = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, 29)
    ws = la.new_workspace(s2)  # the larger of the two
    assert ws.numel() >= la.la_workspace_size(s1)
    cu = torch.as_tensor(w.cu, device="cuda")
    out = torch.empty(w.batch, w.hq, w.d, device="cuda")
    for i in range(12):
        out.fill_(float("nan"))
        la.la_decode(q, k, v, cu, s1 if i % 3 else s2, ws, out, w.scale)
        compare(out.cpu(), ref)
    assert la.la_get_status(ws) == la.LA_OK


# ---- the named workloads, in the launch configuration the benchmark times
@pytest.mark.parametrize("name", ["uniform", "long64k", "long256k", "long512k", "ragged", "gqa"])
def test_named_workloads_full_output(name):
    w = workloads.named(name)
    q, k, v, _ = workloads.make_inputs(w, seed=0, device="cuda")
    out, dec = run_lean(w, q, k, v)
    compare(out.cpu(), reference(w, q, k, v))
    del q, k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("lengths,hq,hkv,d,dt,grid", [
    ([1] * 7, 8, 8, 128, "bf16", 0),          # single-token contexts: every tile is a 1-token tail
    ([300], 1, 1, 64, "f16", 152),            # one head, 2 tiles, 150 idle CTAs
    ([5, 700, 1], 16, 2, 128, "bf16", 3),     # group 8 at d 128 on a 3-CTA grid
    ([256 * 9], 2, 2, 64, "bf16", 9),         # exact tile multiples, one tile per CTA
    ([128 * 40 + 1], 8, 1, 128, "f16", 40),   # MQA (one kv head, group 8)
])
def test_degenerate_shapes(lengths, hq, hkv, d, dt, grid):
    w = workloads.custom(len(lengths), hq, hkv, d, dt, lengths)
    q, k, v, _ = workloads.make_inputs(w, seed=17, device="cuda")
    out, _ = run_lean(w, q, k, v, num_sms=grid)
    compare(out.cpu(), reference(w, q, k, v))


@pytest.mark.parametrize("name", ["tiny", "ragged", "gqa"])
def test_auto_selected_schedule_matches_the_oracle(name):
    w = workloads.named(name)
    q, k, v, _ = workloads.make_inputs(w, seed=2, device="cuda")
    s, kind, pred = la.la_plan_auto(w.batch, w.hq, w.hkv, w.d, w.cu)
    ws = la.new_workspace(s)
    out = torch.empty(w.batch, w.hq, w.d, device="cuda")
    la.la_decode(q, k, v, torch.as_tensor(w.cu, device="cuda"), s, ws, out, w.scale)
    assert la.la_get_status(ws) == la.LA_OK
    compare(out.cpu(), reference(w, q, k, v))


# ---- head dims beyond the LeanTile table, tile sizes, 16-bit outputs
NEW_DIMS = [(d, grp, dt) for d in (80, 96, 256) for grp in (1, 2, 4, 8) for dt in ("f16", "bf16")]


@pytest.mark.parametrize("d,grp,dt", NEW_DIMS)
@pytest.mark.parametrize("grid", [3, 0])
def test_more_head_dims_ragged_tails(d, grp, dt, grid):
    lengths = [1, 63, 65, 1000, 128, 129]
    hkv = 2
    w = workloads.custom(len(lengths), hkv * grp, hkv, d, dt, lengths)
    q, k, v, _ = workloads.make_inputs(w, seed=d * 3 + grp, device="cuda")
    out, _ = run_lean(w, q, k, v, num_sms=grid)
    compare(out.cpu(), reference(w, q, k, v))


@pytest.mark.parametrize("d,T", [(64, 128), (128, 64)])
@pytest.mark.parametrize("grp", [1, 2, 4, 8])
def test_alternative_tile_sizes(d, T, grp):
    lengths = [5000, 1, 200, 3000]
    w = workloads.custom(len(lengths), 2 * grp, 2, d, "bf16", lengths)
    q, k, v, _ = workloads.make_inputs(w, seed=T + grp, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=0, tile_tokens=T)
    assert la.la_schedule_export(dec.sched)[4] == T
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), reference(w, q, k, v))


@pytest.mark.parametrize("out_dt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d,grp", [(128, 1), (64, 8), (96, 4)])
def test_16_bit_outputs_are_the_fp32_result_rounded(out_dt, d, grp):
    w = workloads.custom(3, 2 * grp, 2, d, "bf16", [3000, 17, 9000])
    q, k, v, _ = workloads.make_inputs(w, seed=21, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu)
    out32 = dec(q, k, v, w.scale)
    out16 = torch.empty(w.batch, w.hq, w.d, dtype=out_dt, device="cuda")
    dec(q, k, v, w.scale, out=out16)
    assert dec.status() == la.LA_OK
    assert torch.equal(out16, out32.to(out_dt))  # round to nearest even of the same fp32 values
    ref = reference(w, q, k, v)
    got = out16.double().cpu().numpy().reshape(ref.shape)
    mant = 10 if out_dt == torch.float16 else 7
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - mant)
    assert np.all(np.abs(got - ref) <= 2e-3 + ulp)


@pytest.mark.parametrize("splits", [1, 4])
def test_fixed_split_with_16_bit_output(splits):
    w = workloads.custom(2, 8, 8, 80, "f16", [2000, 700])
    q, k, v, _ = workloads.make_inputs(w, seed=23, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, fixed_splits=splits)
    out32 = dec(q, k, v, w.scale)
    out16 = torch.empty(w.batch, w.hq, w.d, dtype=torch.bfloat16, device="cuda")
    dec(q, k, v, w.scale, out=out16)
    assert torch.equal(out16, out32.to(torch.bfloat16))
    compare(out32.cpu(), reference(w, q, k, v))


@pytest.mark.parametrize("name", ["hd80", "hd96", "hd256", "hd128gqa"])
def test_head_dim_workloads_full_output(name):
    w = workloads.named(name)
    q, k, v, _ = workloads.make_inputs(w, seed=0, device="cuda")
    out, _ = run_lean(w, q, k, v)
    compare(out.cpu(), reference(w, q, k, v))


def test_offsets_beyond_two_to_the_31_elements():
    # 1M-token context, 32 heads, d 128: K alone is 2^32 elements (8.6 GB), so every
    # slab offset past the first half needs 64-bit arithmetic; rows sampled for the oracle
    w = workloads.custom(1, 32, 32, 128, "bf16", [1 << 20])
    q, k, v, _ = workloads.make_inputs(w, seed=29, device="cuda")
    out, _ = run_lean(w, q, k, v)
    rows = np.array([0, 13, 31], np.int64)
    ref = reference(w, q, k, v, rows=rows)
    compare(out.view(32, 128)[rows].cpu(), ref)
    del q, k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("batch,hq,hkv,d,hi", [(4096, 4, 4, 128, 64), (1500, 16, 2, 64, 600), (700, 8, 1, 128, 3000)])
def test_many_short_requests(batch, hq, hkv, d, hi):
    # thousands of units of a few tiles each: most CTAs run long lists of whole units
    lengths = workloads.ragged_lengths(batch, 1, hi, seed=batch, log_uniform=True)
    w = workloads.custom(batch, hq, hkv, d, "bf16", lengths)
    q, k, v, _ = workloads.make_inputs(w, seed=batch, device="cuda")
    out, dec = run_lean(w, q, k, v)
    assert dec.sched.grid > 0
    compare(out.cpu(), reference(w, q, k, v))


@pytest.mark.parametrize("d,grp,T", [(128, 1, 64), (128, 1, 128), (128, 8, 128), (96, 2, 128), (64, 8, 256),
                                     (256, 4, 64)])
def test_ring_depth_does_not_change_the_result(d, grp, T):
    # every warp sees the same tokens in the same order whatever the ring depth
    w = workloads.custom(3, 2 * grp, 2, d, "bf16", [3000, 700, 129])
    q, k, v, _ = workloads.make_inputs(w, seed=d + grp, device="cuda")
    outs = []
    for stages in (0, 2, 3, 4):
        s = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, 0, T)
        la.la_schedule_set_stages(s, stages)
        ws = la.new_workspace(s)
        out = torch.empty(w.batch, w.hq, w.d, device="cuda")
        la.la_decode(q, k, v, torch.as_tensor(w.cu, device="cuda"), s, ws, out, w.scale)
        assert la.la_get_status(ws) == la.LA_OK
        outs.append(out)
    compare(outs[0].cpu(), reference(w, q, k, v))
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("d,T", [(64, 256), (64, 128), (80, 128), (96, 128), (128, 128), (128, 64), (256, 64)])
@pytest.mark.parametrize("grid", [0, 5])
def test_sixteen_query_heads_per_kv_head(d, T, grid):
    # group 16 (two blocks of 8 rows on the tensor-core path) on ragged tails
    w = workloads.custom(4, 32, 2, d, "bf16" if d % 128 else "f16", [1, 255, 257, 1000])
    q, k, v, _ = workloads.make_inputs(w, seed=d + T + grid, device="cuda")
    s = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, grid, T)
    ws = la.new_workspace(s)
    out = torch.empty(w.batch, w.hq, w.d, device="cuda")
    la.la_decode(q, k, v, torch.as_tensor(w.cu, device="cuda"), s, ws, out, w.scale)
    assert la.la_get_status(ws) == la.LA_OK
    compare(out.cpu(), reference(w, q, k, v))


@pytest.mark.parametrize("splits", [1, 3])
def test_sixteen_query_heads_with_fixed_partitions_and_16_bit_output(splits):
    w = workloads.custom(3, 64, 4, 128, "bf16", [3000, 700, 129])
    q, k, v, _ = workloads.make_inputs(w, seed=splits, device="cuda")
    out, _ = run_lean(w, q, k, v, fixed_splits=splits)
    ref = reference(w, q, k, v)
    compare(out.cpu(), ref)
    s = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu)
    ws = la.new_workspace(s)
    o16 = torch.empty(w.batch, w.hq, w.d, dtype=torch.bfloat16, device="cuda")
    la.la_decode(q, k, v, torch.as_tensor(w.cu, device="cuda"), s, ws, o16, w.scale)
    got = o16.double().cpu().numpy().reshape(ref.shape)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    assert np.all(np.abs(got - ref) <= 2e-3 + ulp)


@pytest.mark.parametrize("d,grp", [(64, 3), (128, 5), (128, 6), (96, 7), (80, 12), (256, 3), (64, 14)])
@pytest.mark.parametrize("layout", ["slab", "paged"])
def test_groups_that_are_not_powers_of_two(d, grp, layout):
    # e.g. 28 query over 4 kv heads (group 7) or 40 over 8 (group 5)
    from oracle import layouts
    import oracle
    w = workloads.custom(3, 2 * grp, 2, d, "bf16", [1000, 129, 2500])
    q, k, v, cu = workloads.make_inputs(w, seed=d * grp, device="cuda")
    cu_dev = torch.as_tensor(cu, device="cuda")
    out = torch.empty(w.batch, w.hq, w.d, device="cuda")
    if layout == "slab":
        s = la.la_plan(w.batch, w.hq, w.hkv, w.d, cu, 0)
        ws = la.new_workspace(s)
        la.la_decode(q, k, v, cu_dev, s, ws, out, w.scale)
        ref = reference(w, q, k, v)
    else:
        kc, vc, table, npages = workloads.to_paged(w, k, v, 64, seed=grp)
        s = la.la_plan_kv(w.batch, w.hq, w.hkv, w.d, cu, num_sms=0)
        ws = la.new_workspace(s)
        la.la_decode_kv(q, kc, vc, cu_dev, s, ws, out, w.scale, layout="paged", block_table=table.cuda(),
                        page_size=64, num_pages=npages)
        kk = layouts.gather_paged(kc.cpu().view(torch.int16).numpy(), table.numpy(), cu, 64, w.hkv, w.d)
        vv = layouts.gather_paged(vc.cpu().view(torch.int16).numpy(), table.numpy(), cu, 64, w.hkv, w.d)
        ref = oracle.attend(q.cpu(), kk.astype(np.int16).view(np.uint16), vv.astype(np.int16).view(np.uint16),
                            cu, w.hq, w.hkv, w.d, w.scale, oracle.BF16)
    assert la.la_get_status(ws) == la.LA_OK
    compare(out.cpu(), ref)


@pytest.mark.parametrize("splits", [1, 4])
def test_group_of_five_with_fixed_partitions(splits):
    w = workloads.custom(2, 40, 8, 128, "bf16", [3000, 257])
    q, k, v, _ = workloads.make_inputs(w, seed=5, device="cuda")
    out, _ = run_lean(w, q, k, v, fixed_splits=splits)
    compare(out.cpu(), reference(w, q, k, v))
