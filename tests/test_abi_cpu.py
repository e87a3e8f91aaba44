"""CPU checks of the C ABI: the library loads, exports every declared
symbol, plans exactly like the reference planner, and rejects bad arguments
before it touches a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import decode_phase_attention_gb300 as la
from oracle import plan as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "lean_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(la.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(la.EXPORTED) == names


def cu_of(lengths):
    return [0] + np.cumsum(lengths).tolist()


def lib_tile(d, rows):
    """The library's default LeanTile on the slab layout: the review's table
    (the reference planner's) for d = 64 and 128, except 64 tokens at d = 128
    with <= 2 query rows; 40-64 KiB tiles for the other head dims."""
    if d in (64, 128):
        return 64 if d == 128 and rows <= 2 else P.lean_tile(d)
    return {80: 128, 96: 128, 256: 64}[d]


@pytest.mark.parametrize("d", la.HEAD_DIMS)
@pytest.mark.parametrize("grp", [1, 2, 4, 8])
def test_default_lean_tile(d, grp):
    expect = {64: 256, 80: 128, 96: 128, 256: 64, 128: 64 if grp <= 2 else 128}[d]
    table = {64: 256, 80: 128, 96: 128, 256: 64, 128: 128}[d]
    assert la.la_schedule_export(la.la_plan(2, 2 * grp, 2, d, [0, 900, 1000], 7))[4] == expect
    # the fixed partitions keep the table's size
    assert la.la_schedule_export(la.la_plan_fixed(2, 2 * grp, 2, d, [0, 900, 1000], 2))[4] == table
    if grp <= 2:  # query rows = group x query tokens decide it
        nq = 8 // grp
        assert la.la_schedule_export(la.la_plan_spec(1, 2 * grp, 2, d, nq, [0, 900], 7))[4] == \
            {64: 256, 80: 128, 96: 128, 256: 64, 128: 128}[d]
    # caches keep the table's size (divided over the kv heads of a unit)
    s = la.la_plan_kv(1, 2 * grp, 2, d, [0, 900], heads_per_unit=1, num_sms=7)
    assert la.la_schedule_export(s)[4] == {64: 256, 80: 128, 96: 128, 256: 64, 128: 128}[d]


def shapes():
    r = np.random.default_rng(123)
    out = [(1, 4, 4, 64, [1024], 3), (8, 32, 32, 128, [8192] * 8, 148), (8, 32, 32, 128, [8192] * 8, 152),
           (1, 32, 32, 128, [65536], 152), (2, 8, 8, 64, [300, 5000], 7)]
    for _ in range(60):
        batch = int(r.integers(1, 6))
        hkv = int(r.integers(1, 5))
        grp = int(r.choice([1, 2, 4, 8]))
        d = int(r.choice([64, 128]))
        lengths = r.integers(1, 3000, size=batch).tolist()
        out.append((batch, hkv * grp, hkv, d, lengths, int(r.integers(1, 200))))
    return out


@pytest.mark.parametrize("shape", shapes())
def test_planner_matches_reference_planner_exactly(shape):
    batch, hq, hkv, d, lengths, G = shape
    s = la.la_plan(batch, hq, hkv, d, cu_of(lengths), G)
    T = lib_tile(d, hq // hkv)
    assert la.la_schedule_export(s) == P.export(P.plan_lean(batch, hq, hkv, d, cu_of(lengths), G, T))
    assert s.grid == G


def test_planner_matches_on_the_ragged_and_gqa_workloads():
    import workloads
    for name in ("ragged", "gqa", "long512k"):
        w = workloads.named(name)
        for G in (148, 152, 304):
            s = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, G)
            T = lib_tile(w.d, w.hq // w.hkv)
            assert la.la_schedule_export(s) == P.export(P.plan_lean(w.batch, w.hq, w.hkv, w.d, w.cu.tolist(), G, T))


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 16])
def test_fixed_planner_matches_reference(splits):
    lengths = [1000, 17, 4096, 129, 8000]
    s = la.la_plan_fixed(5, 8, 2, 128, cu_of(lengths), splits)
    assert la.la_schedule_export(s) == P.export(P.plan_fixed(5, 8, 2, 128, cu_of(lengths), splits, 128))


@pytest.mark.parametrize("args,status", [
    ((1, 6, 4, 64, [0, 10], 4), la.LA_ERR_INVALID),             # hq not a multiple of hkv
    ((2, 4, 4, 64, [0, 10, 10], 4), la.LA_ERR_INVALID),         # empty context
    ((1, 4, 4, 64, [1, 10], 4), la.LA_ERR_INVALID),             # cu[0] != 0
    ((1, 4, 4, 112, [0, 10], 4), la.LA_ERR_UNSUPPORTED),        # head dim not built
])
def test_plan_rejects_bad_shapes(args, status):
    with pytest.raises(la.LeanAttentionError) as e:
        la.la_plan(*args)
    assert e.value.status == status


def test_plan_rejects_empty_batch_and_null_offsets_through_the_c_abi():
    h = ctypes.c_void_p()
    cu = np.array([0], np.int32)
    assert la._lib.la_plan(0, 4, 4, 64, cu.ctypes.data_as(ctypes.c_void_p), 4, ctypes.byref(h)) == la.LA_ERR_INVALID
    assert la._lib.la_plan(1, 4, 4, 64, None, 4, ctypes.byref(h)) == la.LA_ERR_INVALID
    assert la._lib.la_plan(1, 4, 4, 64, cu.ctypes.data_as(ctypes.c_void_p), 4, None) == la.LA_ERR_INVALID
    assert la._lib.la_plan_fixed(1, 4, 4, 64, cu.ctypes.data_as(ctypes.c_void_p), 0, ctypes.byref(h)) == la.LA_ERR_INVALID
    assert not h.value


def test_decode_rejects_bad_pointers_before_any_launch():
    s = la.la_plan(1, 4, 4, 64, [0, 1024], 3)
    lib = la._lib
    vp = ctypes.c_void_p
    good = vp(0x10000)  # never dereferenced: validation fails first
    odd = vp(0x10008)
    ws = vp(0x20000)
    # null inputs
    assert lib.la_decode(None, good, good, 0, good, s.handle, ws, good, 0.125, None) == la.LA_ERR_INVALID
    # misaligned k (bulk copies need 16-byte alignment)
    assert lib.la_decode(good, odd, good, 0, good, s.handle, ws, good, 0.125, None) == la.LA_ERR_INVALID
    # bad dtype
    assert lib.la_decode(good, good, good, 7, good, s.handle, ws, good, 0.125, None) == la.LA_ERR_INVALID
    # NaN scale
    assert lib.la_decode(good, good, good, 0, good, s.handle, ws, good, float("nan"), None) == la.LA_ERR_INVALID
    # missing / misaligned workspace
    assert lib.la_decode(good, good, good, 0, good, s.handle, None, good, 0.125, None) == la.LA_ERR_WORKSPACE
    assert lib.la_decode(good, good, good, 0, good, s.handle, vp(0x20010), good, 0.125, None) == la.LA_ERR_WORKSPACE
    # no schedule
    assert lib.la_decode(good, good, good, 0, good, None, ws, good, 0.125, None) == la.LA_ERR_INVALID


def test_decode_host_rejects_bad_arguments_before_any_copy():
    s = la.la_plan(1, 4, 4, 64, [0, 1024], 3)
    lib = la._lib
    vp = ctypes.c_void_p
    h = vp(0x30000)     # host buffers: never read, validation fails first
    good = vp(0x10000)  # device buffers: never dereferenced
    ws = vp(0x20000)

    def call(qh=h, kh=h, vh=h, dt=0, cu=good, sched=s.handle, qd=good, kd=good, vd=good, w=ws, od=good, oh=h,
             scale=0.125):
        return lib.la_decode_host(qh, kh, vh, dt, cu, sched, qd, kd, vd, w, od, oh, ctypes.c_float(scale), None)

    assert call(qh=None) == la.LA_ERR_INVALID
    assert call(oh=None) == la.LA_ERR_INVALID
    assert call(kd=None) == la.LA_ERR_INVALID
    assert call(vd=vp(0x10008)) == la.LA_ERR_INVALID       # misaligned device buffer
    assert call(cu=vp(0x10002)) == la.LA_ERR_INVALID       # misaligned offsets
    assert call(dt=7) == la.LA_ERR_INVALID
    assert call(scale=float("nan")) == la.LA_ERR_INVALID
    assert call(w=None) == la.LA_ERR_WORKSPACE
    assert call(w=vp(0x20010)) == la.LA_ERR_WORKSPACE
    assert call(sched=None) == la.LA_ERR_INVALID
    two = la.la_plan_kv(1, 4, 4, 64, [0, 1024], heads_per_unit=2, num_sms=3)
    assert call(sched=two.handle) == la.LA_ERR_UNSUPPORTED  # several kv heads per unit: caches only


def test_workspace_size_formula():
    s = la.la_plan(1, 4, 4, 64, [0, 1024], 3)
    # header 256 + flags (3 words padded to 256) + 3 records of 1 row of
    # [m, l, 0, 0, O[64]] (68 floats)
    assert la.la_workspace_size(s) == 256 + 256 + 3 * 68 * 4
    # group 8: records of 8 rows, two slots per CTA (from 4 rows a split unit
    # of enough pieces is merged by every CTA that ends on one of them)
    g = la.la_plan(2, 16, 2, 128, [0, 100, 300], 5)
    assert la.la_workspace_size(g) == 256 + 256 + 2 * 5 * 8 * 132 * 4
    two = la.la_plan(2, 4, 2, 128, [0, 100, 300], 5)  # group 2: one slot per CTA
    assert la.la_workspace_size(two) == 256 + 256 + 5 * 2 * 132 * 4


def test_export_size_and_short_buffer():
    s = la.la_plan(1, 4, 4, 64, [0, 1024], 3)
    n = la._lib.la_schedule_export_size(s.handle)
    buf = (ctypes.c_int32 * n)()
    assert la._lib.la_schedule_export(s.handle, buf, n - 1) == la.LA_ERR_INVALID
    assert la._lib.la_schedule_export(s.handle, buf, n) == la.LA_OK


def test_status_strings():
    for code in range(6):
        assert la.status_string(code)


@pytest.mark.parametrize("shape", shapes()[:25])
def test_auto_plan_is_exactly_one_of_the_explicit_partitions(shape):
    batch, hq, hkv, d, lengths, _ = shape
    cu = cu_of(lengths)
    s, kind, pred = la.la_plan_auto(batch, hq, hkv, d, cu, 152)
    assert len(pred) == 3 and all(p > 0 for p in pred)
    units = batch * hkv
    T = lib_tile(d, hq // hkv)
    explicit = {"lean": P.plan_lean(batch, hq, hkv, d, cu, 152, T),
                "naive": P.plan_fixed(batch, hq, hkv, d, cu, 1),
                "fixed_split": P.plan_fixed(batch, hq, hkv, d, cu, max(2, -(-152 // units)))}
    assert la.la_schedule_export(s) == P.export(explicit[kind])
    idx = ["lean", "naive", "fixed_split"].index(kind)
    assert pred[idx] == min(pred)


def test_auto_plan_prefers_stream_k_when_heads_cannot_fill_the_gpu():
    # measured on GB300: one CTA per head 2.5x and the fixed split 1.37x slower than stream-K
    s, kind, pred = la.la_plan_auto(1, 32, 32, 128, [0, 524288], 152)
    assert kind == "lean" and pred[1] > 2 * pred[0] and pred[2] > 1.25 * pred[0]


def test_auto_plan_charges_a_start_up_for_every_cta_an_sm_runs():
    # 2048 one-tile units on 152 SMs: the same bytes, but one CTA per unit pays
    # 14 start-ups per SM where stream-K pays one
    s, kind, pred = la.la_plan_auto(64, 32, 32, 128, cu_of([128] * 64), 152)
    assert kind == "lean" and pred[1] - pred[0] > 30


def test_auto_plan_prefers_whole_heads_for_a_small_context():
    # 56 heads of 1024 tokens (measured on GB300: 14.0 us whole heads vs 16.1 us stream-K)
    s, kind, pred = la.la_plan_auto(1, 56, 56, 64, [0, 1024], 152)
    assert kind == "naive"


@pytest.mark.parametrize("d", la.HEAD_DIMS)
def test_planner_parity_for_every_head_dim_and_tile_size(d):
    r = np.random.default_rng(d)
    for T in la.TILE_SIZES[d]:
        for _ in range(6):
            batch = int(r.integers(1, 5))
            hkv = int(r.integers(1, 4))
            grp = int(r.choice([1, 2, 4, 8]))
            lengths = r.integers(1, 3000, size=batch).tolist()
            G = int(r.integers(1, 160))
            s = la.la_plan(batch, hkv * grp, hkv, d, cu_of(lengths), G, tile_tokens=T)
            assert la.la_schedule_export(s)[4] == T
            assert la.la_schedule_export(s) == P.export(P.plan_lean(batch, hkv * grp, hkv, d, cu_of(lengths), G, T))
    # the default tile of every head dim (one query row per kv head)
    s = la.la_plan(1, 2, 2, d, [0, 1000], 7)
    assert la.la_schedule_export(s)[4] == lib_tile(d, 1)


@pytest.mark.parametrize("d,T", [(64, 64), (64, 512), (128, 256), (80, 64), (256, 128), (96, 256)])
def test_tile_sizes_that_are_not_built_are_rejected(d, T):
    with pytest.raises(la.LeanAttentionError) as e:
        la.la_plan(1, 2, 2, d, [0, 1000], 7, tile_tokens=T)
    assert e.value.status == la.LA_ERR_UNSUPPORTED


def test_decode_ex_rejects_an_unknown_output_type():
    s = la.la_plan(1, 4, 4, 64, [0, 1024], 3)
    p = ctypes.c_void_p(0x10000)
    assert la._lib.la_decode_ex(p, p, p, 0, p, s.handle, ctypes.c_void_p(0x20000), p, 7, 0.125, None) \
        == la.LA_ERR_INVALID


def test_spec_schedule_matches_the_decode_plan_and_sizes_its_records():
    lengths = [300, 17, 1000]
    s = la.la_plan_spec(3, 4, 2, 128, 3, cu_of(lengths), 11)
    assert s.nq == 3
    assert la.la_schedule_export(s) == P.export(P.plan_lean(3, 4, 2, 128, cu_of(lengths), 11))
    # grp 2 x nq 3 = 6 query rows per unit: records of 8 rows (the instance's
    # row count), two slots per CTA
    assert la.la_workspace_size(s) == 256 + 256 + 2 * 11 * 8 * 132 * 4


@pytest.mark.parametrize("hq,hkv,nq,lengths,status", [
    (4, 4, 129, [200, 300], la.LA_ERR_UNSUPPORTED),  # 129 query tokens: more rows than a unit holds
    (4, 4, 5, [100, 4], la.LA_ERR_INVALID),          # a context shorter than its query tokens
    (4, 4, 0, [100, 200], la.LA_ERR_INVALID),
])
def test_spec_schedule_rejections(hq, hkv, nq, lengths, status):
    with pytest.raises(la.LeanAttentionError) as e:
        la.la_plan_spec(len(lengths), hq, hkv, 64, nq, cu_of(lengths), 7)
    assert e.value.status == status


# ---- la_plan_kv: units of two kv heads for token-major / paged caches
MULTI_HEAD = [(64, 2), (80, 2), (80, 8), (96, 2), (96, 4)]


@pytest.mark.parametrize("d,hp", MULTI_HEAD)
def test_multi_head_units_are_the_reference_plan_over_head_groups(d, hp):
    """A unit of hp kv heads is the reference planner's unit over hkv / hp
    heads with 1/hp of the tokens per tile (the tile keeps its bytes)."""
    r = np.random.default_rng(100 + d + hp)
    T = la.TILE_SIZES[d][0] // hp
    for _ in range(8):
        batch = int(r.integers(1, 5))
        hkv = hp * int(r.integers(1, 4))
        grp = int(r.choice([1, 2, 4, 8]))
        lengths = r.integers(1, 3000, size=batch).tolist()
        G = int(r.integers(1, 160))
        s = la.la_plan_kv(batch, hkv * grp, hkv, d, cu_of(lengths), heads_per_unit=hp, num_sms=G)
        assert s.heads_per_unit == hp
        exp = la.la_schedule_export(s)
        assert exp[2] == batch * hkv // hp and exp[4] == T
        assert exp == P.export(P.plan_lean(batch, (hkv // hp) * grp, hkv // hp, d, cu_of(lengths), G, T))


@pytest.mark.parametrize("d,hkv,hp", [(64, 32, 2), (64, 1, 1), (80, 32, 8), (80, 4, 2), (80, 12, 2), (96, 8, 4),
                                       (96, 6, 2), (96, 3, 1), (128, 8, 1), (256, 4, 1)])
def test_plan_kv_default_heads_per_unit(d, hkv, hp):
    """The default: the fewest kv heads whose rows make whole 256-byte pieces
    (d 64: 2, d 96: 4, d 80: 8); if that does not divide hkv, the most built
    count that does."""
    s = la.la_plan_kv(2, hkv, hkv, d, [0, 1000, 3000], num_sms=7)
    assert s.heads_per_unit == hp


def test_plan_kv_picks_one_head_where_rows_are_long_or_heads_odd():
    assert la.la_plan_kv(1, 8, 8, 128, [0, 1000], num_sms=7).heads_per_unit == 1
    assert la.la_plan_kv(1, 3, 3, 64, [0, 1000], num_sms=7).heads_per_unit == 1
    assert la.la_plan_kv(1, 8, 1, 64, [0, 1000], num_sms=7).heads_per_unit == 1
    s = la.la_plan_kv(2, 8, 8, 64, [0, 1000, 1500], heads_per_unit=1, num_sms=7)
    assert la.la_schedule_export(s) == la.la_schedule_export(la.la_plan(2, 8, 8, 64, [0, 1000, 1500], 7))
    # one head per unit with nq > 1 is la_plan_spec's schedule
    s = la.la_plan_kv(2, 8, 4, 128, [0, 100, 150], nq=3, num_sms=5)
    assert s.nq == 3 and s.heads_per_unit == 1
    assert la.la_schedule_export(s) == la.la_schedule_export(la.la_plan_spec(2, 8, 4, 128, 3, [0, 100, 150], 5))


def test_two_head_records_hold_both_heads():
    # d 64, grp 4, nq 2: 8 query rows per kv head, two kv heads per unit
    s = la.la_plan_kv(2, 16, 4, 64, [0, 300, 700], nq=2, num_sms=9)
    assert s.heads_per_unit == 2
    assert la.la_workspace_size(s) == 256 + 256 + 2 * 9 * 2 * 8 * 68 * 4  # 16 rows: two slots per CTA


@pytest.mark.parametrize("kw,status", [
    (dict(hkv=3, hq=6, heads_per_unit=2), la.LA_ERR_INVALID),     # two does not divide three kv heads
    (dict(hkv=4, hq=8, heads_per_unit=3), la.LA_ERR_INVALID),
    (dict(hkv=4, hq=8, heads_per_unit=8), la.LA_ERR_INVALID),     # eight does not divide four kv heads
    (dict(hkv=16, hq=16, heads_per_unit=16), la.LA_ERR_INVALID),
    (dict(hkv=8, hq=8, heads_per_unit=8), la.LA_ERR_UNSUPPORTED),  # d 64 with 8 heads per unit: not built
    (dict(hkv=8, hq=8, heads_per_unit=4), la.LA_ERR_UNSUPPORTED),  # nor with 4 (no faster than 2)
    (dict(hkv=4, hq=8, heads_per_unit=2, d=128), la.LA_ERR_UNSUPPORTED),   # rows already 256 bytes: not built
    (dict(hkv=4, hq=8, heads_per_unit=2, tile_tokens=256), la.LA_ERR_UNSUPPORTED),
    (dict(hkv=4, hq=8, tile_tokens=-1), la.LA_ERR_INVALID),
    (dict(hkv=2, hq=4, nq=129, cu=[0, 200, 400]), la.LA_ERR_UNSUPPORTED),  # 129 query tokens per request
    (dict(hkv=2, hq=64, heads_per_unit=2), la.LA_ERR_UNSUPPORTED),  # query blocks: one kv head per unit
    (dict(hkv=2, hq=16, nq=2, heads_per_unit=2), la.LA_ERR_UNSUPPORTED),  # 16 rows: one kv head per unit
])
def test_plan_kv_rejections(kw, status):
    args = dict(batch=2, hq=8, hkv=4, d=64, cu=[0, 100, 300], nq=1, heads_per_unit=0, tile_tokens=0)
    args.update(kw)
    with pytest.raises(la.LeanAttentionError) as e:
        la.la_plan_kv(args["batch"], args["hq"], args["hkv"], args["d"], args["cu"], nq=args["nq"],
                      heads_per_unit=args["heads_per_unit"], tile_tokens=args["tile_tokens"], num_sms=7)
    assert e.value.status == status


def test_two_head_schedules_are_refused_for_the_slab_layout():
    s = la.la_plan_kv(1, 4, 4, 64, [0, 1024], num_sms=3)
    assert s.heads_per_unit == 2
    p = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x20000)
    assert la._lib.la_decode(p, p, p, 0, p, s.handle, ws, p, ctypes.c_float(0.125), None) == la.LA_ERR_UNSUPPORTED
    assert la._lib.la_decode_static(p, p, p, 0, p, s.handle, p, ctypes.c_float(0.125), None) \
        == la.LA_ERR_UNSUPPORTED


def test_stage_setter_accepts_zero_and_two_to_four():
    s = la.la_plan(1, 4, 4, 64, [0, 1024], 3)
    for n in (0, 2, 3, 4):
        la.la_schedule_set_stages(s, n)
    for n in (-1, 1, 5):
        with pytest.raises(la.LeanAttentionError) as e:
            la.la_schedule_set_stages(s, n)
        assert e.value.status == la.LA_ERR_INVALID
    assert la._lib.la_schedule_set_stages(None, 2) == la.LA_ERR_INVALID


def test_sixteen_query_rows_per_kv_head():
    # group 16 (and group x query tokens up to 16) plans like any other group
    s = la.la_plan(2, 32, 2, 128, [0, 900, 1000], 7)
    assert la.la_schedule_export(s) == P.export(P.plan_lean(2, 32, 2, 128, [0, 900, 1000], 7, 128))
    # records hold 16 rows of (d + 4) floats, two slots per CTA
    assert la.la_workspace_size(s) == 256 + 256 + 2 * 7 * 16 * 132 * 4
    sp = la.la_plan_spec(2, 16, 2, 64, 2, [0, 900, 1000], 7)
    assert la.la_workspace_size(sp) == 256 + 256 + 2 * 7 * 16 * 68 * 4
    # caches: units of one kv head once a kv head has more than 8 rows
    assert la.la_plan_kv(1, 32, 2, 64, [0, 900], num_sms=7).heads_per_unit == 1
    assert la.la_plan_kv(1, 16, 2, 64, [0, 900], num_sms=7).heads_per_unit == 2


@pytest.mark.parametrize("grp", [3, 5, 6, 7, 9, 12, 15])
def test_groups_that_are_not_powers_of_two(grp):
    # units are still (request, kv head); the instance holds the next power of two rows
    lengths = [700, 64, 3000]
    s = la.la_plan(3, 2 * grp, 2, 128, cu_of(lengths), 11)
    assert la.la_schedule_export(s) == P.export(P.plan_lean(3, 2 * grp, 2, 128, cu_of(lengths), 11, 128))
    R = 4 if grp <= 4 else 8 if grp <= 8 else 16
    slots = 11 if R < 4 else 2 * 11
    assert la.la_workspace_size(s) == 256 + 256 + slots * R * 132 * 4


# ---- query blocks: more query rows per kv head than one unit holds
# (d, group, query tokens) -> (query blocks per kv head, rows of one
# block's instance). A unit holds 128 rows where the tcgen05 kernel is built
# (d = 64, 96, 128), else 16: the fewest equal blocks of whole query heads
# whose rows fit.
QUERY_BLOCKS = [
    (256, 32, 1, 1, 128), (256, 17, 1, 1, 128), (256, 64, 1, 1, 128), (256, 128, 1, 2, 128),
    (256, 96, 1, 2, 128), (256, 200, 1, 4, 128), (256, 65, 1, 5, 16), (256, 2, 40, 2, 128), (256, 8, 3, 1, 128),
    (256, 1, 16, 1, 16), (256, 34, 2, 2, 128), (256, 130, 1, 5, 128),
    (80, 32, 1, 1, 128), (80, 17, 1, 1, 128), (80, 128, 1, 1, 128), (80, 256, 1, 2, 128), (80, 8, 3, 1, 128),
    (80, 1, 16, 1, 16), (80, 2, 100, 2, 128),
    (64, 32, 1, 1, 128), (64, 17, 1, 1, 128), (64, 128, 1, 1, 128), (64, 256, 1, 2, 128), (64, 192, 1, 2, 128),
    (64, 8, 4, 1, 128), (64, 16, 9, 2, 128), (64, 1, 16, 1, 16), (64, 3, 7, 1, 128), (64, 2, 100, 2, 128),
    (128, 16, 1, 1, 16), (128, 64, 1, 1, 128), (128, 130, 1, 2, 128),
]


@pytest.mark.parametrize("d,grp,nq,qb,R", QUERY_BLOCKS)
def test_query_blocks_are_units_of_their_own(d, grp, nq, qb, R):
    # a kv head with more rows than a unit holds becomes qb units, one per
    # block of grp / qb query heads: the schedule is the planner's over
    # hkv * qb heads of grp / qb query heads each
    lengths = [700, 128, 3000]
    hkv, G = 2, 11
    # units of more than 16 rows: 128-token tiles (64 at d = 256); else the head dim's default tile
    T = (64 if d == 256 else 128) if R == 128 else {64: 256, 80: 128, 96: 128, 128: 128, 256: 64}[d]
    s = la.la_plan_spec(3, hkv * grp, hkv, d, nq, cu_of(lengths), G)
    assert s.query_blocks == qb and s.heads_per_unit == 1
    assert la.la_schedule_export(s) == P.export(P.plan_lean(3, hkv * grp, hkv * qb, d, cu_of(lengths), G, T))
    # a record: R rows of [m, l, 0, 0, O[d]] on the 16-row kernel; on the
    # tcgen05 kernel (R = 128) columns over the rows, padded to 16 bytes;
    # two per CTA (with a ready flag each) from 4 rows on
    rec = R * (d + 4) if R < 128 else -(-R * (d + 2) // 4) * 4
    slots = G if R < 4 else 2 * G
    assert la.la_workspace_size(s) == 256 + 256 + slots * rec * 4
    if nq == 1:
        assert la.la_schedule_export(la.la_plan(3, hkv * grp, hkv, d, cu_of(lengths), G)) \
            == la.la_schedule_export(s)
        f = la.la_plan_fixed(3, hkv * grp, hkv, d, cu_of(lengths), 3)
        assert la.la_schedule_export(f) == P.export(P.plan_fixed(3, hkv * grp, hkv * qb, d, cu_of(lengths), 3, T))
    kv = la.la_plan_kv(3, hkv * grp, hkv, d, cu_of(lengths), nq=nq, num_sms=G)
    assert kv.query_blocks == qb and kv.heads_per_unit == 1


def test_query_blocks_of_a_single_kv_head():
    # multi-query attention at d = 256: 128 query heads on one kv head (2 blocks of 64)
    s = la.la_plan(2, 128, 1, 256, [0, 900, 1000], 7)
    assert s.query_blocks == 2
    assert la.la_schedule_export(s) == P.export(P.plan_lean(2, 128, 2, 256, [0, 900, 1000], 7, 64))
    s, kind, _ = la.la_plan_auto(2, 128, 1, 256, [0, 900, 1000], 152)
    assert s.query_blocks == 2
    # at d = 80 and 96 the tcgen05 kernel holds all 128 rows, at d = 256 64
    assert la.la_plan(2, 128, 1, 80, [0, 900, 1000], 7).query_blocks == 1
    assert la.la_plan(2, 128, 1, 96, [0, 900, 1000], 7).query_blocks == 1
    assert la.la_plan(2, 64, 1, 256, [0, 900, 1000], 7).query_blocks == 1
    with pytest.raises(la.LeanAttentionError) as e:
        la.la_plan_kv(1, 64, 1, 80, [0, 900], heads_per_unit=2, num_sms=7)
    assert e.value.status == la.LA_ERR_UNSUPPORTED  # more than 16 rows: one kv head per unit


def test_wide_units_hold_the_whole_group():
    # d = 128: 64 query heads on one kv head are one unit of 64 rows on the
    # 128-row tcgen05 instance, with 128-token tiles
    s = la.la_plan(2, 64, 1, 128, [0, 900, 1000], 7)
    assert s.query_blocks == 1
    assert la.la_schedule_export(s) == P.export(P.plan_lean(2, 64, 1, 128, [0, 900, 1000], 7, 128))
    assert la.la_workspace_size(s) == 256 + 256 + 2 * 7 * 128 * 130 * 4  # two record slots per CTA
    assert la.la_schedule_export(la.la_plan(2, 64, 1, 64, [0, 900, 1000], 7))[4] == 128
    for bad in (64, 256):  # the wide instance is built for 128-token tiles only
        with pytest.raises(la.LeanAttentionError) as e:
            la.la_plan(2, 64, 1, 64, [0, 900, 1000], 7, tile_tokens=bad)
        assert e.value.status == la.LA_ERR_UNSUPPORTED
    with pytest.raises(la.LeanAttentionError) as e:
        la.la_plan_spec(1, 4, 4, 64, 129, [0, 1000], 7)  # 129 query tokens: more than a unit holds
    assert e.value.status == la.LA_ERR_UNSUPPORTED


def test_partition_choice_for_wide_units():
    # one unit over every SM: its 152 CTAs share the merge, so stream-K
    # still wins over the fixed split; 16 units: stream-K
    s, kind, pred = la.la_plan_auto(1, 64, 1, 128, [0, 262144], 152)
    assert kind == "lean" and pred[0] < pred[2] < pred[1]
    s, kind, pred = la.la_plan_auto(16, 64, 1, 128, cu_of([32768] * 16), 152)
    assert kind == "lean" and pred[0] < pred[2] < pred[1]


def test_unit_counts_beyond_32_bits_are_rejected():
    # a million requests of 4096 query heads: more query rows than the
    # planner counts in 32 bits
    with pytest.raises(la.LeanAttentionError) as e:
        la.la_plan(1 << 20, 4096, 1, 64, np.arange((1 << 20) + 1, dtype=np.int32), 7)
    assert e.value.status == la.LA_ERR_UNSUPPORTED


def _structure(exp):
    """(G, U, segments, cta_seg, unit_host, unit_fin) from a schedule export."""
    G, U, nseg = exp[1], exp[2], exp[5]
    base = 8 + 2 * (G + 1) + (U + 1)
    segs = [exp[base + 5 * i: base + 5 * i + 5] for i in range(nseg)]
    cta_seg = exp[8 + G + 1 + U + 1: 8 + G + 1 + U + 1 + G + 1]
    rest = base + 5 * nseg
    return G, U, segs, cta_seg, exp[rest: rest + U], exp[rest + U: rest + 2 * U]


@pytest.mark.parametrize("seed", range(6))
def test_split_units_of_wide_schedules_have_the_shape_the_shared_merge_needs(seed):
    # The tcgen05 kernel merges a split unit on every CTA whose last segment
    # is a piece of it, and a CTA keeps at most two records (its first
    # segment's, its last segment's). Both rest on the stream-K structure:
    # a host piece is its CTA's last segment, the CTAs between host and
    # finisher hold only that unit, the finisher's piece is its first segment,
    # and no split piece sits between a CTA's first and last segments.
    rng = np.random.default_rng(seed)
    batch = int(rng.integers(1, 6))
    lengths = rng.integers(1, 40000, size=batch).tolist()
    grp = int(rng.choice([32, 48, 64, 128]))
    hkv = int(rng.integers(1, 3))
    d = int(rng.choice([64, 80, 96, 128]))
    G = int(rng.choice([5, 19, 64, 152]))
    s = la.la_plan(batch, grp * hkv, hkv, d, cu_of(lengths), G)
    G, U, segs, cta_seg, host, fin = _structure(la.la_schedule_export(s))
    split = {P.HOST, P.NONHOST}
    merges = {}
    for g in range(G):
        mine = segs[cta_seg[g]:cta_seg[g + 1]]
        for i, sg in enumerate(mine):
            if sg[3] in split:
                assert i == 0 or i == len(mine) - 1  # only a first or last segment is a split piece
            if sg[3] == P.HOST:
                assert i == len(mine) - 1 and host[sg[0]] == g
        if mine and mine[-1][3] in split:
            merges.setdefault(mine[-1][0], []).append(g)  # this CTA merges a share of that unit
    for u in range(U):
        h0, h1 = host[u], fin[u]
        if h0 == h1:
            assert u not in merges  # a whole unit
            continue
        for c in range(h0 + 1, h1):  # the CTAs between hold only this unit
            assert cta_seg[c + 1] - cta_seg[c] == 1 and segs[cta_seg[c]][0] == u
        assert segs[cta_seg[h1]][0] == u and segs[cta_seg[h1]][3] == P.NONHOST  # the finisher's first segment
        fin_only = cta_seg[h1 + 1] - cta_seg[h1] == 1
        assert merges[u] == list(range(h0, h1 + (1 if fin_only else 0)))
