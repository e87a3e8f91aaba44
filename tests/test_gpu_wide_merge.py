"""The tcgen05 kernel's merge of split units, against the float64 oracle.
Every piece of a split unit writes a record and each CTA that ends on a
piece of the unit merges an equal share of its rows x d outputs: one unit
over every SM (a share of a few dozen outputs, several threads per output),
17 rows (a handful of outputs per share), the 128-row instance, d = 256,
finishers whose piece is their only segment (they merge a share too),
units split over two CTAs whose finisher goes on to another unit (the host
merges alone, from registers), two calls on one workspace, and bounded
waits that run out in both kinds of merge."""
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


def structure(sched):
    """(segments, cta_seg) of a schedule: segments as [unit, t0, t1, kind, peer]."""
    exp = la.la_schedule_export(sched)
    G, U, nseg = exp[1], exp[2], exp[5]
    base = 8 + 2 * (G + 1) + (U + 1)
    segs = [exp[base + 5 * i: base + 5 * i + 5] for i in range(nseg)]
    cta_seg = exp[8 + G + 1 + U + 1: 8 + G + 1 + U + 1 + G + 1]
    return segs, cta_seg


def merging_ctas(sched, unit):
    """CTAs whose last segment is a piece of a split unit."""
    segs, cta_seg = structure(sched)
    out = []
    for g in range(len(cta_seg) - 1):
        last = segs[cta_seg[g + 1] - 1]
        if last[0] == unit and last[3] in (la.SEG_HOST, la.SEG_NONHOST):
            out.append(g)
    return out


CASES = [
    # (batch, hq, hkv, d, dtype, lengths, grid)
    (1, 64, 1, 128, "bf16", [40000], 0),        # one unit over every CTA, 64 rows
    (1, 17, 1, 64, "f16", [50000], 0),          # 17 rows: a few outputs per CTA
    (1, 128, 1, 80, "bf16", [20000], 0),        # the 128-row instance
    (1, 64, 1, 256, "bf16", [12000], 0),        # d = 256, 64-token tiles
    (1, 100, 1, 96, "f16", [9000], 0),          # 100 rows, d 96
    (4, 32, 1, 128, "bf16", [5000, 3000, 7000, 100], 7),  # units over two or three CTAs
    (3, 48, 2, 64, "bf16", [777, 4096, 2000], 19),
    (1, 128, 1, 128, "bf16", [200000], 0),      # 128 rows over every CTA: the most shared memory a merge takes
    (1, 64, 1, 256, "f16", [60000], 0),         # d = 256 over every CTA
    (1, 128, 1, 80, "bf16", [100000], 0),       # d = 80, 128 rows over every CTA
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_split_units_match_the_oracle(case):
    batch, hq, hkv, d, dt, lengths, grid = CASES[case]
    w = workloads.custom(batch, hq, hkv, d, dt, lengths)
    q, k, v, _ = workloads.make_inputs(w, seed=71 + case, device="cuda")
    exact = reference(w, q, k, v)
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=grid)
    for _ in range(2):  # twice: the second call reuses the workspace's flags and records
        out = dec(q, k, v, w.scale)
        assert dec.status() == la.LA_OK
        compare(out.cpu(), exact)


@pytest.mark.parametrize("grid", [4, 8])
def test_finisher_whose_piece_is_its_only_segment_merges_a_share(grid):
    # two units of 32 LeanTiles over 4 or 8 CTAs: every CTA range ends on a
    # unit boundary or inside one, so each unit's finisher holds nothing else
    w = workloads.custom(2, 64, 1, 128, "bf16", [4096, 4096])
    q, k, v, _ = workloads.make_inputs(w, seed=5, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=grid)
    segs, cta_seg = structure(dec.sched)
    fin = next(s[4] for s in segs if s[0] == 0 and s[3] == la.SEG_HOST)
    assert cta_seg[fin + 1] - cta_seg[fin] == 1
    assert merging_ctas(dec.sched, 0) == list(range(grid // 2))  # host, the CTAs between, the finisher
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), reference(w, q, k, v))


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_merged_shares_write_16_bit_outputs(out_dtype):
    w = workloads.custom(1, 48, 1, 128, "bf16", [30000])
    q, k, v, _ = workloads.make_inputs(w, seed=9, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu)
    o32 = dec(q, k, v, w.scale)
    o16 = torch.empty(tuple(q.shape), dtype=out_dtype, device="cuda")
    la.la_decode(q, k, v, dec.cu_dev, dec.sched, dec.workspace, o16, w.scale)
    assert dec.status() == la.LA_OK
    assert torch.equal(o16, o32.to(out_dtype))


def test_wait_that_runs_out_poisons_only_that_unit():
    # unit 0 over CTAs 0-3 of 8, its finisher (CTA 3) never raises its flag:
    # the CTAs merging with it time out and write NaN; CTA 3's own share,
    # which needs no flag of its own, is exact; unit 1 is untouched
    w = workloads.custom(2, 64, 1, 128, "bf16", [4096, 4096])
    q, k, v, _ = workloads.make_inputs(w, seed=6, device="cuda")
    exact = reference(w, q, k, v).reshape(w.batch, w.hq, w.d)
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=8)
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=3, spin_timeout_ns=50_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_ERR_TIMEOUT
    got = out.cpu().double().numpy().reshape(exact.shape)
    # shares are ranges of e = dim * rows + row over 4 CTAs: dims 0-95 NaN, 96-127 exact
    assert np.isnan(got[0, :, :96]).all()
    compare(got[0, :, 96:], exact[0, :, 96:])
    compare(got[1], exact[1])
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=-1, spin_timeout_ns=2_000_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), exact.reshape(w.batch, w.hq, w.d))


def test_sole_host_merges_alone_and_times_out_alone():
    # two units of 32 LeanTiles over 3 CTAs (22, 21, 21 tiles): unit 0 is
    # CTA 0's and CTA 1's first segment, so CTA 0 merges it alone; unit 1 is
    # CTA 1's last segment and CTA 2's only one, so both merge a share
    w = workloads.custom(2, 64, 1, 128, "bf16", [4096, 4096])
    q, k, v, _ = workloads.make_inputs(w, seed=7, device="cuda")
    exact = reference(w, q, k, v).reshape(w.batch, w.hq, w.d)
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=3)
    segs, cta_seg = structure(dec.sched)
    assert [segs[cta_seg[g]][3] for g in range(3)] == [la.SEG_HOST, la.SEG_NONHOST, la.SEG_NONHOST]
    assert merging_ctas(dec.sched, 0) == [0] and merging_ctas(dec.sched, 1) == [1, 2]
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), exact)
    # CTA 1 never raises the flag of its first segment (unit 0's tail)
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=1, spin_timeout_ns=50_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_ERR_TIMEOUT
    got = out.cpu().double().numpy().reshape(exact.shape)
    assert np.isnan(got[0]).all()
    compare(got[1], exact[1])
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=-1, spin_timeout_ns=2_000_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), exact)
