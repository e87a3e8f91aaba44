"""The 16-row kernel's shared merge of split units, against the float64
oracle. From 4 record rows (query-head groups of 3-16, speculative rows,
units of several kv heads), a unit split into at least 4 pieces whose host
would read at least 96 KiB of peer records is merged by every CTA that
ends on one of its pieces, each an equal share of its rows x d outputs;
smaller merges stay with the host. Cases: units over tens of CTAs and over
every SM, groups 3, 4, 8 and 16, d = 64, 80, 96, 128 and 256, speculative
rows, two kv heads per unit in a token-major cache, ragged tails,
finishers that go on to another unit, two calls on one workspace, 16-bit
outputs, bounded waits that run out, and units left to the host."""
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


def structure(sched):
    """(segments, cta_seg) of a schedule: segments as [unit, t0, t1, kind, peer]."""
    exp = la.la_schedule_export(sched)
    G, U, nseg = exp[1], exp[2], exp[5]
    base = 8 + 2 * (G + 1) + (U + 1)
    segs = [exp[base + 5 * i: base + 5 * i + 5] for i in range(nseg)]
    cta_seg = exp[8 + G + 1 + U + 1: 8 + G + 1 + U + 1 + G + 1]
    return segs, cta_seg


def pieces(sched):
    """Pieces of every split unit: {unit: CTAs host .. finisher}."""
    segs, cta_seg = structure(sched)
    out = {}
    for g in range(len(cta_seg) - 1):
        for s in segs[cta_seg[g]:cta_seg[g + 1]]:
            if s[3] == la.SEG_HOST:
                out[s[0]] = list(range(g, s[4] + 1))
    return out


def shared_units(sched, rows, d):
    """Units merged shared: at least 4 pieces and 96 KiB of peer records
    (records of `rows` rows of d + 4 floats)."""
    return [u for u, c in pieces(sched).items() if len(c) >= 4 and (len(c) - 1) * rows * (d + 4) * 4 >= 96 * 1024]


CASES = [
    # (batch, hq, hkv, d, dtype, lengths, grid, nq, record rows, some unit shared)
    (1, 32, 4, 128, "bf16", [32768], 0, 1, 8, True),          # group 8: units over ~38 CTAs
    (1, 128, 8, 128, "bf16", [32768], 0, 1, 16, True),        # group 16: ~19 CTAs per unit
    (4, 128, 8, 128, "bf16", [8192] * 4, 0, 1, 16, False),    # group 16, 4-5 pieces: the host merges
    (1, 16, 1, 128, "f16", [120000], 0, 1, 16, True),         # one unit over every CTA
    (1, 16, 2, 64, "bf16", [60000], 0, 1, 8, True),           # d 64, group 8
    (1, 16, 2, 80, "f16", [30000], 0, 1, 8, True),            # d 80, group 8
    (1, 32, 2, 96, "bf16", [40000], 0, 1, 16, True),          # d 96, group 16
    (1, 32, 2, 256, "bf16", [20000], 0, 1, 16, True),         # d 256, group 16
    (3, 8, 2, 128, "bf16", [5000, 129, 9000], 0, 2, 8, True),  # 4 query heads x 2 tokens = 8 rows
    (2, 12, 2, 128, "f16", [11000, 4000], 0, 1, 8, True),     # group 6 on the 8-row instance (2 spare rows)
    (4, 16, 2, 128, "bf16", [1, 255, 70000, 130], 0, 1, 8, True),  # ragged tails
    (1, 8, 2, 128, "bf16", [32768], 0, 1, 4, True),           # group 4: records of 4 rows
    (1, 3, 1, 64, "f16", [50000], 0, 1, 4, True),             # group 3, d 64
    (2, 16, 1, 128, "bf16", [4096, 4096], 8, 1, 16, False),   # two units of 4 pieces on 8 CTAs: host
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_shared_merge_matches_the_oracle(case):
    batch, hq, hkv, d, dt, lengths, grid, nq, rows, some_shared = CASES[case]
    w = workloads.custom(batch, hq, hkv, d, dt, lengths, nq=nq)
    q, k, v, _ = workloads.make_inputs(w, seed=91 + case, device="cuda")
    exact = reference(w, q, k, v)
    if nq == 1:
        dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=grid)
        sched = dec.sched
    else:
        sched = la.la_plan_spec(w.batch, w.hq, w.hkv, w.d, nq, w.cu, grid)
    assert bool(shared_units(sched, rows, d)) == some_shared
    ws = la.new_workspace(sched)
    cu = torch.as_tensor(w.cu, dtype=torch.int32, device="cuda")
    for _ in range(2):  # twice: the second call reuses the workspace's flags and records
        out = torch.empty(tuple(q.shape), device="cuda")
        la.la_decode(q, k, v, cu, sched, ws, out, w.scale)
        assert la.la_get_status(ws) == la.LA_OK
        compare(out.cpu(), exact)


def test_two_kv_heads_per_unit_in_a_token_major_cache():
    # d 64, group 4, two kv heads per unit: records of 8 rows
    w = workloads.custom(1, 16, 4, 64, "bf16", [50000])
    q, k, v, cu = workloads.make_inputs(w, seed=5, device="cuda")
    kc, vc = workloads.to_token_major(w, k, v)
    s = la.la_plan_kv(w.batch, w.hq, w.hkv, w.d, w.cu, heads_per_unit=2)
    assert s.heads_per_unit == 2 and shared_units(s, 8, w.d)
    ws = la.new_workspace(s)
    out = torch.empty(w.batch, w.hq, w.d, device="cuda")
    la.la_decode_kv(q, kc, vc, torch.as_tensor(w.cu, device="cuda"), s, ws, out, w.scale, layout="token_major")
    assert la.la_get_status(ws) == la.LA_OK
    code = oracle.BF16
    kk = layouts.gather_token_major(kc.cpu().view(torch.int16).numpy().view(np.uint16), cu, w.hkv, w.d)
    vv = layouts.gather_token_major(vc.cpu().view(torch.int16).numpy().view(np.uint16), cu, w.hkv, w.d)
    ref = oracle.attend(q.cpu(), kk.astype(np.uint16), vv.astype(np.uint16), w.cu, w.hq, w.hkv, w.d, w.scale, code)
    compare(out.cpu(), ref)


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_shared_merge_writes_16_bit_outputs(out_dtype):
    w = workloads.custom(1, 128, 8, 128, "bf16", [30000])
    q, k, v, _ = workloads.make_inputs(w, seed=9, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu)
    o32 = dec(q, k, v, w.scale)
    o16 = torch.empty(tuple(q.shape), dtype=out_dtype, device="cuda")
    la.la_decode(q, k, v, dec.cu_dev, dec.sched, dec.workspace, o16, w.scale)
    assert dec.status() == la.LA_OK
    assert torch.equal(o16, o32.to(out_dtype))


def test_wait_that_runs_out_poisons_the_shares_that_wait_for_it():
    # one unit of 128 LeanTiles (group 16, d 128) over 16 CTAs: every CTA
    # merges one of the 16 query rows. CTA 3 never raises its flag: the
    # other fifteen time out and write NaN; CTA 3's own share (row 3), which
    # needs no flag of its own, is exact
    w = workloads.custom(1, 16, 1, 128, "bf16", [16384])
    q, k, v, _ = workloads.make_inputs(w, seed=6, device="cuda")
    exact = reference(w, q, k, v).reshape(w.hq, w.d)
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=16)
    assert pieces(dec.sched) == {0: list(range(16))} and shared_units(dec.sched, 16, w.d) == [0]
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=3, spin_timeout_ns=50_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_ERR_TIMEOUT
    got = out.cpu().double().numpy().reshape(exact.shape)
    others = [r for r in range(w.hq) if r != 3]
    assert np.isnan(got[others]).all()
    compare(got[3], exact[3])
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=-1, spin_timeout_ns=2_000_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), exact.reshape(w.batch, w.hq, w.d))


def test_small_merges_stay_with_the_host():
    # one unit over 6 CTAs (group 16, 42 KiB of peer records): merged at
    # the host, as before; the host's wait running out poisons the whole unit
    w = workloads.custom(1, 16, 1, 128, "bf16", [6000])
    q, k, v, _ = workloads.make_inputs(w, seed=8, device="cuda")
    exact = reference(w, q, k, v)
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=6)
    assert pieces(dec.sched) == {0: list(range(6))} and not shared_units(dec.sched, 16, w.d)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), exact)
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=1, spin_timeout_ns=50_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_ERR_TIMEOUT
    assert torch.isnan(out).all()
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=-1, spin_timeout_ns=2_000_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), exact)
