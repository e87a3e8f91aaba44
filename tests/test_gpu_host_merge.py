"""The host CTA's reduction of units split over many CTAs, against the
float64 oracle: units over tens of CTAs (small batches and wide query-head
groups on both kernels, so the host stages its peers' records in batches),
a few (long MHA contexts), ragged tails and small grids; two calls on one
workspace; 16-bit outputs; and a bounded wait that runs out."""
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


CASES = [
    # (batch, hq, hkv, d, dtype, lengths, grid)
    (1, 32, 4, 128, "bf16", [32768], 0),             # group 8, 4 units over 152 CTAs: ~37 peers
    (1, 64, 4, 128, "bf16", [20000], 0),             # group 16: several staged batches
    (1, 8, 8, 128, "f16", [40000], 0),               # MHA, 19 CTAs per unit
    (1, 2, 2, 64, "f16", [70000], 0),                # MHA d 64, 76 CTAs per unit: two staged batches
    (2, 64, 1, 128, "bf16", [9000, 23456], 0),       # tcgen05 kernel, 64 rows (lane replicas)
    (1, 128, 1, 64, "bf16", [30000], 0),             # tcgen05 kernel, 128 rows, d 64
    (1, 48, 1, 96, "f16", [17000], 0),               # tcgen05 kernel, 48 rows, d 96
    (5, 32, 4, 64, "bf16", [3000, 17, 20000, 257, 9000], 0),
    (3, 8, 2, 80, "bf16", [5000, 129, 7777], 23),     # d 80, small grid
    (2, 16, 16, 256, "f16", [4000, 2500], 40),        # d 256
    (4, 32, 8, 128, "bf16", [1, 255, 70000, 130], 7),  # ragged tails, 7 CTAs
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_host_merge_matches_the_oracle(case):
    batch, hq, hkv, d, dt, lengths, grid = CASES[case]
    w = workloads.custom(batch, hq, hkv, d, dt, lengths)
    q, k, v, _ = workloads.make_inputs(w, seed=31 + case, device="cuda")
    exact = reference(w, q, k, v)
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=grid)
    for _ in range(2):  # twice: the second call reuses the workspace's flags and records
        out = dec(q, k, v, w.scale)
        assert dec.status() == la.LA_OK
        compare(out.cpu(), exact)


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("shape", [(1, 64, 4, 128), (1, 64, 1, 128)])
def test_host_merge_writes_16_bit_outputs(shape, out_dtype):
    batch, hq, hkv, d = shape
    w = workloads.custom(batch, hq, hkv, d, "bf16", [26000])
    q, k, v, _ = workloads.make_inputs(w, seed=5, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu)
    o32 = dec(q, k, v, w.scale)
    o16 = torch.empty(tuple(q.shape), dtype=out_dtype, device="cuda")
    la.la_decode(q, k, v, dec.cu_dev, dec.sched, dec.workspace, o16, w.scale)
    assert dec.status() == la.LA_OK
    assert torch.equal(o16, o32.to(out_dtype))


def test_wait_that_runs_out_among_many_peers_poisons_only_that_unit():
    # a unit over tens of CTAs (staged merge): one peer never raises its flag
    w = workloads.custom(1, 32, 4, 128, "bf16", [32768])
    q, k, v, _ = workloads.make_inputs(w, seed=4, device="cuda")
    exact = reference(w, q, k, v).reshape(w.hkv, w.hq // w.hkv, w.d)
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu)
    exp = la.la_schedule_export(dec.sched)
    G, U, nseg = exp[1], exp[2], exp[5]
    base = 8 + 2 * (G + 1) + (U + 1)
    segs = [exp[base + 5 * i: base + 5 * i + 5] for i in range(nseg)]
    cta_seg = exp[8 + G + 1 + U + 1: 8 + G + 1 + U + 1 + G + 1]
    unit, fin = next((s[0], s[4]) for g in range(G) for s in segs[cta_seg[g]:cta_seg[g + 1]]
                     if s[3] == la.SEG_HOST and s[4] - g > 10)
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=fin, spin_timeout_ns=50_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_ERR_TIMEOUT
    got = out.cpu().double().numpy().reshape(exact.shape)
    assert np.isnan(got[unit]).all()
    others = [u for u in range(w.hkv) if u != unit]
    assert not np.isnan(got[others]).any()
    compare(got[others], exact[others])
    la.la_schedule_set_debug(dec.sched, skip_signal_cta=-1, spin_timeout_ns=2_000_000_000)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), exact.reshape(-1, w.d))
