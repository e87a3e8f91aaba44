"""la_decode_host: one call that copies host inputs in, decodes and copies the
output back, all enqueued by the library on one stream. Checked against the
float64 oracle, with pinned and with pageable host buffers, on two calls in
a row that reuse the device buffers."""
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


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("case", ["ragged_gqa", "mha_d128"])
def test_decode_from_host_buffers_matches_the_oracle(case, pinned):
    if case == "ragged_gqa":
        w = workloads.custom(4, 32, 4, 64, "bf16", [3000, 17, 20000, 257])
    else:
        w = workloads.custom(3, 8, 8, 128, "f16", [9000, 129, 4000])
    q, k, v, _ = workloads.make_inputs(w, seed=21, device="cpu")
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    exact = reference(w, q, k, v)
    sched = la.la_plan(w.batch, w.hq, w.hkv, w.d, w.cu, 0)
    ws = la.new_workspace(sched)
    cu = torch.as_tensor(w.cu, dtype=torch.int32, device="cuda")
    qd, kd, vd = (torch.empty_like(t, device="cuda") for t in (q, k, v))
    od = torch.empty(tuple(q.shape), device="cuda")
    stream = torch.cuda.Stream()
    for _ in range(2):
        oh = torch.full(tuple(q.shape), float("nan"))
        if pinned:
            oh = oh.pin_memory()
        la.la_decode_host(q, k, v, cu, sched, ws, qd, kd, vd, od, oh, w.scale, stream=stream)
        stream.synchronize()
        assert la.la_get_status(ws, stream) == la.LA_OK
        compare(oh, exact)
