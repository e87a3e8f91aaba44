"""Stream order with programmatic dependent launches: the decode kernels are
launched so that their CTAs may be placed while the kernel before them on
the stream finishes, and wait for it before touching memory. A kernel that
writes the inputs just before the call, on the same stream and without a
synchronisation, must therefore be seen in full by the call."""
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


@pytest.mark.parametrize("shape", [(2, 32, 32, 128, [20000, 3000]),   # 16-row kernel, CUDA-core path
                                   (2, 64, 8, 128, [9000, 17000]),    # 16-row kernel, tensor-core path
                                   (2, 64, 1, 128, [9000, 17000])])   # tcgen05 kernel
def test_a_kernel_writing_v_just_before_the_call_is_seen(shape):
    batch, hq, hkv, d, lengths = shape
    w = workloads.custom(batch, hq, hkv, d, "bf16", lengths)
    q, k, v, _ = workloads.make_inputs(w, seed=21, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu)
    first = dec(q, k, v, w.scale).clone()
    for step in range(3):
        v.mul_(2.0)  # an elementwise kernel on the same stream, no synchronisation
        out = dec(q, k, v, w.scale)
        torch.cuda.synchronize()
        assert dec.status() == la.LA_OK
        assert torch.equal(out, first * 2.0 ** (step + 1))  # V x 2 scales O exactly


def test_a_kernel_writing_k_and_q_just_before_the_call_is_seen():
    w = workloads.custom(3, 32, 4, 128, "f16", [5000, 700, 12000])
    q, k, v, _ = workloads.make_inputs(w, seed=22, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu)
    dec(q, k, v, w.scale)
    k.neg_()         # two kernels on the stream right before the call
    q.mul_(0.5)
    out = dec(q, k, v, w.scale)
    assert dec.status() == la.LA_OK
    compare(out.cpu(), reference(w, q, k, v))


def test_back_to_back_calls_on_one_workspace_each_see_their_own_inputs():
    w = workloads.custom(1, 8, 8, 128, "bf16", [40000])
    q, k, v, _ = workloads.make_inputs(w, seed=23, device="cuda")
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu)
    qs = [q * s for s in (1.0, -1.0, 0.25, 2.0)]
    outs = [dec(qq, k, v, w.scale).clone() for qq in qs]  # four calls in a row, no synchronisation
    torch.cuda.synchronize()
    assert dec.status() == la.LA_OK
    for qq, o in zip(qs, outs):
        compare(o.cpu(), reference(w, qq, k, v))
