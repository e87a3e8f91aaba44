"""Helpers for the GPU parity tests: run the library, run the oracle on the
same bytes, compare with the tolerances of the float64 check (max-abs 2e-3
and relative L2 1e-3 for fp16/bf16 inputs with fp32 accumulation)."""
import numpy as np
import torch

import decode_phase_attention_gb300 as la
import oracle

MAX_ABS = 2e-3
REL_L2 = 1e-3


def oracle_code(dtype):
    return {torch.float16: oracle.F16, torch.bfloat16: oracle.BF16}[dtype]


def reference(w, q, k, v, rows=None):
    return oracle.attend(q.cpu(), k.cpu(), v.cpu(), w.cu, w.hq, w.hkv, w.d, w.scale,
                         oracle_code(q.dtype), rows=rows, nq=w.nq)


def compare(got, ref):
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    assert np.all(np.isfinite(got)), "non-finite outputs"
    err = float(np.abs(got - ref).max())
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert err <= MAX_ABS and rel <= REL_L2, f"max-abs {err:.3g}, rel-L2 {rel:.3g}"
    return err, rel


def run_lean(w, q, k, v, num_sms=0, fixed_splits=None, scale=None):
    dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, w.cu, num_sms=num_sms, device=q.device,
                         fixed_splits=fixed_splits)
    out = dec(q, k, v, w.scale if scale is None else scale)
    st = dec.status()
    assert st == la.LA_OK, la.status_string(st)
    return out, dec
