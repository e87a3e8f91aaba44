"""Python binding of the LeanAttention decode library (liblean_attn.so).

Argument marshalling only: every step of the computation runs in the CUDA
library behind the C ABI of include/lean_attn.h, under the same names
(la_plan, la_plan_fixed, la_workspace_size, la_workspace_init, la_decode,
la_get_status, la_schedule_export, ...). PyTorch supplies device memory and
streams. There is no CPU fallback: if the shared library is missing the
import fails.
"""
import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblean_attn.so")

LA_OK, LA_ERR_INVALID, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT, LA_ERR_WORKSPACE = range(6)
LA_F16, LA_BF16 = 0, 1
LA_OUT_F32, LA_OUT_F16, LA_OUT_BF16 = 0, 1, 2
HEAD_DIMS = (64, 80, 96, 128, 256)
# built LeanTile sizes; the first is the review's table size (the default, except at
# d = 128 with <= 2 query rows per kv head on the slab layout, where it is 64)
TILE_SIZES = {64: (256, 128), 80: (128,), 96: (128,), 128: (128, 64), 256: (64,)}
SEG_WHOLE, SEG_NONHOST, SEG_HOST, SEG_PARTIAL = range(4)
KV_SLAB, KV_TOKEN_MAJOR, KV_PAGED = range(3)


class KvDesc(ctypes.Structure):
    """la_kv_desc: layout of the K/V caches."""
    _fields_ = [("layout", ctypes.c_int), ("block_table", ctypes.c_void_p), ("max_blocks", ctypes.c_int),
                ("page_size", ctypes.c_int), ("num_pages", ctypes.c_longlong)]
EXPORTED = ["la_plan", "la_plan_ex", "la_plan_spec", "la_plan_kv", "la_plan_fixed", "la_plan_auto", "la_decode_ex", "la_decode_kv", "la_schedule_grid", "la_workspace_size", "la_workspace_init",
            "la_decode", "la_decode_static", "la_decode_host", "la_get_status", "la_schedule_export_size", "la_schedule_export",
            "la_schedule_set_debug", "la_schedule_set_stages", "la_schedule_set_trace", "la_device_capacity",
            "la_schedule_destroy",
            "la_status_string"]


class LeanAttentionError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    c_int, c_size, vp, c_float, c_ll = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float, ctypes.c_longlong
    pp = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "la_plan": (c_int, [c_int, c_int, c_int, c_int, vp, c_int, pp]),
        "la_plan_ex": (c_int, [c_int, c_int, c_int, c_int, vp, c_int, c_int, pp]),
        "la_plan_spec": (c_int, [c_int, c_int, c_int, c_int, c_int, vp, c_int, pp]),
        "la_plan_kv": (c_int, [c_int, c_int, c_int, c_int, c_int, vp, c_int, c_int, c_int, pp]),
        "la_decode_ex": (c_int, [vp, vp, vp, c_int, vp, vp, vp, vp, c_int, c_float, vp]),
        "la_decode_kv": (c_int, [vp, vp, vp, c_int, vp, ctypes.POINTER(KvDesc), vp, vp, vp, c_int, c_float, vp]),
        "la_plan_fixed": (c_int, [c_int, c_int, c_int, c_int, vp, c_int, pp]),
        "la_plan_auto": (c_int, [c_int, c_int, c_int, c_int, vp, c_int, pp, ctypes.POINTER(ctypes.c_double)]),
        "la_schedule_grid": (c_int, [vp]),
        "la_workspace_size": (c_size, [vp]),
        "la_workspace_init": (c_int, [vp, c_size, vp]),
        "la_decode": (c_int, [vp, vp, vp, c_int, vp, vp, vp, vp, c_float, vp]),
        "la_decode_static": (c_int, [vp, vp, vp, c_int, vp, vp, vp, c_float, vp]),
        "la_decode_host": (c_int, [vp, vp, vp, c_int, vp, vp, vp, vp, vp, vp, vp, vp, c_float, vp]),
        "la_get_status": (c_int, [vp, vp]),
        "la_schedule_export_size": (c_size, [vp]),
        "la_schedule_export": (c_int, [vp, vp, c_size]),
        "la_schedule_set_debug": (c_int, [vp, c_int, c_ll]),
        "la_schedule_set_stages": (c_int, [vp, c_int]),
        "la_schedule_set_trace": (c_int, [vp, vp]),
        "la_device_capacity": (c_int, [c_int, c_int, ctypes.POINTER(c_int), ctypes.POINTER(c_int)]),
        "la_schedule_destroy": (None, [vp]),
        "la_status_string": (ctypes.c_char_p, [c_int]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def status_string(status):
    return _lib.la_status_string(int(status)).decode()


def _check(status, what):
    if status != LA_OK:
        raise LeanAttentionError(status, what)


class Schedule:
    """Owns an la_schedule; destroyed with the object."""

    def __init__(self, handle, batch, hq, hkv, d, cu, nq=1):
        self._h = handle
        self.batch, self.hq, self.hkv, self.d = batch, hq, hkv, d
        self.cu = cu
        self.nq = nq
        per_request = la_schedule_export(self)[2] // batch  # units per request: hkv * query_blocks / heads_per_unit
        # kv heads of one unit, and query blocks per kv head (one of the two is 1)
        self.heads_per_unit = max(1, hkv // per_request)
        self.query_blocks = max(1, per_request // hkv)

    @property
    def handle(self):
        return self._h

    @property
    def grid(self):
        return _lib.la_schedule_grid(self._h)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.la_schedule_destroy(h)


def _cu_array(cu_seqlens_k):
    cu = np.ascontiguousarray(np.asarray(cu_seqlens_k, dtype=np.int64))
    if cu.ndim != 1 or cu.size < 2:
        raise ValueError("cu_seqlens_k must be 1-D with batch + 1 entries")
    if cu.min() < 0 or cu.max() > np.iinfo(np.int32).max:
        raise ValueError("cu_seqlens_k out of int32 range")
    return np.ascontiguousarray(cu, dtype=np.int32)


def la_plan(batch, hq, hkv, d, cu_seqlens_k, num_sms=0, tile_tokens=0):
    """Stream-K tile planner; num_sms <= 0 uses one CTA per SM of the current device.

    tile_tokens 0 picks the LeanTile of the head dim (la_plan), else la_plan_ex
    with that LeanTile size.
    """
    cu = _cu_array(cu_seqlens_k)
    if cu.size != batch + 1:
        raise ValueError("cu_seqlens_k must have batch + 1 entries")
    h = ctypes.c_void_p()
    cup = cu.ctypes.data_as(ctypes.c_void_p)
    if tile_tokens:
        _check(_lib.la_plan_ex(batch, hq, hkv, d, cup, int(num_sms), int(tile_tokens), ctypes.byref(h)),
               "la_plan_ex")
    else:
        _check(_lib.la_plan(batch, hq, hkv, d, cup, int(num_sms), ctypes.byref(h)), "la_plan")
    return Schedule(h.value, batch, hq, hkv, d, cu)


def la_plan_spec(batch, hq, hkv, d, nq, cu_seqlens_k, num_sms=0):
    """Stream-K schedule for nq query tokens per request (the last nq tokens of each
    context, causal among themselves); q and out are then [batch, nq, hq, d]."""
    cu = _cu_array(cu_seqlens_k)
    if cu.size != batch + 1:
        raise ValueError("cu_seqlens_k must have batch + 1 entries")
    h = ctypes.c_void_p()
    _check(_lib.la_plan_spec(batch, hq, hkv, d, int(nq), cu.ctypes.data_as(ctypes.c_void_p), int(num_sms),
                             ctypes.byref(h)), "la_plan_spec")
    return Schedule(h.value, batch, hq, hkv, d, cu, nq=int(nq))


def la_plan_kv(batch, hq, hkv, d, cu_seqlens_k, nq=1, heads_per_unit=0, tile_tokens=0, num_sms=0):
    """Stream-K schedule for token-major / paged caches: units of heads_per_unit
    kv heads (0: two when d is 64, 80 or 96 and hkv is even), tile_tokens tokens
    of each head per tile (0: the default), nq query tokens per request."""
    cu = _cu_array(cu_seqlens_k)
    if cu.size != batch + 1:
        raise ValueError("cu_seqlens_k must have batch + 1 entries")
    h = ctypes.c_void_p()
    _check(_lib.la_plan_kv(batch, hq, hkv, d, int(nq), cu.ctypes.data_as(ctypes.c_void_p), int(heads_per_unit),
                           int(tile_tokens), int(num_sms), ctypes.byref(h)), "la_plan_kv")
    return Schedule(h.value, batch, hq, hkv, d, cu, nq=int(nq))


def la_plan_fixed(batch, hq, hkv, d, cu_seqlens_k, splits):
    """Fixed-partition baselines: splits == 1 one CTA per unit, > 1 FlashDecoding-style split."""
    cu = _cu_array(cu_seqlens_k)
    if cu.size != batch + 1:
        raise ValueError("cu_seqlens_k must have batch + 1 entries")
    h = ctypes.c_void_p()
    _check(_lib.la_plan_fixed(batch, hq, hkv, d, cu.ctypes.data_as(ctypes.c_void_p), int(splits),
                              ctypes.byref(h)), "la_plan_fixed")
    return Schedule(h.value, batch, hq, hkv, d, cu)


def la_plan_auto(batch, hq, hkv, d, cu_seqlens_k, num_sms=0):
    """Pick stream-K, one-CTA-per-unit or fixed split by predicted time.

    Returns (schedule, kind, predicted_us) where kind is "lean", "naive" or
    "fixed_split" and predicted_us the three predictions in that order.
    """
    cu = _cu_array(cu_seqlens_k)
    if cu.size != batch + 1:
        raise ValueError("cu_seqlens_k must have batch + 1 entries")
    h = ctypes.c_void_p()
    pred = (ctypes.c_double * 3)()
    _check(_lib.la_plan_auto(batch, hq, hkv, d, cu.ctypes.data_as(ctypes.c_void_p), int(num_sms),
                             ctypes.byref(h), pred), "la_plan_auto")
    sched = Schedule(h.value, batch, hq, hkv, d, cu)
    head = la_schedule_export(sched)[:8]
    kind = "lean" if head[6] == 0 else ("naive" if head[7] == 1 else "fixed_split")
    return sched, kind, list(pred)


def la_workspace_size(sched):
    return int(_lib.la_workspace_size(sched.handle))


def la_schedule_export(sched):
    n = int(_lib.la_schedule_export_size(sched.handle))
    buf = np.zeros(n, dtype=np.int32)
    _check(_lib.la_schedule_export(sched.handle, buf.ctypes.data_as(ctypes.c_void_p), n),
           "la_schedule_export")
    return buf.tolist()


def la_schedule_set_debug(sched, skip_signal_cta=-1, spin_timeout_ns=2_000_000_000):
    _check(_lib.la_schedule_set_debug(sched.handle, int(skip_signal_cta), int(spin_timeout_ns)),
           "la_schedule_set_debug")


def la_schedule_set_stages(sched, stages=0):
    """Ring stages the decode kernel cycles through (0: the library's choice)."""
    _check(_lib.la_schedule_set_stages(sched.handle, int(stages)), "la_schedule_set_stages")


def la_schedule_set_trace(sched, trace=None):
    """Record a per-CTA timeline into `trace` (int64 device tensor of grid*8 words); None stops."""
    if trace is not None and trace.numel() * trace.element_size() < sched.grid * 8 * 8:
        raise ValueError("trace buffer smaller than grid * 8 words")
    ptr = None if trace is None else ctypes.c_void_p(trace.data_ptr())
    _check(_lib.la_schedule_set_trace(sched.handle, ptr), "la_schedule_set_trace")


TRACE_WORDS = 8
TRACE_FIELDS = ["sm", "start", "first_tile", "tiles_done", "wait_ns", "end", "tiles", "segments"]


def la_device_capacity(d, grp):
    per_sm, sms = ctypes.c_int(), ctypes.c_int()
    _check(_lib.la_device_capacity(d, grp, ctypes.byref(per_sm), ctypes.byref(sms)),
           "la_device_capacity")
    return per_sm.value, sms.value


# ---------------------------------------------------------------- torch side
def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def new_workspace(sched, device=None):
    """A zeroed device workspace (uint8 tensor, 256-byte aligned) for a schedule."""
    import torch
    n = la_workspace_size(sched)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def la_workspace_init(workspace, stream=None):
    _check(_lib.la_workspace_init(ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                  _stream_handle(stream)), "la_workspace_init")


def la_decode(q, k, v, cu_seqlens_k, sched, workspace, out, scale, stream=None):
    """Enqueue one decode-attention call (shapes as in include/lean_attn.h)."""
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda and out.is_cuda and cu_seqlens_k.is_cuda
            and workspace.is_cuda):
        raise ValueError("la_decode takes device tensors")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k and v must share one dtype")
    dt = {torch.float16: LA_F16, torch.bfloat16: LA_BF16}.get(q.dtype)
    if dt is None:
        raise ValueError("q, k, v must be float16 or bfloat16")
    out_dt = {torch.float32: LA_OUT_F32, torch.float16: LA_OUT_F16, torch.bfloat16: LA_OUT_BF16}.get(out.dtype)
    if out_dt is None or cu_seqlens_k.dtype != torch.int32:
        raise ValueError("out must be float32, float16 or bfloat16 and cu_seqlens_k int32")
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("cu_seqlens_k", cu_seqlens_k)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    b, hq, hkv, d = sched.batch, sched.hq, sched.hkv, sched.d
    kv_elems = int(sched.cu[-1]) * hkv * d
    if q.numel() != b * sched.nq * hq * d or out.numel() != b * sched.nq * hq * d:
        raise ValueError("q / out do not match the schedule's [batch, nq, hq, d]")
    if k.numel() < kv_elems or v.numel() < kv_elems:
        raise ValueError("k / v are smaller than the schedule's contexts")
    if cu_seqlens_k.numel() != b + 1:
        raise ValueError("cu_seqlens_k does not match the schedule's batch")
    if workspace.numel() * workspace.element_size() < la_workspace_size(sched):
        raise ValueError("workspace smaller than la_workspace_size")
    args = (ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()), dt,
            ctypes.c_void_p(cu_seqlens_k.data_ptr()), sched.handle, ctypes.c_void_p(workspace.data_ptr()),
            ctypes.c_void_p(out.data_ptr()))
    if out_dt == LA_OUT_F32:
        _check(_lib.la_decode(*args, float(scale), _stream_handle(stream)), "la_decode")
    else:
        _check(_lib.la_decode_ex(*args, out_dt, float(scale), _stream_handle(stream)), "la_decode_ex")
    return out


def la_decode_static(q, k, v, cu_seqlens_k, sched, out, scale, stream=None):
    """la_decode without a workspace or any device allocation.

    For callers that cannot allocate device memory (a plugin without access
    to its host program's allocator, or a serving loop whose HBM is all
    reserved up front). The scratch lives in a fixed 4 MiB array inside the
    library that every call shares: do not let two calls overlap on the
    GPU. In-kernel failures show up as NaN outputs (there is no status word).
    """
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda and out.is_cuda and cu_seqlens_k.is_cuda):
        raise ValueError("la_decode_static takes device tensors")
    dt = {torch.float16: LA_F16, torch.bfloat16: LA_BF16}.get(q.dtype)
    if dt is None or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, float16 or bfloat16")
    if out.dtype != torch.float32 or cu_seqlens_k.dtype != torch.int32:
        raise ValueError("out must be float32 and cu_seqlens_k int32")
    b, hq, hkv, d = sched.batch, sched.hq, sched.hkv, sched.d
    kv_elems = int(sched.cu[-1]) * hkv * d
    if not all(t.is_contiguous() for t in (q, k, v, out, cu_seqlens_k)):
        raise ValueError("tensors must be contiguous")
    if (q.numel() != b * sched.nq * hq * d or out.numel() != b * sched.nq * hq * d or k.numel() < kv_elems
            or v.numel() < kv_elems or cu_seqlens_k.numel() != b + 1):
        raise ValueError("tensor sizes do not match the schedule")
    _check(_lib.la_decode_static(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                 ctypes.c_void_p(v.data_ptr()), dt,
                                 ctypes.c_void_p(cu_seqlens_k.data_ptr()), sched.handle,
                                 ctypes.c_void_p(out.data_ptr()), float(scale),
                                 _stream_handle(stream)), "la_decode_static")
    return out


def la_decode_host(q_host, k_host, v_host, cu_seqlens_k, sched, workspace, q_dev, k_dev, v_dev, out_dev,
                   out_host, scale, stream=None):
    """One decode call on host inputs: the library enqueues the copies of q, k, v
    to the device buffers, the decode and the copy of out back to out_host on
    `stream` (no synchronisation). Host tensors should be pinned."""
    import torch
    for name, t, dev in (("q_host", q_host, False), ("k_host", k_host, False), ("v_host", v_host, False),
                         ("out_host", out_host, False), ("q_dev", q_dev, True), ("k_dev", k_dev, True),
                         ("v_dev", v_dev, True), ("out_dev", out_dev, True), ("cu_seqlens_k", cu_seqlens_k, True),
                         ("workspace", workspace, True)):
        if t.is_cuda != dev or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {'device' if dev else 'host'} tensor")
    dt = {torch.float16: LA_F16, torch.bfloat16: LA_BF16}.get(q_host.dtype)
    if dt is None or any(t.dtype != q_host.dtype for t in (k_host, v_host, q_dev, k_dev, v_dev)):
        raise ValueError("q, k, v (host and device) must share one dtype, float16 or bfloat16")
    if out_host.dtype != torch.float32 or out_dev.dtype != torch.float32 or cu_seqlens_k.dtype != torch.int32:
        raise ValueError("out must be float32 and cu_seqlens_k int32")
    b, hq, hkv, d = sched.batch, sched.hq, sched.hkv, sched.d
    n_q = b * sched.nq * hq * d
    kv_elems = int(sched.cu[-1]) * hkv * d
    if any(t.numel() != n_q for t in (q_host, q_dev, out_host, out_dev)) or \
            any(t.numel() < kv_elems for t in (k_host, v_host, k_dev, v_dev)) or cu_seqlens_k.numel() != b + 1:
        raise ValueError("tensor sizes do not match the schedule")
    if workspace.numel() * workspace.element_size() < la_workspace_size(sched):
        raise ValueError("workspace smaller than la_workspace_size")
    vp = ctypes.c_void_p
    _check(_lib.la_decode_host(vp(q_host.data_ptr()), vp(k_host.data_ptr()), vp(v_host.data_ptr()), dt,
                               vp(cu_seqlens_k.data_ptr()), sched.handle, vp(q_dev.data_ptr()),
                               vp(k_dev.data_ptr()), vp(v_dev.data_ptr()), vp(workspace.data_ptr()),
                               vp(out_dev.data_ptr()), vp(out_host.data_ptr()), float(scale),
                               _stream_handle(stream)), "la_decode_host")
    return out_host


def la_decode_kv(q, k_cache, v_cache, cu_seqlens_k, sched, workspace, out, scale, layout="token_major",
                 block_table=None, page_size=0, num_pages=0, stream=None):
    """Decode attention over a token-major ([tokens, hkv, d]) or paged
    ([pages, page_size, hkv, d] + block table) K/V cache."""
    import torch
    code = {"slab": KV_SLAB, "token_major": KV_TOKEN_MAJOR, "paged": KV_PAGED}[layout]
    if not (q.is_cuda and k_cache.is_cuda and v_cache.is_cuda and out.is_cuda and cu_seqlens_k.is_cuda
            and workspace.is_cuda):
        raise ValueError("la_decode_kv takes device tensors")
    dt = {torch.float16: LA_F16, torch.bfloat16: LA_BF16}.get(q.dtype)
    if dt is None or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise ValueError("q and the caches must share one dtype, float16 or bfloat16")
    out_dt = {torch.float32: LA_OUT_F32, torch.float16: LA_OUT_F16, torch.bfloat16: LA_OUT_BF16}.get(out.dtype)
    if out_dt is None or cu_seqlens_k.dtype != torch.int32:
        raise ValueError("out must be float32, float16 or bfloat16 and cu_seqlens_k int32")
    b, hq, hkv, d = sched.batch, sched.hq, sched.hkv, sched.d
    if q.numel() != b * sched.nq * hq * d or out.numel() != b * sched.nq * hq * d \
            or cu_seqlens_k.numel() != b + 1:
        raise ValueError("q / out / cu_seqlens_k do not match the schedule")
    desc = KvDesc(code, None, 0, 0, 0)
    if code == KV_PAGED:
        if block_table is None or not block_table.is_cuda or block_table.dtype != torch.int32 \
                or block_table.dim() != 2 or block_table.shape[0] != b or not block_table.is_contiguous():
            raise ValueError("paged layout needs a contiguous int32 device block table [batch, max_blocks]")
        need = int(num_pages) * int(page_size) * hkv * d
        desc = KvDesc(code, block_table.data_ptr(), block_table.shape[1], int(page_size), int(num_pages))
    else:
        need = int(sched.cu[-1]) * hkv * d
    if k_cache.numel() < need or v_cache.numel() < need:
        raise ValueError("caches are smaller than the layout implies")
    for t in (q, k_cache, v_cache, out, cu_seqlens_k):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if workspace.numel() * workspace.element_size() < la_workspace_size(sched):
        raise ValueError("workspace smaller than la_workspace_size")
    _check(_lib.la_decode_kv(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_cache.data_ptr()),
                             ctypes.c_void_p(v_cache.data_ptr()), dt, ctypes.c_void_p(cu_seqlens_k.data_ptr()),
                             ctypes.byref(desc), sched.handle, ctypes.c_void_p(workspace.data_ptr()),
                             ctypes.c_void_p(out.data_ptr()), out_dt, float(scale), _stream_handle(stream)),
           "la_decode_kv")
    return out


def la_get_status(workspace, stream=None):
    return int(_lib.la_get_status(ctypes.c_void_p(workspace.data_ptr()), _stream_handle(stream)))


class LeanDecoder:
    """Convenience holder: a schedule, its workspace and the device offsets."""

    def __init__(self, batch, hq, hkv, d, cu_seqlens_k, num_sms=0, device="cuda", fixed_splits=None,
                 auto=False, tile_tokens=0, out_dtype=None, nq=1, heads_per_unit=None):
        """heads_per_unit not None: plan with la_plan_kv (token-major / paged caches, 0 = its default)."""
        import torch
        self.predicted_us = None
        self.out_dtype = out_dtype or torch.float32
        self.nq = nq
        if heads_per_unit is not None:
            self.sched = la_plan_kv(batch, hq, hkv, d, cu_seqlens_k, nq, heads_per_unit, tile_tokens, num_sms)
            self.kind = "lean"
        elif nq > 1:
            self.sched, self.kind = la_plan_spec(batch, hq, hkv, d, nq, cu_seqlens_k, num_sms), "lean"
        elif auto:
            self.sched, self.kind, self.predicted_us = la_plan_auto(batch, hq, hkv, d, cu_seqlens_k, num_sms)
        elif fixed_splits is None:
            self.sched = la_plan(batch, hq, hkv, d, cu_seqlens_k, num_sms, tile_tokens)
            self.kind = "lean"
        else:
            self.sched = la_plan_fixed(batch, hq, hkv, d, cu_seqlens_k, fixed_splits)
            self.kind = "naive" if fixed_splits == 1 else "fixed_split"
        self.workspace = new_workspace(self.sched, device)
        self.cu_dev = torch.as_tensor(self.sched.cu, dtype=torch.int32, device=device)
        self.batch, self.hq, self.hkv, self.d = batch, hq, hkv, d

    def __call__(self, q, k, v, scale, out=None, stream=None):
        import torch
        if out is None:
            shape = (self.batch, self.hq, self.d) if self.nq == 1 else (self.batch, self.nq, self.hq, self.d)
            out = torch.empty(*shape, dtype=self.out_dtype, device=q.device)
        return la_decode(q, k, v, self.cu_dev, self.sched, self.workspace, out, scale, stream)

    def status(self, stream=None):
        return la_get_status(self.workspace, stream)
