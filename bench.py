"""Benchmark: LeanAttention stream-K decode attention on GB300.

One step is one decode-attention call over one batch: the LeanTile loop,
the partial exchange, the host-CTA reduction and the normalisation, all in
one launch of the library's kernel (the schedule is planned once for the
batch, outside the timed region; its host time is reported as plan_us).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--kernel lean|naive|fixed_split|auto] [--impl ours|reference]

The headline workload is the 512k-token context (batch 1, 32/32 heads,
d 128, fp16: 8.6 GB of K+V), the largest of the decode configurations.
value = K+V bytes read / kernel time, summed over ranks (GB/s); the kernel
time is taken with CUDA events on the launching stream around the K timed
back-to-back calls, which follow the warm-up calls with no idle gap (only
the synchronisation the contract asks for). The same JSON line carries, as
nested records measured the same way in the same process, the ragged batch,
the uniform batch, the 64k and 256k contexts and the grouped-query batch,
the headline at the LeanTile table's 128-token tile, and the two fixed
partitions (one CTA per unit; fixed split plus merge launch) as ablations.
Inputs larger than 4x L2 are not flushed between calls (the next call
cannot hit in L2); smaller ones get a 256 MiB write before every call.
e2e = the same metric through la_decode_host: q, K, V copied from pinned
host memory, the decode, and the output copied back, inside every timed
step. --impl reference times the float64 CPU oracle instead. Under torchrun
every rank runs an independent replica (the path has no cross-GPU exchange)
and the slowest rank's time is reported.
"""
import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention µs/call and KV-read GB/s as % of GB300 HBM peak, 1 GPU"
FLUSH_BYTES = 256 << 20
L2_BYTES = 129 * 10**6
NOMINAL_HBM_GBS = 8000.0
HEADLINE = "long512k"
# the other decode configurations, measured in the same run as nested records
EXTRA_WORKLOADS = ["ragged", "uniform", "long64k", "long256k", "gqa"]
EXTRA_STEPS_MAX = 200   # timed calls of a nested record: min(K, this)
SETTLE_SECONDS = 0.1    # warm-up calls go on until at least this much GPU time


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--kernel", default="lean", choices=["lean", "naive", "fixed_split", "auto"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--grid", type=int, default=0, help="stream-K grid; 0 = one CTA per SM")
    ap.add_argument("--tile", type=int, default=0, help="LeanTile tokens; 0 = the head dim's default")
    ap.add_argument("--out-dtype", default="f32", choices=["f32", "f16", "bf16"])
    ap.add_argument("--kv-layout", default="slab", choices=["slab", "token_major", "paged"])
    ap.add_argument("--page-size", type=int, default=64)
    ap.add_argument("--stages", type=int, default=0, help="ring stages (0: the library's choice)")
    ap.add_argument("--heads-per-unit", type=int, default=0,
                    help="token-major / paged caches: kv heads per unit (0 = la_plan_kv's choice)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--flush", action="store_true", help="flush L2 before every timed call")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="headline only: no nested workloads, table tile or ablations")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def _code_only(text):
    """Source text without comments and with whitespace collapsed."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_digest(kernel="lean_decode_kernel", csrc=None):
    """Digest of one decode kernel's device code (its template, the shared
    helpers and producer, its parameters and instances), comments and layout
    ignored: a profile stays valid across edits that change no code of the
    kernel it measured."""
    if kernel == "lean_wide_kernel":
        keep = lambda f: f in ("la_wide.cuh", "la_kernel.cuh", "la_internal.h", "la_kernels_wide.cu")
    else:
        keep = lambda f: (f in ("la_kernel.cuh", "la_internal.h") or
                          (f.startswith("la_kernels_d") and f.endswith(".cu")))
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "decode_phase_attention_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if keep(f):
            h.update(f.encode())
            h.update(_code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def decode_kernel_name(w, sched):
    """The stream-K kernel a schedule runs: the tcgen05 one for units of more
    than 16 query rows, else the 16-row one."""
    rows = w.hq // w.hkv // sched.query_blocks * w.nq
    return "lean_wide_kernel" if rows > 16 else "lean_decode_kernel"


def profile_name(workload, kv_layout="slab", page_size=0, kernel="lean_decode_kernel"):
    """Name of the committed ncu summary of a stream-K kernel on a workload and cache layout."""
    suffix = "" if kv_layout == "slab" else ("_token_major" if kv_layout == "token_major" else f"_paged{page_size}")
    return f"{kernel}_{workload}{suffix}"


def profiled_traffic(name, d, tile):
    """DRAM bytes per launch from the committed ncu summary, if it is for this
    kernel source and this kernel instance (head dim, LeanTile)."""
    path = os.path.join(ROOT, "profiles", f"{name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    src = re.search(r"kernel_source_digest:\s*([0-9a-f]+)", text)
    tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    inst = re.search(r"lean_decode_kernel<(\d+), (\d+),", text)
    wide = re.search(r"lean_wide_kernel<(\d+),", text)
    if not src or not tr or not (inst or wide):
        return None
    kernel = "lean_wide_kernel" if wide else "lean_decode_kernel"
    if src.group(1) != kernel_source_digest(kernel):
        return None
    shape = (int(wide.group(1)), 128) if wide else (int(inst.group(1)), int(inst.group(2)))
    if shape != (d, tile):
        return None
    return int(tr.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, interval_ms=20):
        self.index = index
        self.interval_ms = interval_ms
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _rows(self, t0, t1):
        rows = []
        for ts, line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10 and t0 <= ts <= t1:
                rows.append(parts)
        return rows

    @staticmethod
    def _stats(rows):
        mhz = sorted(float(p[2]) for p in rows if p[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for p in rows:
            for n, val in zip(names, p[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        watts = [float(p[4]) for p in rows if p[4].replace(".", "").isdigit()]
        return {"sm_mhz": mhz[len(mhz) // 2] if mhz else None,
                "sm_max_mhz": float(rows[0][3]) if rows and rows[0][3].replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(watts) if watts else None}

    def summary(self, load0, t0, t1):
        """Clocks over [t0, t1] (the timed region, wall clock) and over the
        loaded window [load0, t1] (warm-up and timed calls back to back).
        The top-level figures are the timed region's when a sample fell
        inside it, else the loaded window's."""
        if self.proc is None:
            return None
        inside = self._stats(self._rows(t0, t1 + 0.03))
        loaded = self._stats(self._rows(load0, t1 + 0.03))
        if not loaded["samples"]:
            return None
        top = dict(inside if inside["samples"] else loaded)
        top["in_timed_region"] = bool(inside["samples"])
        top["timed_region"] = inside
        top["warmup_and_timed"] = loaded
        return top


def max_over_ranks(x, device=None):
    """The slowest rank's value (every rank runs an independent replica)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def summarize_trace(tr):
    """Per-CTA timeline of one call: balance of busy time and host-CTA waits (microseconds)."""
    import numpy as np
    t0 = tr[:, 1].min()
    busy = (tr[:, 3] - tr[:, 1]) / 1e3
    end = (tr[:, 5] - t0) / 1e3
    first = (tr[:, 2] - tr[:, 1]) / 1e3
    wait = tr[:, 4] / 1e3
    active = tr[:, 6] > 0

    def stats(x):
        x = x[active]
        return {"min": round(float(x.min()), 2), "mean": round(float(x.mean()), 2),
                "max": round(float(x.max()), 2)}
    return {"ctas": int(active.sum()), "tile_loop_us": stats(busy), "end_us": stats(end),
            "first_tile_latency_us": stats(first), "host_wait_us": stats(wait),
            "tiles_per_cta": stats(tr[:, 6].astype(float)),
            "launch_skew_us": round(float((tr[active, 1].max() - t0) / 1e3), 2)}


def algorithmic_bytes(w, export, out_bytes=4):
    """Bytes a call must move: K+V once, q, out, and every partial record
    written once and read once (one per non-host or fixed-split piece)."""
    kv = w.kv_bytes()
    q = w.batch * w.nq * w.hq * w.d * 2
    out = w.batch * w.nq * w.hq * w.d * out_bytes
    G, U, nseg = export[1], export[2], export[5]
    base = 8 + 2 * (G + 1) + (U + 1)
    pieces = sum(1 for i in range(nseg) if export[base + 5 * i + 3] in (1, 3))
    rows = w.batch * w.nq * w.hq // U  # query rows of a unit (all its kv heads, or one query block)
    rec = rows * (w.d + 2) * 4
    return kv, kv + q + out + 2 * pieces * rec


def uses_flush(w, args):
    """Inputs under 4x L2 get an L2 flush before every timed call."""
    return args.flush or w.kv_bytes() < L2_BYTES * 4


def workload_config(w, args):
    """The workload a line measures: the same dict in both arms."""
    kv = w.kv_bytes()
    return {"workload": w.description, "name": w.name, "batch": w.batch, "hq": w.hq, "hkv": w.hkv,
            "head_dim": w.d, "query_tokens": w.nq, "dtype": w.dtype,
            "total_context_tokens": w.total_tokens, "kv_bytes": kv, "seed": args.seed,
            "l2": ("flushed before every timed call (256 MiB write, then 256 MiB read so no dirty line "
                   "is written back inside the call)" if uses_flush(w, args) else
                   f"no flush: K+V ({kv / 1e9:.2f} GB) exceed 4x the 129 MB L2, so no call finds its "
                   f"inputs in L2")}


def row_bytes_of(w, cu):
    """K+V bytes attributed to each (request, query token, query head) row:
    its kv head's K and V shared over the rows that read them."""
    import numpy as np
    nrows = w.batch * w.nq * w.hq  # row r = (b * nq + i) * hq + h
    rows_per_kv = (w.hq // w.hkv) * w.nq
    return np.array([2 * (cu[r // (w.nq * w.hq) + 1] - cu[r // (w.nq * w.hq)]) * w.d * 2 / rows_per_kv
                     for r in range(nrows)])


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    import workloads

    w = workloads.named(args.workload, seed=args.seed)
    q, k, v, cu = workloads.make_inputs(w, seed=args.seed, device="cpu")
    code = {"f16": oracle.F16, "bf16": oracle.BF16}[w.dtype]
    cores = os.cpu_count() or 1
    nrows = w.batch * w.nq * w.hq
    row_bytes = row_bytes_of(w, cu)
    per_step = cores
    qn, kn, vn = (t.view(torch.int16).numpy().view(np.uint16) for t in (q, k, v))
    pos = 0

    def step():
        nonlocal pos
        rows = np.array([(pos + i) % nrows for i in range(per_step)], dtype=np.int64)
        pos = (pos + per_step) % nrows
        oracle.attend(qn, kn, vn, cu, w.hq, w.hkv, w.d, w.scale, code, rows=rows, threads=cores, nq=w.nq)
        return float(row_bytes[rows].sum())

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    total = 0.0
    for _ in range(args.steps):
        total += step()
    dt = time.perf_counter() - t0
    gbs = total / dt / 1e9
    sample = (f"{per_step} (request, query, head) rows per step, cycling over the {nrows} rows of the "
              f"workload; float64 two-pass softmax over the exact {w.dtype} inputs")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w, q, k, v, cu, seconds, single_seconds=2.0):
    """The float64 oracle on the host cores over the workload's rows, cycled,
    for about `seconds`; then the same with one thread for `single_seconds`.
    q, k, v are host tensors (the pinned copies the e2e leg reads)."""
    import numpy as np
    import torch

    import oracle

    code = {"f16": oracle.F16, "bf16": oracle.BF16}[w.dtype]
    cores = os.cpu_count() or 1
    qn, kn, vn = (t.view(torch.int16).numpy().view(np.uint16) for t in (q, k, v))
    nrows = w.batch * w.nq * w.hq
    row_bytes = row_bytes_of(w, cu)

    def run(threads, budget):
        # rows in chunks of one per thread until the time budget is spent (at least one chunk)
        t0 = time.perf_counter()
        done, pos, evals = 0.0, 0, 0
        while True:
            rows = np.array([(pos + i) % nrows for i in range(threads)], dtype=np.int64)
            pos = (pos + threads) % nrows
            oracle.attend(qn, kn, vn, cu, w.hq, w.hkv, w.d, w.scale, code, rows=rows, threads=threads, nq=w.nq)
            done += float(row_bytes[rows].sum())
            evals += threads
            if time.perf_counter() - t0 >= budget:
                break
        return done, evals, time.perf_counter() - t0

    done, evals, dt = run(cores, seconds)
    d1, e1, t1 = run(1, single_seconds)
    return {"value": round(done / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{evals} row evaluations (the workload's {nrows} (request, query, head) rows, "
                      f"cycled) in {dt:.1f} s, {cores} rows at a time",
            "single_thread": {"value": round(d1 / t1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"{e1} row evaluations in {t1:.1f} s on one thread"}}


# ------------------------------------------------------------------ our arm
class Case:
    """One workload on the device: its inputs, a schedule and the call."""

    def __init__(self, la, torch, w, args, dev, stream, kernel="lean", tile=0, inputs=None, layout="slab"):
        import workloads
        self.la, self.torch, self.w, self.dev, self.stream = la, torch, w, dev, stream
        if inputs is None:
            inputs = workloads.make_inputs(w, seed=args.seed, device=dev)
        self.q, self.k, self.v, self.cu = inputs
        grid = args.grid if args.grid > 0 else (w.grid if w.name == "tiny" else 0)
        self.layout = layout
        slab = layout == "slab" or kernel != "lean"
        plan_times = []
        for _ in range(21):
            t0 = time.perf_counter()
            if not slab:
                la.la_plan_kv(w.batch, w.hq, w.hkv, w.d, self.cu, w.nq, args.heads_per_unit, tile, grid)
            elif w.nq > 1:
                la.la_plan_spec(w.batch, w.hq, w.hkv, w.d, w.nq, self.cu, grid)
            else:
                la.la_plan(w.batch, w.hq, w.hkv, w.d, self.cu, grid, tile)
            plan_times.append((time.perf_counter() - t0) * 1e6)
        self.plan_us = sorted(plan_times)[len(plan_times) // 2]
        if not slab:
            dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, self.cu, num_sms=grid, device=dev, nq=w.nq,
                                 tile_tokens=tile, heads_per_unit=args.heads_per_unit)
        elif w.nq > 1:
            dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, self.cu, num_sms=grid, device=dev, nq=w.nq)
        elif kernel == "lean":
            dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, self.cu, num_sms=grid, device=dev, tile_tokens=tile)
        elif kernel == "naive":
            dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, self.cu, device=dev, fixed_splits=1)
        elif kernel == "auto":
            dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, self.cu, num_sms=grid, device=dev, auto=True)
        else:
            per_sm, sms = la.la_device_capacity(w.d, w.hq // w.hkv)
            splits = -(-sms // (w.batch * w.hkv))
            dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, self.cu, device=dev, fixed_splits=max(1, splits))
        if args.stages:
            la.la_schedule_set_stages(dec.sched, args.stages)
        self.dec = dec
        self.kernel = kernel
        self.export = la.la_schedule_export(dec.sched)
        units = self.export[2]
        self.launches_per_call = 2 if (dec.kind == "fixed_split" and dec.sched.grid > units) else 1
        out_torch = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[args.out_dtype]
        self.out = torch.empty(*self.q.shape, dtype=out_torch, device=dev)
        self.use_flush = uses_flush(w, args)
        self.flush = torch.empty(FLUSH_BYTES if self.use_flush else 1, dtype=torch.uint8, device=dev)
        self.clean = torch.ones(FLUSH_BYTES // 4 if self.use_flush else 1, dtype=torch.int32, device=dev)
        if slab:
            q, k, v, out = self.q, self.k, self.v, self.out

            def call():
                dec(q, k, v, w.scale, out=out, stream=stream)
        else:
            if layout == "token_major":
                kc, vc = workloads.to_token_major(w, self.k, self.v)
                table, npages = None, 0
            else:
                kc, vc, table, npages = workloads.to_paged(w, self.k, self.v, args.page_size, seed=args.seed)
                table = table.to(dev)
            self.k, self.v = kc, vc  # the caches are what the call reads
            cu_dev = torch.as_tensor(self.cu, dtype=torch.int32, device=dev)
            q, out = self.q, self.out

            def call():
                la.la_decode_kv(q, kc, vc, cu_dev, dec.sched, dec.workspace, out, w.scale, layout=layout,
                                block_table=table, page_size=args.page_size, num_pages=npages, stream=stream)
        self.call = call

    def flush_l2(self):
        # write 256 MiB (evicts every line), then read another 256 MiB so the
        # written lines go back to HBM before the timed call, not during it
        self.flush.zero_()
        self.clean.max()

    def one(self):
        if self.use_flush:
            self.flush_l2()
        self.call()

    def check(self):
        st = self.dec.status()
        if st != self.la.LA_OK:
            raise RuntimeError(f"kernel reported: {self.la.status_string(st)}")

    def time(self, steps, warmup, world, marks=None):
        """Warm-up, then `steps` timed calls; returns the mean call time (ms).

        Warm-up: max(3, warmup) calls, then more back to back until at least
        SETTLE_SECONDS of GPU time has run, so clocks and power are in their
        loaded state. The timed calls follow after only the synchronisation
        (and, under torchrun, the barrier) that brackets the timed region.
        marks, if given, receives the wall-clock bounds of the loaded window
        and of the timed region for the clock record."""
        import torch.distributed as dist
        torch, stream, dev = self.torch, self.stream, self.dev
        n0 = max(3, warmup)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        load0 = time.time()
        e0.record(stream)
        for _ in range(n0):
            self.one()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        self.check()
        est = max(e0.elapsed_time(e1) / 1e3 / n0, 1e-6)
        n_settle = min(20000, max(0, math.ceil(SETTLE_SECONDS / est) - n0))
        for _ in range(n_settle):
            self.one()
        self.warmup_calls = n0 + n_settle
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        wall0 = time.time()
        if marks is not None:
            torch.cuda.nvtx.range_push("timed")
        if self.use_flush:
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            for i in range(steps):
                self.flush_l2()
                starts[i].record(stream)
                self.call()
                ends[i].record(stream)
        else:
            starts = [torch.cuda.Event(enable_timing=True)]
            ends = [torch.cuda.Event(enable_timing=True)]
            starts[0].record(stream)
            for _ in range(steps):
                self.call()
            ends[0].record(stream)
        if marks is not None:
            torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        wall1 = time.time()
        if marks is not None:
            marks.update(load0=load0, t0=wall0, t1=wall1)
        mean_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / steps
        self.check()
        return mean_ms

    def spread(self, n):
        """Single calls, events around each (p10, p90 in microseconds)."""
        torch = self.torch
        sp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, e in sp:
            if self.use_flush:
                self.flush_l2()
            a.record(self.stream)
            self.call()
            e.record(self.stream)
        torch.cuda.synchronize(self.dev)
        t = sorted(a.elapsed_time(e) for a, e in sp)
        return round(t[len(t) // 10] * 1e3, 2), round(t[(9 * len(t)) // 10] * 1e3, 2)

    def kernel_name(self):
        return decode_kernel_name(self.w, self.dec.sched)

    def tile(self):
        return self.export[4]

    def roofline(self, mean_ms, peak, peaks_measured, args, profile_key=None):
        w = self.w
        kv_bytes, algo = algorithmic_bytes(w, self.export, self.out.element_size())
        ws = algo - kv_bytes - self.q.numel() * self.q.element_size() - self.out.numel() * self.out.element_size()
        achieved = algo / (mean_ms * 1e-3) / 1e9
        traffic = None
        if self.kernel == "lean" and args.heads_per_unit == 0:
            name = profile_name(profile_key or w.name, self.layout, args.page_size, self.kernel_name())
            traffic = profiled_traffic(name, w.d, self.tile())
        return {"bound": "hbm", "kernel": self.kernel_name(),
                "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_source": "measured hbm_gbs (copy, burst)" if peaks_measured else "fallback 6.8 TB/s",
                "traffic": traffic, "algorithmic_bytes_per_launch": algo,
                "workspace_bytes_per_call": ws, "workspace_frac_of_kv": round(ws / kv_bytes, 6)}

    def free(self):
        for name in ("q", "k", "v", "out", "flush", "clean", "dec", "call"):
            if hasattr(self, name):
                delattr(self, name)


def record(case, mean_ms, peak, peaks_measured, args, world, steps):
    """A nested record: one workload measured like the headline."""
    kv = case.w.kv_bytes()
    p10, p90 = case.spread(min(20, steps))
    return {"workload": case.w.description, "us_per_call": round(mean_ms * 1e3, 3),
            "value": round(world * kv / (mean_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
            "kv_read_frac_of_measured_hbm": round(kv / (mean_ms * 1e-3) / 1e9 / peak, 4),
            "kv_read_frac_of_8tbs_nominal": round(kv / (mean_ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
            "steps": steps, "warmup_calls": case.warmup_calls, "tile_tokens": case.tile(),
            "schedule": case.dec.kind, "grid": case.dec.sched.grid, "kv_bytes": kv,
            "single_call_p10_us": p10, "single_call_p90_us": p90,
            "gpu_launches": steps * case.launches_per_call,
            "roofline": case.roofline(mean_ms, peak, peaks_measured, args)}


def run_ours(args, rank, world, local_rank):
    import torch

    import decode_phase_attention_gb300 as la
    import workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    w = workloads.named(args.workload, seed=args.seed)
    sampler = ClockSampler(local_rank)
    if rank == 0:
        sampler.start()

    case = Case(la, torch, w, args, dev, stream, kernel=args.kernel, tile=args.tile, layout=args.kv_layout)
    marks = {}
    mean_ms = case.time(args.steps, args.warmup, world, marks)
    mean_ms = max_over_ranks(mean_ms, dev)
    p10, p90 = case.spread(min(50, args.steps))
    G = case.dec.sched.grid

    # one extra traced call (outside the timed region): per-CTA balance and host waits
    trace = torch.zeros(G * la.TRACE_WORDS, dtype=torch.int64, device=dev)
    la.la_schedule_set_trace(case.dec.sched, trace)
    case.call()
    torch.cuda.synchronize(dev)
    la.la_schedule_set_trace(case.dec.sched, None)
    cta_trace = summarize_trace(trace.view(G, la.TRACE_WORDS).cpu().numpy())
    case.check()

    kv_bytes = w.kv_bytes()
    value = world * kv_bytes / (mean_ms * 1e-3) / 1e9
    roof = case.roofline(mean_ms, peak, peaks is not None, args)

    # the same workload at the LeanTile table's size (128 tokens at d = 128)
    # and the two fixed partitions, on the same inputs
    variants = {}
    if not args.no_extras and args.kernel == "lean" and args.kv_layout == "slab" and w.nq == 1:
        runs = []
        if w.d == 128 and case.tile() != 128:
            runs.append(("table_tile", "lean", 128))
        runs += [("naive_one_cta_per_unit", "naive", 0), ("fixed_split_plus_merge", "fixed_split", 0)]
        for key, kern, tile in runs:
            c = Case(la, torch, w, args, dev, stream, kernel=kern, tile=tile,
                     inputs=(case.q, case.k, case.v, case.cu))
            ms = max_over_ranks(c.time(args.steps, args.warmup, world), dev)
            variants[key] = {"us_per_call": round(ms * 1e3, 3), "tile_tokens": c.tile(),
                             "schedule": c.dec.kind, "grid": c.dec.sched.grid,
                             "value": round(world * kv_bytes / (ms * 1e-3) / 1e9, 3), "unit": "GB/s",
                             "kv_read_frac_of_measured_hbm": round(kv_bytes / (ms * 1e-3) / 1e9 / peak, 4),
                             "ratio_to_headline_time": round(ms / mean_ms, 4)}
            c.free()

    # end to end through the C ABI: la_decode_host copies q, K, V from pinned
    # host memory, decodes, and copies the output back, every step
    e2e = None
    host = None
    slab_f32 = args.kv_layout == "slab" and args.out_dtype == "f32"
    if (not args.no_e2e and slab_f32) or (not args.no_cpu_baseline and world == 1 and rank == 0):
        host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (case.q, case.k, case.v)]
        for h, t in zip(host, (case.q, case.k, case.v)):
            h.copy_(t)
    if not args.no_e2e and slab_f32:
        qh, kh, vh = host
        outh = torch.empty(case.out.shape, dtype=torch.float32, pin_memory=True)
        dec = case.dec
        n_e2e = max(1, min(args.e2e_steps, args.steps))

        def e2e_step():
            la.la_decode_host(qh, kh, vh, dec.cu_dev, dec.sched, dec.workspace, case.q, case.k, case.v,
                              case.out, outh, w.scale, stream=stream)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        case.check()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        case.check()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, dev)
        h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
        e2e = {"value": round(world * kv_bytes / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
               "us_per_call": round(e2e_ms * 1e3, 2), "steps": n_e2e,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": outh.numel() * outh.element_size(),
               "api": "la_decode_host (one C-ABI call per step: three host-to-device copies, the decode, "
                      "one device-to-host copy, on one stream)"}

    cpu = None
    if not args.no_cpu_baseline and world == 1 and rank == 0:
        cpu = cpu_baseline(w, host[0], host[1], host[2], case.cu, args.cpu_seconds)
    host = None

    config = workload_config(w, args)
    run = {"kernel": args.kernel, "schedule": case.dec.kind, "tile_tokens": case.tile(),
           "out_dtype": args.out_dtype, "kv_heads_per_unit": case.dec.sched.heads_per_unit,
           "query_blocks_per_kv_head": case.dec.sched.query_blocks,
           "ring_stages": args.stages or "library default",
           "kv_layout": args.kv_layout + (f" (page {args.page_size})" if args.kv_layout == "paged" else ""),
           "predicted_us": case.dec.predicted_us, "grid": G,
           "plan_us": round(case.plan_us, 1),
           "plan_note": "median host time of the planner call, outside the timed region",
           "timing": ("CUDA events around the K back-to-back calls" if not case.use_flush else
                      "CUDA events around each call, after a 256 MiB L2 flush"),
           "warmup_calls_issued": case.warmup_calls,
           "warmup_note": (f"max(3, W) warm-up calls, then more back to back until >= {SETTLE_SECONDS} s of "
                           "GPU time; the timed calls follow after one synchronisation"),
           "single_call_p10_us": p10, "single_call_p90_us": p90}
    launches = case.launches_per_call
    case.free()
    del case
    torch.cuda.empty_cache()

    configs = {}
    if not args.no_extras and args.kv_layout == "slab" and args.kernel == "lean":
        steps = min(args.steps, EXTRA_STEPS_MAX)
        for name in EXTRA_WORKLOADS:
            if name == args.workload:
                continue
            wx = workloads.named(name, seed=args.seed)
            c = Case(la, torch, wx, args, dev, stream)
            ms = max_over_ranks(c.time(steps, args.warmup, world), dev)
            rec = record(c, ms, peak, peaks is not None, args, world, steps)
            if name == "ragged" and wx.d == 128 and c.tile() != 128:
                inputs = (c.q, c.k, c.v, c.cu)
                for key, kern, tile in (("table_tile", "lean", 128), ("naive_one_cta_per_unit", "naive", 0),
                                        ("fixed_split_plus_merge", "fixed_split", 0)):
                    cv = Case(la, torch, wx, args, dev, stream, kernel=kern, tile=tile, inputs=inputs)
                    msv = max_over_ranks(cv.time(steps, args.warmup, world), dev)
                    rec[key] = {"us_per_call": round(msv * 1e3, 3), "tile_tokens": cv.tile(),
                                "schedule": cv.dec.kind, "grid": cv.dec.sched.grid,
                                "value": round(world * wx.kv_bytes() / (msv * 1e-3) / 1e9, 3),
                                "ratio_to_default_time": round(msv / ms, 4)}
                    cv.free()
            configs[name] = rec
            c.free()
            del c
            torch.cuda.empty_cache()
    sampler.stop()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean_ms, 6),
        "us_per_call": round(mean_ms * 1e3, 3),
        "kv_read_frac_of_measured_hbm": round(kv_bytes / (mean_ms * 1e-3) / 1e9 / peak, 4),
        "kv_read_frac_of_8tbs_nominal": round(kv_bytes / (mean_ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": config,
        "run": run,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "table_tile_us": variants.get("table_tile", {}).get("us_per_call"),
        "variants": variants,
        "configs": configs,
        "cta_trace": cta_trace,
        "gpu_launches": args.steps * launches,
        "clocks": sampler.summary(marks["load0"], marks["t0"], marks["t1"]),
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
