"""Benchmark: LeanAttention stream-K decode attention on GB300.

One step is one decode-attention call over one batch: the LeanTile loop,
the partial exchange, the host-CTA reduction and the normalisation, all in
one launch of the library's kernel (the schedule is planned once for the
batch, outside the timed region; its host time is reported as plan_us).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--kernel lean|naive|fixed_split] [--impl ours|reference]

value = K+V bytes read / kernel time, summed over ranks (GB/s); the kernel
time is taken with CUDA events on the launching stream around the K timed
back-to-back calls (single-call spread reported separately).
Inputs larger than 4x L2 are not flushed between calls (the next call
cannot hit in L2); smaller ones get a 256 MiB write before every call. e2e = the same metric with the
inputs copied from pinned host memory and the output copied back inside
every timed step. --impl reference times the float64 CPU oracle instead.
Under torchrun every rank runs an independent replica (the path has no
cross-GPU exchange) and the slowest rank's time is reported.
"""
import argparse
import hashlib
import json
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="uniform")
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
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
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

    def summary(self, t0, t1):
        if self.proc is None:
            return None
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 <= r[0] <= t1 + 0.06]
        used = inside if inside else rows
        if not used:
            return None
        mhz = sorted(float(p[2]) for _, p in used if p[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, p in used:
            for n, val in zip(names, p[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": mhz[len(mhz) // 2] if mhz else None,
                "sm_max_mhz": float(used[0][1][3]) if used[0][1][3].replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(used),
                "in_timed_region": bool(inside)}


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
    nrows = w.batch * w.nq * w.hq  # row r = (b * nq + i) * hq + h
    rows_per_kv = (w.hq // w.hkv) * w.nq
    row_bytes = np.array([2 * (cu[r // (w.nq * w.hq) + 1] - cu[r // (w.nq * w.hq)]) * w.d * 2 / rows_per_kv
                          for r in range(nrows)])
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
        "config": {"workload": w.description, "batch": w.batch, "hq": w.hq, "hkv": w.hkv, "head_dim": w.d,
                   "total_context_tokens": w.total_tokens, "kv_bytes": w.kv_bytes(), "seed": args.seed},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w, q, k, v, cu, seconds, single_seconds=2.0):
    """The float64 oracle on the host cores over the workload's rows, cycled,
    for about `seconds`; then the same with one thread for `single_seconds`."""
    import numpy as np
    import torch

    import oracle

    code = {"f16": oracle.F16, "bf16": oracle.BF16}[w.dtype]
    cores = os.cpu_count() or 1
    qn, kn, vn = (t.view(torch.int16).numpy().view(np.uint16) for t in (q, k, v))
    nrows = w.batch * w.nq * w.hq  # row r = (b * nq + i) * hq + h
    rows_per_kv = (w.hq // w.hkv) * w.nq
    row_bytes = np.array([2 * (cu[r // (w.nq * w.hq) + 1] - cu[r // (w.nq * w.hq)]) * w.d * 2 / rows_per_kv
                          for r in range(nrows)])

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
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import decode_phase_attention_gb300 as la
    import workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workloads.named(args.workload, seed=args.seed)
    q, k, v, cu = workloads.make_inputs(w, seed=args.seed, device=dev)
    grid = args.grid if args.grid > 0 else (w.grid if args.workload == "tiny" else 0)
    plan_times = []
    for _ in range(21):
        t0 = time.perf_counter()
        if args.kv_layout != "slab" and args.kernel == "lean":
            la.la_plan_kv(w.batch, w.hq, w.hkv, w.d, cu, w.nq, args.heads_per_unit, args.tile, grid)
        else:
            la.la_plan(w.batch, w.hq, w.hkv, w.d, cu, grid if grid > 0 else 0, args.tile)
        plan_times.append((time.perf_counter() - t0) * 1e6)
    plan_us = sorted(plan_times)[len(plan_times) // 2]
    out_torch = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[args.out_dtype]
    if args.kv_layout != "slab" and args.kernel == "lean":
        dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, cu, num_sms=grid, device=dev, nq=w.nq,
                             tile_tokens=args.tile, heads_per_unit=args.heads_per_unit)
    elif w.nq > 1:
        dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, cu, num_sms=grid, device=dev, nq=w.nq)
    elif args.kernel == "lean":
        dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, cu, num_sms=grid, device=dev, tile_tokens=args.tile)
    elif args.kernel == "naive":
        dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, cu, device=dev, fixed_splits=1)
    elif args.kernel == "auto":
        dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, cu, num_sms=grid, device=dev, auto=True)
    else:
        per_sm, sms = la.la_device_capacity(w.d, w.hq // w.hkv)
        splits = -(-sms // (w.batch * w.hkv))
        dec = la.LeanDecoder(w.batch, w.hq, w.hkv, w.d, cu, device=dev, fixed_splits=max(1, splits))
    if args.stages:
        la.la_schedule_set_stages(dec.sched, args.stages)
    G = dec.sched.grid
    units = la.la_schedule_export(dec.sched)[2]
    launches_per_call = 2 if (dec.kind == "fixed_split" and dec.sched.grid > units) else 1
    stream = torch.cuda.current_stream(dev)
    out = torch.empty(*q.shape, dtype=out_torch, device=dev)
    # K+V well above L2 (129 MB) cannot be served from L2 by the next call; smaller
    # inputs get a 256 MiB write between calls to flush L2.
    use_flush = args.flush or w.kv_bytes() < L2_BYTES * 4
    flush = torch.empty(FLUSH_BYTES if use_flush else 1, dtype=torch.uint8, device=dev)
    clean = torch.ones(FLUSH_BYTES // 4 if use_flush else 1, dtype=torch.int32, device=dev)

    def flush_l2():
        # write 256 MiB (evicts every line), then read another 256 MiB so the
        # written lines go back to HBM before the timed call, not during it
        flush.zero_()
        clean.max()

    if args.kv_layout == "slab":
        def call():
            dec(q, k, v, w.scale, out=out, stream=stream)
    else:
        if args.kv_layout == "token_major":
            kc, vc = workloads.to_token_major(w, k, v)
            table, npages = None, 0
        else:
            kc, vc, table, npages = workloads.to_paged(w, k, v, args.page_size, seed=args.seed)
            table = table.to(dev)
        del k, v
        k, v = kc, vc  # the e2e leg copies these caches
        cu_dev = torch.as_tensor(cu, dtype=torch.int32, device=dev)

        def call():
            la.la_decode_kv(q, kc, vc, cu_dev, dec.sched, dec.workspace, out, w.scale, layout=args.kv_layout,
                            block_table=table, page_size=args.page_size, num_pages=npages, stream=stream)

    # warm-up (also uploads the schedule)
    for _ in range(max(3, args.warmup)):
        if use_flush:
            flush_l2()
        call()
    torch.cuda.synchronize(dev)
    st = dec.status()
    if st != la.LA_OK:
        raise RuntimeError(f"kernel reported: {la.status_string(st)}")

    sampler = ClockSampler(local_rank)
    if rank == 0:
        sampler.start()
        time.sleep(0.2)
    # Timed region: K back-to-back calls between two events on the launching
    # stream (with L2 flushes, when used, timed per call instead).
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps if use_flush else 1)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps if use_flush else 1)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    torch.cuda.nvtx.range_push("timed")
    if use_flush:
        for i in range(args.steps):
            flush_l2()
            starts[i].record(stream)
            call()
            ends[i].record(stream)
    else:
        starts[0].record(stream)
        for i in range(args.steps):
            call()
        ends[0].record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    wall1 = time.time()
    sampler.stop()
    if use_flush:
        mean_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    else:
        mean_ms = starts[0].elapsed_time(ends[0]) / args.steps
    # spread of single calls (outside the timed region): events around each call
    n_spread = min(50, args.steps)
    sp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_spread)]
    for a, e in sp:
        if use_flush:
            flush_l2()
        a.record(stream)
        call()
        e.record(stream)
    torch.cuda.synchronize(dev)
    times_ms = sorted(a.elapsed_time(e) for a, e in sp)
    mean_ms = max_over_ranks(mean_ms, dev)
    st = dec.status()
    if st != la.LA_OK:
        raise RuntimeError(f"kernel reported: {la.status_string(st)}")

    # one extra traced call (outside the timed region): per-CTA balance and host waits
    trace = torch.zeros(G * la.TRACE_WORDS, dtype=torch.int64, device=dev)
    la.la_schedule_set_trace(dec.sched, trace)
    call()
    torch.cuda.synchronize(dev)
    la.la_schedule_set_trace(dec.sched, None)
    cta_trace = summarize_trace(trace.view(G, la.TRACE_WORDS).cpu().numpy())

    kv_bytes, algo_bytes = algorithmic_bytes(w, la.la_schedule_export(dec.sched), out.element_size())
    ws_bytes = algo_bytes - kv_bytes - q.numel() * q.element_size() - out.numel() * out.element_size()
    value = world * kv_bytes / (mean_ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        outh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        n_e2e = max(1, min(args.e2e_steps, args.steps))
        for _ in range(2):
            q.copy_(qh, non_blocking=True), k.copy_(kh, non_blocking=True), v.copy_(vh, non_blocking=True)
            call()
            outh.copy_(out, non_blocking=True)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            q.copy_(qh, non_blocking=True)
            k.copy_(kh, non_blocking=True)
            v.copy_(vh, non_blocking=True)
            call()
            outh.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        e2e_ms = max_over_ranks(e2e_ms, dev)
        h2d = (q.numel() + k.numel() + v.numel()) * q.element_size()
        e2e = {"value": round(world * kv_bytes / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
               "us_per_call": round(e2e_ms * 1e3, 2), "steps": n_e2e,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out.numel() * out.element_size()}

    if rank != 0:
        return
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    achieved = algo_bytes / (mean_ms * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(w, q.cpu(), k.cpu(), v.cpu(), cu, args.cpu_seconds)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean_ms, 6),
        "us_per_call": round(mean_ms * 1e3, 3),
        "kv_read_frac_of_measured_hbm": round(kv_bytes / (mean_ms * 1e-3) / 1e9 / peak, 4),
        "kv_read_frac_of_8tbs_nominal": round(kv_bytes / (mean_ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.description, "kernel": args.kernel, "schedule": dec.kind,
                   "tile_tokens": la.la_schedule_export(dec.sched)[4], "out_dtype": args.out_dtype,
                   "kv_heads_per_unit": dec.sched.heads_per_unit,
                   "query_blocks_per_kv_head": dec.sched.query_blocks,
                   "ring_stages": args.stages or "library default",
                   "kv_layout": args.kv_layout + (f" (page {args.page_size})" if args.kv_layout == "paged" else ""),
                   "predicted_us": dec.predicted_us, "grid": G,
                   "batch": w.batch, "hq": w.hq, "hkv": w.hkv, "head_dim": w.d,
                   "total_context_tokens": w.total_tokens, "kv_bytes": kv_bytes,
                   "l2": ("flushed before every timed call (256 MiB write, then 256 MiB read so no "
                          "dirty line is written back inside the call)" if use_flush else
                          f"no flush: K+V ({kv_bytes / 1e9:.2f} GB) exceed 4x the 129 MB L2"),
                   "plan_us": round(plan_us, 1), "plan_note": "median host time of the planner call, outside the timed region",
                   "seed": args.seed,
                   "timing": ("CUDA events around the K back-to-back calls" if not use_flush else
                              "CUDA events around each call, after a 256 MiB L2 flush"),
                   "single_call_p10_us": round(times_ms[len(times_ms) // 10] * 1e3, 2),
                   "single_call_p90_us": round(times_ms[(9 * len(times_ms)) // 10] * 1e3, 2)},
        "roofline": {"bound": "hbm", "kernel": decode_kernel_name(w, dec.sched),
                     "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": "measured hbm_gbs (copy, burst)" if peaks else "fallback 6.8 TB/s",
                     "traffic": (profiled_traffic(profile_name(args.workload, args.kv_layout, args.page_size,
                                                               decode_kernel_name(w, dec.sched)),
                                                  w.d, la.la_schedule_export(dec.sched)[4])
                                 if args.kernel == "lean" and args.heads_per_unit == 0 else None),
                     "algorithmic_bytes_per_launch": algo_bytes,
                     "workspace_bytes_per_call": ws_bytes,
                     "workspace_frac_of_kv": round(ws_bytes / kv_bytes, 6)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "cta_trace": cta_trace,
        "gpu_launches": args.steps * launches_per_call,
        "clocks": sampler.summary(wall0, wall1),
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
