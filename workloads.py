"""Seeded synthetic inputs for decode-phase attention.

This module only draws numbers: it holds no step of the attention method.
The test suite and the benchmark use it to feed the same bytes to the CUDA
library and to the CPU oracle (the oracle receives copies of the exact
fp16/bf16 tensors the GPU reads; neither side regenerates them).

Layout of one batch (the library's and the oracle's layout):
  q   [batch, hq, d]
  k,v request b occupies a [hkv, L_b, d] slab at element offset hkv*cu[b]*d,
      L_b = cu[b+1] - cu[b]; with equal lengths this is [batch, hkv, L, d].
  cu  int32 [batch+1], cu[0] = 0, the running sum of the context lengths.

The named workloads are the decode shapes the LeanAttention evaluation
sweeps (context length, batch, head count, head dim, ragged batches and
grouped-query heads); the pages' own model runs and 500-sample sweep need
trained weights and are replaced by these i.i.d. N(0, 1) inputs.
"""
import math
from dataclasses import dataclass, field

import numpy as np


@dataclass
class Workload:
    name: str
    batch: int
    hq: int
    hkv: int
    d: int
    dtype: str  # "f16" or "bf16"
    lengths: list = field(default_factory=list)
    grid: int = 0  # 0: the library's default (one persistent CTA per SM)
    outlier_frac: float = 0.0  # fraction of key rows multiplied by outlier_scale
    outlier_scale: float = 8.0
    description: str = ""
    nq: int = 1  # query tokens per request (the last nq tokens of the context)

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d)

    @property
    def cu(self):
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)

    @property
    def total_tokens(self):
        return int(sum(self.lengths))

    def kv_bytes(self):
        """Bytes of K plus V the attention must read once."""
        return 2 * self.hkv * self.d * 2 * self.total_tokens


def _seed(*parts):
    """A 63-bit seed from integer parts (splitmix-style mixing, plain integers)."""
    x = 0x9E3779B97F4A7C15
    for p in parts:
        x = (x ^ (int(p) & 0xFFFFFFFFFFFFFFFF)) * 0xBF58476D1CE4E5B9 & 0xFFFFFFFFFFFFFFFF
        x ^= x >> 31
    return x & 0x7FFFFFFFFFFFFFFF


def ragged_lengths(n, lo, hi, seed, log_uniform):
    rng = np.random.default_rng(_seed(seed, 0x1E9, n, lo, hi, int(log_uniform)))
    if log_uniform:
        x = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
        return [int(min(hi, max(lo, math.floor(v)))) for v in x]
    return [int(v) for v in rng.integers(lo, hi + 1, size=n)]


def named(name, seed=0):
    """The benchmark and parity workloads, by name."""
    if name == "tiny":
        return Workload(name, 1, 4, 4, 64, "f16", [1024], grid=3,
                        description="tiny exact check: batch 1, 4/4 heads, d 64, ctx 1024, "
                                    "fp16, grid forced to 3 CTAs")
    if name == "uniform":
        return Workload(name, 8, 32, 32, 128, "bf16", [8192] * 8,
                        description="uniform decode batch: batch 8, 32/32 heads, d 128, "
                                    "ctx 8192 per request, bf16")
    if name.startswith("long"):
        ctx = {"long64k": 65536, "long256k": 262144, "long512k": 524288}[name]
        return Workload(name, 1, 32, 32, 128, "f16", [ctx],
                        description=f"long context: batch 1, 32/32 heads, d 128, ctx {ctx}, fp16")
    if name == "ragged":
        lens = ragged_lengths(16, 1024, 131072, seed, log_uniform=True)
        return Workload(name, 16, 32, 32, 128, "bf16", lens,
                        description="ragged batch: 16 requests, 32/32 heads, d 128, ctx "
                                    "log-uniform in [1024, 131072], bf16")
    if name == "ragged_div5":
        # the ragged batch with every length divided by 5 (1.74 GB of K+V
        # instead of 8.7): the same mix of short and long requests at a size
        # a many-pass profiler capture can hold
        lens = [max(1, n // 5) for n in ragged_lengths(16, 1024, 131072, seed, log_uniform=True)]
        return Workload(name, 16, 32, 32, 128, "bf16", lens,
                        description="ragged batch, lengths / 5: 16 requests, 32/32 heads, d 128, ctx "
                                    "log-uniform in [1024, 131072] divided by 5, bf16")
    if name == "gqa":
        lens = ragged_lengths(8, 16384, 65536, seed, log_uniform=False)
        return Workload(name, 8, 64, 8, 64, "bf16", lens, outlier_frac=0.01,
                        description="GQA small-head: batch 8, 64 query over 8 kv heads, d 64, "
                                    "ctx uniform in [16384, 65536], bf16, 1% of keys x8")
    if name in ("hd80", "hd96", "hd256"):
        d = int(name[2:])
        heads = 16 if d == 256 else 32
        return Workload(name, 4, heads, heads, d, "bf16", [32768] * 4,
                        description=f"head dim {d}: batch 4, {heads}/{heads} heads, d {d}, ctx 32768, bf16")
    if name.startswith("mha_"):
        # sweep shapes, e.g. mha_h56_b1_c65536_d64: batch b, h/h heads, d, equal contexts, fp16
        parts = dict((p[0], int(p[1:])) for p in name.split("_")[1:])
        h, b, c, d = parts["h"], parts["b"], parts["c"], parts["d"]
        return Workload(name, b, h, h, d, "f16", [c] * b,
                        description=f"sweep: batch {b}, {h}/{h} heads, d {d}, ctx {c}, fp16")
    if name.startswith("gqa_"):
        # grouped-query sweep shapes, e.g. gqa_h32_k8_b1_c32768_d128: batch b, h query over k kv
        # heads, d, equal contexts, bf16
        parts = dict((p[0], int(p[1:])) for p in name.split("_")[1:])
        h, kv, b, c, d = parts["h"], parts["k"], parts["b"], parts["c"], parts["d"]
        return Workload(name, b, h, kv, d, "bf16", [c] * b,
                        description=f"GQA sweep: batch {b}, {h} query over {kv} kv heads, d {d}, ctx {c}, bf16")
    if name.startswith("spec"):
        # speculative-decoding verification: specN = N draft tokens per
        # request (spec4: 4), each attending causally to the ones before it
        n = int(name[4:] or 4)
        return Workload(name, 8, 32, 32, 128, "bf16", [8192] * 8, nq=n,
                        description=f"speculative verification: batch 8, {n} query tokens per request, "
                                    f"32/32 heads, d 128, ctx 8192, bf16, causal among the {n}")
    if name == "hd128gqa":
        return Workload(name, 4, 32, 4, 128, "bf16", [32768] * 4,
                        description="GQA d 128: batch 4, 32 query over 4 kv heads, d 128, ctx 32768, bf16")
    raise KeyError(name)


NAMES = ["tiny", "uniform", "long64k", "long256k", "long512k", "ragged", "gqa"]
EXTRA_NAMES = ["hd80", "hd96", "hd256", "hd128gqa", "spec4"]


def make_inputs(w, seed=0, device="cpu"):
    """Draw q, k, v for a workload; returns (q, k, v, cu_host_np).

    Each (request, kv head) slab of K and V is drawn from its own generator
    seeded by (seed, slab, tensor), N(0, 1) in float32, then rounded to the
    workload's dtype (round to nearest even). For the grouped-query workload
    a seeded 1% of key rows is multiplied by 8 before rounding (a power of
    two, so the rounding is unchanged).
    """
    import torch

    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
    dev = torch.device(device)
    cu = w.cu
    gen = torch.Generator(device=dev)

    gen.manual_seed(_seed(seed, 0xA11, 0))
    qshape = (w.batch, w.hq, w.d) if w.nq == 1 else (w.batch, w.nq, w.hq, w.d)
    q = torch.randn(*qshape, generator=gen, device=dev, dtype=torch.float32).to(tdt)
    n_kv = w.hkv * w.total_tokens * w.d
    k = torch.empty(n_kv, dtype=tdt, device=dev)
    v = torch.empty(n_kv, dtype=tdt, device=dev)
    for b in range(w.batch):
        L = int(cu[b + 1] - cu[b])
        for h in range(w.hkv):
            off = (w.hkv * int(cu[b]) + h * L) * w.d
            for which, dst in ((1, k), (2, v)):
                gen.manual_seed(_seed(seed, b, h, which))
                x = torch.randn(L, w.d, generator=gen, device=dev, dtype=torch.float32)
                if which == 1 and w.outlier_frac > 0:
                    gen.manual_seed(_seed(seed, b, h, 3))
                    rows = torch.rand(L, generator=gen, device=dev) < w.outlier_frac
                    x[rows] *= w.outlier_scale
                dst[off:off + L * w.d] = x.reshape(-1).to(tdt)
    return q, k, v, cu


def custom(batch, hq, hkv, d, dtype, lengths, grid=0, name="custom", nq=1):
    return Workload(name, batch, hq, hkv, d, dtype, list(lengths), grid=grid, nq=nq,
                    description=f"{name}: batch {batch}, {hq}/{hkv} heads, d {d}, {dtype}, nq {nq}")


def to_token_major(w, k, v):
    """Re-lay slab-layout K and V as [total tokens, hkv, d] (same values)."""
    out = []
    for x in (k, v):
        y = x.new_empty(w.total_tokens * w.hkv * w.d)
        cu = w.cu
        for b in range(w.batch):
            L = int(cu[b + 1] - cu[b])
            slab = x[w.hkv * int(cu[b]) * w.d: w.hkv * int(cu[b + 1]) * w.d].view(w.hkv, L, w.d)
            y[int(cu[b]) * w.hkv * w.d: int(cu[b + 1]) * w.hkv * w.d] = slab.transpose(0, 1).reshape(-1)
        out.append(y)
    return out[0], out[1]


def to_paged(w, k, v, page_size, seed=0, spare_pages=3, fill=float("nan")):
    """Re-lay slab-layout K and V as a paged cache [pages, page_size, hkv, d].

    Pages are handed out in a seeded random order; unused slots of the last
    page of each request, the spare pages and the unused block-table
    entries (-1) hold junk (NaN by default) so that reading them shows up.
    Returns (k_cache, v_cache, block_table [batch, max_blocks] int32, num_pages).
    """
    import torch

    cu = w.cu
    blocks = [-(-int(cu[b + 1] - cu[b]) // page_size) for b in range(w.batch)]
    num_pages = sum(blocks) + spare_pages
    max_blocks = max(blocks) + 1
    rng = np.random.default_rng(_seed(seed, 0xB10C, page_size))
    perm = rng.permutation(num_pages)
    table = np.full((w.batch, max_blocks), -1, dtype=np.int32)
    nxt = 0
    for b in range(w.batch):
        for i in range(blocks[b]):
            table[b, i] = perm[nxt]
            nxt += 1
    caches = []
    for x in (k, v):
        c = x.new_full((num_pages, page_size, w.hkv, w.d), fill)
        for b in range(w.batch):
            L = int(cu[b + 1] - cu[b])
            slab = x[w.hkv * int(cu[b]) * w.d: w.hkv * int(cu[b + 1]) * w.d].view(w.hkv, L, w.d)
            tok_major = slab.transpose(0, 1)  # [L, hkv, d]
            for i in range(blocks[b]):
                t0, t1 = i * page_size, min(L, (i + 1) * page_size)
                c[int(table[b, i]), : t1 - t0] = tok_major[t0:t1]
        caches.append(c.reshape(-1))
    return caches[0], caches[1], torch.as_tensor(table), num_pages
