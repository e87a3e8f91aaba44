"""Reference tile planner for LeanAttention's stream-K decomposition.

TEST INFRASTRUCTURE ONLY: used by the test suite to check the library's
planner, never by the product path. It shares no code with the library.

What it follows (xllm-io paper review of LeanAttention):
  * "3.3 LeanTile": the smallest unit of work is a LeanTile of 256 tokens at
    head dim 64 and 128 tokens at head dim 128.
  * "3.4 stream-K style decomposition": LeanTile iterations are laid out on
    one line along the context, the total work is divided evenly over the
    CTAs, and a CTA may cross head and request boundaries.
  * "3.5 execution flow": grid size G, I_G = I / G iterations per CTA, then
    a host CTA and a finishing CTA per output tile; non-host CTAs hand their
    partial result to the host through global memory.
  * "4.3 hardware-aware work distribution": G equal to the number of output
    tiles behaves like FlashAttention-2, G a multiple of it like
    FlashDecoding.

Readings where the pages are silent (each is stated in the design notes):
  * the unit of work ("output tile") is (request b, kv head); under grouped
    query attention all query heads of one kv head share the unit;
  * units are ordered request-major, then kv head, then tile index;
  * I / G is not an integer in general: the first I mod G CTAs take one
    extra iteration;
  * a context that is not a multiple of the LeanTile ends in a partial tile;
  * the host of a unit is the lowest CTA that touches it, the one holding
    its first iteration; the finisher holds its last iteration.

This module computes the schedule the slow, direct way: it writes down the
owner of every single iteration and groups consecutive iterations, so it
does not share the library's range arithmetic.
"""

WHOLE, NONHOST, HOST, PARTIAL = 0, 1, 2, 3
LEAN, FIXED = 0, 1
MAGIC = 0x4C41


def lean_tile(d):
    """LeanTile size in tokens ("3.3 LeanTile" table)."""
    table = {64: 256, 128: 128}
    if d not in table:
        raise ValueError(f"no LeanTile size for head dim {d}")
    return table[d]


def _units(batch, hkv, d, cu, T=None):
    T = lean_tile(d) if T is None else T
    if T <= 0:
        raise ValueError("tile size must be positive")
    tiles = []
    for b in range(batch):
        L = cu[b + 1] - cu[b]
        if L <= 0:
            raise ValueError("every request needs a non-empty context")
        n = -(-L // T)  # ceil
        for _h in range(hkv):
            tiles.append(n)
    return T, tiles


def _iteration_owner_even(I, G):
    """owner[i] = CTA of iteration i when I iterations are split evenly over G CTAs."""
    owner = []
    for g in range(G):
        count = I // G + (1 if g < I % G else 0)
        owner.extend([g] * count)
    assert len(owner) == I
    return owner


def _prefix_counts(owner, G):
    """cta_iter[g] = number of iterations owned by CTAs below g."""
    counts = [0] * G
    for g in owner:
        counts[g] += 1
    prefix = [0]
    for c in counts:
        prefix.append(prefix[-1] + c)
    return prefix


def _segments_from_owner(owner, unit_iter, G, kind_rule):
    """Group consecutive iterations of one CTA inside one unit into segments."""
    U = len(unit_iter) - 1
    unit_of = []
    for u in range(U):
        unit_of.extend([u] * (unit_iter[u + 1] - unit_iter[u]))
    per_cta = [[] for _ in range(G)]
    i = 0
    I = len(owner)
    while i < I:
        g, u = owner[i], unit_of[i]
        j = i
        while j < I and owner[j] == g and unit_of[j] == u:
            j += 1
        per_cta[g].append([u, i - unit_iter[u], j - unit_iter[u]])
        i = j
    unit_host = [owner[unit_iter[u]] for u in range(U)]
    unit_fin = [owner[unit_iter[u + 1] - 1] for u in range(U)]
    segs = []
    cta_seg = [0]
    for g in range(G):
        for u, t0, t1 in per_cta[g]:
            kind, peer = kind_rule(g, u, t0, t1, unit_iter, unit_host, unit_fin)
            segs.append((u, t0, t1, kind, peer))
        cta_seg.append(len(segs))
    return segs, cta_seg, unit_host, unit_fin


def plan_lean(batch, hq, hkv, d, cu, G, T=None):
    """Stream-K schedule over G CTAs (T: LeanTile tokens, default from the table)."""
    if hq % hkv != 0 or G <= 0:
        raise ValueError("bad shape")
    T, tiles = _units(batch, hkv, d, cu, T)
    unit_iter = [0]
    for n in tiles:
        unit_iter.append(unit_iter[-1] + n)
    I = unit_iter[-1]
    owner = _iteration_owner_even(I, G)
    cta_iter = _prefix_counts(owner, G)

    def kind_rule(g, u, t0, t1, unit_iter, unit_host, unit_fin):
        n = unit_iter[u + 1] - unit_iter[u]
        if t0 == 0 and t1 == n:
            return WHOLE, -1
        if t0 == 0:
            return HOST, unit_fin[u]
        return NONHOST, -1

    segs, cta_seg, unit_host, unit_fin = _segments_from_owner(owner, unit_iter, G, kind_rule)
    return dict(kind=LEAN, splits=0, G=G, U=len(tiles), I=I, T=T, cta_iter=cta_iter,
                unit_iter=unit_iter, cta_seg=cta_seg, segs=segs, unit_host=unit_host,
                unit_fin=unit_fin)


def plan_fixed(batch, hq, hkv, d, cu, splits, T=None):
    """Fixed partition: every unit cut into min(splits, tiles) even pieces, one CTA each.

    splits == 1 is the FlashAttention-2 decode partition (one CTA per unit);
    splits > 1 is the FlashDecoding fixed split, whose pieces are merged by a
    separate reduction launch.
    """
    if hq % hkv != 0 or splits <= 0:
        raise ValueError("bad shape")
    T, tiles = _units(batch, hkv, d, cu, T)
    unit_iter = [0]
    for n in tiles:
        unit_iter.append(unit_iter[-1] + n)
    owner = []
    g = 0
    for n in tiles:
        k = min(splits, n)
        for s in range(k):
            lo, hi = (s * n) // k, ((s + 1) * n) // k
            owner.extend([g] * (hi - lo))
            g += 1
    G = g
    cta_iter = _prefix_counts(owner, G)

    def kind_rule(c, u, t0, t1, unit_iter, unit_host, unit_fin):
        n = unit_iter[u + 1] - unit_iter[u]
        if t0 == 0 and t1 == n:
            return WHOLE, -1
        return PARTIAL, -1

    segs, cta_seg, unit_host, unit_fin = _segments_from_owner(owner, unit_iter, G, kind_rule)
    return dict(kind=FIXED, splits=splits, G=G, U=len(tiles), I=unit_iter[-1], T=T,
                cta_iter=cta_iter, unit_iter=unit_iter, cta_seg=cta_seg, segs=segs,
                unit_host=unit_host, unit_fin=unit_fin)


def export(p):
    """Flatten a schedule into the int32 layout of la_schedule_export.

    [MAGIC, G, U, I, T, nseg, kind, splits]
    cta_iter[G+1], unit_iter[U+1], cta_seg[G+1],
    segs[nseg * 5] as (unit, tile_begin, tile_end, kind, peer),
    unit_host[U], unit_fin[U]
    """
    out = [MAGIC, p["G"], p["U"], p["I"], p["T"], len(p["segs"]), p["kind"], p["splits"]]
    out += p["cta_iter"] + p["unit_iter"] + p["cta_seg"]
    for s in p["segs"]:
        out += list(s)
    out += p["unit_host"] + p["unit_fin"]
    return out
