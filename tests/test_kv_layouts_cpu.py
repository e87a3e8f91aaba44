"""Token-major and paged K/V layouts, host side: the oracle's gathers are
pinned against hand-built caches, the input generators' re-layouts gather
back to the slab layout exactly, and bad cache descriptors are refused
before anything reaches a GPU."""
import ctypes

import numpy as np
import pytest
import torch

import decode_phase_attention_gb300 as la
import workloads
from oracle import layouts


def slab_inputs(lengths, hkv, d, seed=0):
    r = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return cu, r.normal(size=int(cu[-1]) * hkv * d)


def test_token_major_gather_reads_row_cu_plus_t():
    lengths, hkv, d = [3, 5, 1], 2, 4
    cu, slab = slab_inputs(lengths, hkv, d)
    cache = np.zeros((int(cu[-1]), hkv, d))
    for b, L in enumerate(lengths):
        for h in range(hkv):
            for t in range(L):
                cache[cu[b] + t, h] = slab[(hkv * cu[b] + h * L + t) * d:(hkv * cu[b] + h * L + t + 1) * d]
    np.testing.assert_array_equal(layouts.gather_token_major(cache, cu, hkv, d), slab)


def test_paged_gather_follows_the_block_table():
    lengths, hkv, d, P = [5, 9], 2, 4, 4
    cu, slab = slab_inputs(lengths, hkv, d, seed=1)
    table = np.array([[3, 0, -1], [1, 4, 2]], np.int32)  # request 1 needs 3 pages
    cache = np.full((5, P, hkv, d), np.nan)
    for b, L in enumerate(lengths):
        for h in range(hkv):
            for t in range(L):
                cache[table[b, t // P], t % P, h] = slab[(hkv * cu[b] + h * L + t) * d:(hkv * cu[b] + h * L + t + 1) * d]
    got = layouts.gather_paged(cache, table, cu, P, hkv, d)
    np.testing.assert_array_equal(got, slab)


@pytest.mark.parametrize("P", [16, 64, 256])
def test_generated_layouts_gather_back_to_the_slab(P):
    w = workloads.custom(3, 4, 2, 64, "bf16", [300, 17, 1000])
    q, k, v, cu = workloads.make_inputs(w, seed=4)
    ktm, vtm = workloads.to_token_major(w, k, v)
    kp, vp, table, npages = workloads.to_paged(w, k, v, P, seed=4)
    for src, dst in ((k, ktm), (v, vtm)):
        np.testing.assert_array_equal(layouts.gather_token_major(dst.float().numpy(), cu, w.hkv, w.d),
                                      src.float().numpy())
    for src, dst in ((k, kp), (v, vp)):
        np.testing.assert_array_equal(layouts.gather_paged(dst.float().numpy(), table.numpy(), cu, P, w.hkv, w.d),
                                      src.float().numpy())
    assert torch.isnan(kp.float()).any()  # junk in the unused slots


def _desc(layout, table_ptr=0x30000, max_blocks=4, page=64, pages=10):
    return la.KvDesc(layout, table_ptr, max_blocks, page, pages)


@pytest.mark.parametrize("desc,status", [
    (_desc(la.KV_PAGED, page=48), la.LA_ERR_INVALID),            # not a power of two
    (_desc(la.KV_PAGED, page=8), la.LA_ERR_INVALID),             # too small
    (_desc(la.KV_PAGED, table_ptr=0), la.LA_ERR_INVALID),        # no block table
    (_desc(la.KV_PAGED, max_blocks=1), la.LA_ERR_INVALID),       # table too narrow for 200 tokens / 64
    (_desc(la.KV_PAGED, pages=0), la.LA_ERR_INVALID),
    (_desc(la.KV_PAGED, pages=1 << 30), la.LA_ERR_UNSUPPORTED),  # more than 2^31 - 1 rows
    (_desc(7), la.LA_ERR_INVALID),                               # unknown layout
])
def test_bad_cache_descriptors_are_refused_before_any_launch(desc, status):
    s = la.la_plan(2, 4, 4, 128, [0, 200, 300], 5)
    p = ctypes.c_void_p(0x10000)
    assert la._lib.la_decode_kv(p, p, p, 1, p, ctypes.byref(desc), s.handle, ctypes.c_void_p(0x20000), p, 0,
                                0.1, None) == status


def test_small_pages_on_the_narrow_swizzle_path_are_unsupported():
    # d = 80 with group 4 reads 32-byte swizzled boxes: a 16-token page is a 512-byte piece
    s = la.la_plan(1, 8, 2, 80, [0, 500], 5)
    p = ctypes.c_void_p(0x10000)
    d = _desc(la.KV_PAGED, page=16, max_blocks=40, pages=64)
    assert la._lib.la_decode_kv(p, p, p, 1, p, ctypes.byref(d), s.handle, ctypes.c_void_p(0x20000), p, 0,
                                0.1, None) == la.LA_ERR_UNSUPPORTED
