"""Gather K or V from a token-major or paged cache into the slab layout the
oracle reads (request b: a [hkv, L_b, d] slab at element hkv*cu[b]*d).

TEST INFRASTRUCTURE ONLY. Plain per-token indexing from the layout
definitions, so the oracle reads the caches the library reads:
  token-major  [total tokens, hkv, d]: token t of request b, head h at row cu[b] + t
  paged        [num_pages, page_size, hkv, d]: token t of request b in page
               block_table[b, t // page_size], slot t % page_size
"""
import numpy as np


def gather_token_major(cache, cu, hkv, d):
    cache = np.asarray(cache).reshape(-1, hkv, d)
    out = []
    for b in range(len(cu) - 1):
        L = int(cu[b + 1] - cu[b])
        for h in range(hkv):
            rows = [cache[int(cu[b]) + t, h, :] for t in range(L)]
            out.append(np.stack(rows))
    return np.concatenate([x.reshape(-1) for x in out])


def gather_paged(cache, block_table, cu, page_size, hkv, d):
    cache = np.asarray(cache).reshape(-1, page_size, hkv, d)
    block_table = np.asarray(block_table)
    out = []
    for b in range(len(cu) - 1):
        L = int(cu[b + 1] - cu[b])
        for h in range(hkv):
            rows = [cache[int(block_table[b, t // page_size]), t % page_size, h, :] for t in range(L)]
            out.append(np.stack(rows))
    return np.concatenate([x.reshape(-1) for x in out])
