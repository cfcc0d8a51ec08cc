"""Decode against a paged K/V cache, float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[AscendC FA-2] section 9 ("Extensions: integration with RoPE and a paged KV
cache") replaces the K/V block loads with a gather from a paged cache.  The
page gives no format, so this module takes the common one:

  * k_cache, v_cache: [num_pages, page_size, H_kv, D]; a page holds
    page_size consecutive positions of one sequence, all K/V heads;
  * block_table: [B, max_pages] int; position j of sequence b lives in page
    block_table[b, j // page_size], row j % page_size;
  * seq_lens: [B]; sequence b has seq_lens[b] cached positions, and its Nq
    new queries sit at positions seq_lens[b] - Nq + i (as in contiguous
    decode).

The result is the plain definition applied to each sequence's gathered keys
and values: attention_grouped with q_offset = seq_lens[b] - Nq.
"""

import numpy as np

from .attention import MASK_NONE, attention_grouped


def gather_pages(cache, block_table_row, seq_len, page_size):
    """Contiguous [seq_len, H_kv, D] rows of one sequence, position by position."""
    cache = np.asarray(cache)
    rows = [cache[int(block_table_row[j // page_size]), j % page_size] for j in range(seq_len)]
    if not rows:
        return np.zeros((0,) + cache.shape[2:], dtype=np.float64)
    return np.stack(rows).astype(np.float64)


def attention_paged(q, k_cache, v_cache, block_table, seq_lens, page_size, scale, mask_kind=MASK_NONE,
                    win_l=-1, win_r=-1):
    """O [B, H, Nq, D] and LSE [B, H, Nq] for queries q [B, H, Nq, D] (float64)."""
    q = np.asarray(q, dtype=np.float64)
    B, H, Nq, D = q.shape
    o = np.zeros_like(q)
    lse = np.full((B, H, Nq), -np.inf)
    for b in range(B):
        n = int(seq_lens[b])
        k = gather_pages(k_cache, block_table[b], n, page_size).transpose(1, 0, 2)[None]   # [1, H_kv, n, D]
        v = gather_pages(v_cache, block_table[b], n, page_size).transpose(1, 0, 2)[None]
        if n == 0:
            continue
        ob, lb = attention_grouped(q[b:b + 1], k, v, scale, mask_kind, win_l, win_r, q_offset=n - Nq)
        o[b] = ob[0]
        lse[b] = lb[0]
    return o, lse
