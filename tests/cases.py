"""Small hand-built cases for the tests (explicit arrays instead of random draws)."""
from __future__ import annotations

import numpy as np

import workloads as W


def explicit_case(*, q_rows, keys, q_scale, k_scale, weights, block_size=16, sparse_count=3,
                  sparse_mode=0, cmp_ratio=1, seq_len_k=None, s1=None, seq_lens_q=None,
                  scale_dtype=W.F16, qk_dtype=W.INT8, block_table=None, num_blocks=None):
    """One BSND batch.  ``q_rows[r][h]`` is a short list (the first dims of head h of row r; the
    rest are zero); ``keys[j]`` likewise for compressed key j; ``q_scale[r][h]``/``weights[r][h]``
    are dicts head -> value (missing heads are 0); ``k_scale[j]`` per key."""
    H, D = W.NUM_HEADS_Q, W.HEAD_DIM
    s1 = len(q_rows) if s1 is None else s1
    nkeys = len(keys)
    if seq_len_k is None:
        seq_len_k = nkeys * cmp_ratio
    pages = max(1, -(-nkeys // block_size))
    if num_blocks is None:
        num_blocks = pages
    qdt = np.int8 if qk_dtype == W.INT8 else np.uint8
    query = np.zeros((1, s1, H, D), dtype=qdt)
    key = np.zeros((num_blocks, block_size, 1, D), dtype=qdt)
    sdt = np.float16 if scale_dtype == W.F16 else np.float32
    qs = np.zeros((1, s1, H), dtype=sdt)
    ws = np.zeros((1, s1, H), dtype=sdt)
    ks = np.zeros((num_blocks, block_size, 1), dtype=sdt)
    if block_table is None:
        block_table = np.arange(pages, dtype=np.int32).reshape(1, -1)
    block_table = np.asarray(block_table, dtype=np.int32).reshape(1, -1)
    for r, heads in enumerate(q_rows):
        for h, vec in heads.items():
            query[0, r, int(h), :len(vec)] = vec
    for r in range(len(q_rows)):
        for h, v in q_scale[r].items():
            qs[0, r, int(h)] = v
        for h, v in weights[r].items():
            ws[0, r, int(h)] = v
    for j, vec in enumerate(keys):
        pg = block_table[0, j // block_size]
        key[pg, j % block_size, 0, :len(vec)] = vec
        ks[pg, j % block_size, 0] = k_scale[j]
    slq = None if seq_lens_q is None else np.asarray(seq_lens_q, dtype=np.int32)
    return W.Case(name="explicit", layout_q="BSND", qk_dtype=qk_dtype, scale_dtype=scale_dtype,
                  batch=1, s1=s1, total_q=0, block_size=block_size, num_blocks=num_blocks,
                  max_blocks_per_seq=block_table.shape[1], sparse_count=sparse_count,
                  sparse_mode=sparse_mode, cmp_ratio=cmp_ratio, query=query, key=key,
                  weights=ws, q_scale=qs, k_scale=ks, seq_lens_q=slq,
                  seq_lens_k=np.array([seq_len_k], dtype=np.int32), block_table=block_table)


def logical_keys(case, b):
    """Gather batch b's compressed keys in logical order through the block_table: [Lc, D], [Lc]."""
    lc = -(-int(case.seq_lens_k[b]) // case.cmp_ratio)
    j = np.arange(lc)
    pages = case.block_table[b, j // case.block_size]
    slots = j % case.block_size
    return case.key[pages, slots, 0, :], case.k_scale[pages, slots, 0]
