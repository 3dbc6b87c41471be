"""Pins of the oracle's downstream sparse-attention gather: a case worked by hand, numpy's fancy
indexing through the block_table as an independent formulation (BSND and TND, contiguous and
strided pools), the padding and error conventions, and the chain from the oracle's own indices."""
import numpy as np

import oracle
import workloads as W


def _numpy_gather(case, idx, pool, entry_bytes, stride):
    """The same gather by vectorised indexing: row -> batch by arithmetic (BSND) or searchsorted on
    the prefix sums (TND), then byte offsets page * stride + slot * entry_bytes."""
    rows, k = idx.shape
    r = np.arange(rows)
    if case.layout_q == "BSND":
        b = r // case.s1
    else:
        b = np.searchsorted(case.seq_lens_q, r, side="right")
    j = idx.astype(np.int64)
    valid = j >= 0
    jj = np.where(valid, j, 0)
    page = case.block_table[b[:, None], jj // case.block_size].astype(np.int64)
    off = page * stride + (jj % case.block_size) * entry_bytes
    flat = pool.reshape(-1)
    out = flat[off[..., None] + np.arange(entry_bytes)]
    out[~valid] = 0
    return out, valid.sum(axis=1).astype(np.int32)


def test_hand_worked_example():
    # two pages of two 16-byte entries plus a third page; byte t of slot s of page p is 32p + 16s + t
    case = W.make_case("g", batch=1, s1=1, seq_lens_k=[4], block_size=16, sparse_count=4, seed=0)
    case.block_size = 2
    case.num_blocks = 3
    case.max_blocks_per_seq = 2
    case.block_table = np.array([[2, 0]], np.int32)
    pool = np.arange(96, dtype=np.uint8).reshape(3, 32)
    idx = np.array([[3, 0, -1, 2]], np.int32)
    out, counts, err = oracle.gather_kv(case, idx, pool, 16)
    assert err == 0 and counts.tolist() == [3]
    # j = 3: page table[1] = 0, slot 1 -> bytes 16..31;  j = 0: page 2, slot 0 -> bytes 64..79
    assert out[0, 0].tolist() == list(range(16, 32))
    assert out[0, 1].tolist() == list(range(64, 80))
    assert out[0, 2].tolist() == [0] * 16
    assert out[0, 3].tolist() == list(range(0, 16))        # j = 2: page 0, slot 0


def test_matches_numpy_indexing_bsnd_and_tnd():
    cases = [W.make_case("gb", batch=3, s1=2, seq_lens_k=[700, 90, 1500], block_size=64, sparse_count=128, seed=2),
             W.make_case("gt", layout_q="TND", q_lens=[3, 0, 5], seq_lens_k=[300, 50, 999], block_size=32,
                         sparse_count=64, seed=3)]
    for case in cases:
        for entry_bytes, pad in ((16, 0), (48, 32), (1152, 0)):
            pool = W.kv_pool(case, entry_bytes, pad, seed=4)
            stride = case.block_size * entry_bytes + pad
            idx = W.random_indices(case, seed=entry_bytes + pad)
            out, counts, err = oracle.gather_kv(case, idx, pool, entry_bytes, stride if pad else 0)
            ref, ref_counts = _numpy_gather(case, idx, pool, entry_bytes, stride)
            assert err == 0
            assert np.array_equal(out, ref)
            assert np.array_equal(counts, ref_counts)


def test_errors_give_zero_entries():
    case = W.make_case("ge", batch=2, s1=1, seq_lens_k=[100, 40], block_size=32, sparse_count=8, seed=5)
    pool = W.kv_pool(case, 32, 0, seed=6)
    lc1 = 40
    idx = np.array([[0, 99, -1, -1, -1, -1, -1, -1],
                    [lc1, -5, 3, -1, -1, -1, -1, -1]], np.int32)
    out, counts, err = oracle.gather_kv(case, idx, pool, 32)
    assert err == oracle.ERR_LENGTH                   # j = Lc of batch 1, and j = -5
    assert counts.tolist() == [2, 1]
    assert not out[1, 0].any() and not out[1, 1].any() and out[1, 2].any()
    # without seq_lens_k only the block_table's capacity bounds j: j = 40 of batch 1 is read
    out2, counts2, err2 = oracle.gather_kv(case, idx, pool, 32, use_seq_lens_k=False)
    assert err2 == oracle.ERR_LENGTH and counts2.tolist() == [2, 2]
    # a page outside the pool
    case.block_table[0, 3] = case.num_blocks
    out3, counts3, err3 = oracle.gather_kv(case, idx, pool, 32)
    assert err3 == oracle.ERR_LENGTH | oracle.ERR_PAGE and counts3.tolist() == [1, 1]
    assert not out3[0, 1].any()


def test_tnd_rows_past_the_last_prefix_sum():
    case = W.make_case("gp", layout_q="TND", q_lens=[2, 2], seq_lens_k=[64, 64], block_size=32, sparse_count=4,
                       seed=7)
    case.total_q = 6                                  # rows 4 and 5 belong to no batch
    pool = W.kv_pool(case, 16, 0, seed=8)
    idx = np.full((6, 4), -1, np.int32)
    idx[:, 0] = 1
    idx[5, 0] = -1
    out, counts, err = oracle.gather_kv(case, idx, pool, 16)
    assert err == oracle.ERR_LENGTH
    assert counts.tolist() == [1, 1, 1, 1, 0, 0]


def test_chain_from_the_oracles_indices():
    case = W.make_case("gc", batch=4, s1=2, seq_lens_k=[3000, 1717, 260, 97], block_size=128, sparse_count=256,
                       sparse_mode=3, seed=9)
    idx, _, err = oracle.score_topk(case)
    assert err == 0
    pool = W.kv_pool(case, 64, 16, seed=10)
    out, counts, err = oracle.gather_kv(case, idx, pool, 64, case.block_size * 64 + 16)
    assert err == 0
    assert np.array_equal(counts, (idx >= 0).sum(axis=1))
    ref, _ = _numpy_gather(case, idx, pool, 64, case.block_size * 64 + 16)
    assert np.array_equal(out, ref)
