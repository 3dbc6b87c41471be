"""The downstream sparse-attention gather on the GPU (qli_gather_kv) against the oracle: gathered
bytes and per-row counts identical, -1 and invalid indices zero-filled with their error bits, at
small and full sizes, after the indexer on the same stream (needs a GB300)."""
import numpy as np
import pytest

import oracle
import workloads as W
from checker import check, visible_counts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qli():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_token_block_gb300 import build as B
    B.build()
    import sparse_attention_token_block_gb300 as Q
    return Q


def _dev(a):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _gpu_gather(Q, case, idx, pool, entry_bytes, kv_stride=0, with_seq_lens_k=True):
    import torch
    p = Q.make_problem(**W.problem_kwargs(case))
    rows, k = idx.shape
    out = torch.full((rows, k, entry_bytes), 0xA5, dtype=torch.uint8, device="cuda")
    counts = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(64, dtype=torch.int32, device="cuda")
    Q.check(Q.workspace_init(ws), "workspace_init")
    Q.check(Q.gather_kv(p, _dev(case.seq_lens_q), _dev(case.seq_lens_k) if with_seq_lens_k else None,
                        _dev(case.block_table), _dev(idx), _dev(pool), entry_bytes, out, counts, kv_stride, ws),
            "gather_kv")
    st, bits = Q.get_device_error(ws)
    return out.cpu().numpy(), counts.cpu().numpy(), bits


CASES = {
    "bsnd": lambda: W.make_case("gb", batch=3, s1=2, seq_lens_k=[700, 90, 1500], block_size=64, sparse_count=128,
                                seed=2),
    "tnd": lambda: W.make_case("gt", layout_q="TND", q_lens=[3, 0, 5], seq_lens_k=[300, 50, 999], block_size=32,
                               sparse_count=64, seed=3),
    "cmp4": lambda: W.make_case("gc", batch=2, s1=3, seq_lens_k=[4001, 777], block_size=16, sparse_count=200,
                                cmp_ratio=4, seed=4),
    "k1": lambda: W.make_case("g1", batch=5, s1=1, seq_lens_k=[1, 2, 3, 40, 100], block_size=16, sparse_count=1,
                              seed=5),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("entry_bytes,pad", [(16, 0), (48, 32), (512, 0), (1152, 16), (4112, 0)])
def test_gather_matches_oracle(qli, name, entry_bytes, pad):
    case = CASES[name]()
    pool = W.kv_pool(case, entry_bytes, pad, seed=7)
    stride = case.block_size * entry_bytes + pad if pad else 0
    idx = W.random_indices(case, seed=entry_bytes)
    out, counts, bits = _gpu_gather(qli, case, idx, pool, entry_bytes, stride)
    ref, ref_counts, err = oracle.gather_kv(case, idx, pool, entry_bytes, stride)
    assert err == 0 and bits == 0
    assert np.array_equal(counts, ref_counts)
    assert np.array_equal(out, ref)


def test_largest_entry(qli):
    case = W.make_case("gl", batch=2, s1=1, seq_lens_k=[40, 17], block_size=16, sparse_count=8, seed=6)
    pool = W.kv_pool(case, 65536, 0, seed=8)
    idx = W.random_indices(case, seed=1)
    out, counts, bits = _gpu_gather(qli, case, idx, pool, 65536)
    ref, ref_counts, err = oracle.gather_kv(case, idx, pool, 65536)
    assert bits == err == 0 and np.array_equal(counts, ref_counts) and np.array_equal(out, ref)


def test_invalid_indices_and_pages(qli):
    case = W.make_case("ge", batch=2, s1=1, seq_lens_k=[100, 40], block_size=32, sparse_count=8, seed=5)
    pool = W.kv_pool(case, 32, 0, seed=6)
    idx = np.array([[0, 99, -1, -1, -1, -1, -1, -1],
                    [40, -5, 3, 63, 64, -1, 7, -1]], np.int32)
    for with_k in (True, False):
        out, counts, bits = _gpu_gather(qli, case, idx, pool, 32, with_seq_lens_k=with_k)
        ref, ref_counts, err = oracle.gather_kv(case, idx, pool, 32, use_seq_lens_k=with_k)
        assert bits == err and err != 0
        assert np.array_equal(counts, ref_counts) and np.array_equal(out, ref)
    case.block_table[0, 3] = case.num_blocks + 2
    out, counts, bits = _gpu_gather(qli, case, idx, pool, 32)
    ref, ref_counts, err = oracle.gather_kv(case, idx, pool, 32)
    assert bits == err == (oracle.ERR_LENGTH | oracle.ERR_PAGE)
    assert np.array_equal(counts, ref_counts) and np.array_equal(out, ref)


def test_tnd_rows_past_the_last_prefix_sum(qli):
    case = W.make_case("gp", layout_q="TND", q_lens=[2, 2], seq_lens_k=[64, 64], block_size=32, sparse_count=4,
                       seed=7)
    case.total_q = 6
    pool = W.kv_pool(case, 16, 0, seed=8)
    idx = np.full((6, 4), -1, np.int32)
    idx[:, 0] = 1
    idx[5, 0] = -1
    out, counts, bits = _gpu_gather(qli, case, idx, pool, 16)
    ref, ref_counts, err = oracle.gather_kv(case, idx, pool, 16)
    assert bits == err == oracle.ERR_LENGTH
    assert np.array_equal(counts, ref_counts) and np.array_equal(out, ref)


def test_rejects_bad_arguments(qli):
    import torch
    case = CASES["bsnd"]()
    p = qli.make_problem(**W.problem_kwargs(case))
    idx = _dev(W.random_indices(case, seed=1))
    pool = _dev(W.kv_pool(case, 64, 0, seed=1))
    out = torch.empty((case.rows, case.sparse_count, 64), dtype=torch.uint8, device="cuda")
    bt, slk = _dev(case.block_table), _dev(case.seq_lens_k)
    bad = lambda st: qli.STATUS_NAMES[st] == "QLI_ERR_INVALID_ARG"
    assert bad(qli.gather_kv(p, None, slk, bt, idx, pool, 24, out))           # not a multiple of 16
    assert bad(qli.gather_kv(p, None, slk, bt, idx, pool, 0, out))
    assert bad(qli.gather_kv(p, None, slk, bt, idx, pool, 65552, out))        # above 64 KiB
    assert bad(qli.gather_kv(p, None, slk, bt, idx, pool, 64, out, kv_stride=64 * 64 - 16))
    assert bad(qli.gather_kv(p, None, slk, bt, idx, pool, 64, out, kv_stride=64 * 64 + 8))
    assert bad(qli.gather_kv(p, None, slk, bt, idx, pool.data_ptr() + 8, 64, out))
    assert bad(qli.gather_kv(p, None, slk, bt, idx, pool, 64, out.data_ptr() + 4))
    assert bad(qli.gather_kv(p, None, slk, bt, None, pool, 64, out))
    assert qli.gather_kv(p, None, slk, bt, idx, pool, 64, out) == qli.QLI_OK
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["long_decode", "fp8_compressed_decode"])
def test_after_the_indexer_at_full_size(qli, name):
    """The decode workloads at full size: the indexer, then the gather of 512-byte entries on the
    same stream with no synchronisation between them; the GPU indices checked against the oracle,
    every gathered byte against the oracle's gather of those indices."""
    import torch
    case = W.WORKLOADS[name]()
    p = qli.make_problem(**W.problem_kwargs(case))
    ix = qli.Indexer(p)
    d = W.to_device(case)
    entry = 512
    pool = W.kv_pool(case, entry, 0, seed=11)
    out = torch.empty((case.rows, case.sparse_count, entry), dtype=torch.uint8, device="cuda")
    counts = torch.empty(case.rows, dtype=torch.int32, device="cuda")
    idx_dev = ix.run(**d)
    qli.check(qli.gather_kv(p, d["seq_lens_q"], d["seq_lens_k"], d["block_table"], idx_dev, _dev(pool), entry, out,
                            counts, 0, ix.workspace), "gather_kv")
    assert ix.device_error()[0] == qli.QLI_OK
    gpu_idx = idx_dev.cpu().numpy()
    ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True)
    assert err == 0
    _, _, fails = check(gpu_idx, ora_idx, ora_scores, visible_counts(case, oracle), case.sparse_count)
    assert not fails, fails[:5]
    ref, ref_counts, err = oracle.gather_kv(case, gpu_idx, pool, entry)
    assert err == 0
    assert np.array_equal(counts.cpu().numpy(), ref_counts)
    assert np.array_equal(out.cpu().numpy(), ref)


def test_after_a_plan_replay(qli):
    """The gather enqueued straight after an execution-plan replay (a CUDA graph whose last kernel
    is the top-k) reads that replay's indices."""
    import torch
    case = W.WORKLOADS["fp8_compressed_decode"]()
    p = qli.make_problem(**W.problem_kwargs(case))
    ix = qli.Indexer(p)
    d = W.to_device(case)
    plan = ix.plan(**d)
    entry = 256
    pool = _dev(W.kv_pool(case, entry, 0, seed=12))
    out = torch.empty((case.rows, case.sparse_count, entry), dtype=torch.uint8, device="cuda")
    counts = torch.empty(case.rows, dtype=torch.int32, device="cuda")
    ix.out.fill_(-1)                              # stale indices: the gather must see the replay's
    torch.cuda.synchronize()
    plan.launch()
    qli.check(qli.gather_kv(p, d["seq_lens_q"], d["seq_lens_k"], d["block_table"], ix.out, pool, entry, out,
                            counts, 0, ix.workspace), "gather_kv")
    torch.cuda.synchronize()
    assert ix.device_error()[0] == qli.QLI_OK
    gpu_idx = ix.out.cpu().numpy()
    assert (gpu_idx[:, 0] >= 0).all()
    ref, ref_counts, err = oracle.gather_kv(case, gpu_idx, pool.cpu().numpy(), entry)
    assert err == 0
    assert np.array_equal(counts.cpu().numpy(), ref_counts)
    assert np.array_equal(out.cpu().numpy(), ref)
    plan.close()
