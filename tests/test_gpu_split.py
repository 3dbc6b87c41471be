"""The top-k in two stages -- the split-local selection in the one-token score kernel, then the
merge of the splits' candidates -- against the CPU oracle, through the C ABI (needs a GB300).

The score kernel splits a row's key tiles over about 300 CTAs, so the cases are sized for what
each stage sees: a CTA's share of a row ("unit") is cut into chunks at aligned 4096-key
boundaries; a chunk longer than k keeps its exact top k, a shorter one keeps every key; the merge
takes the row's candidates when at most 24576 of them remain and otherwise orders the whole score
line."""
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from checker import check, check_scores, row_tau, visible_counts

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


def run(Q, case, split, return_value=0):
    import torch
    p = Q.make_problem(**W.problem_kwargs(case), split_topk=split, return_value=return_value)
    ix = Q.Indexer(p)
    d = W.to_device(case)
    out = ix.run(**d).cpu().numpy()
    vals = ix.values.cpu().numpy() if return_value else None
    torch.cuda.synchronize()
    st, bits = ix.device_error()
    return ix, out, vals, st, bits


def assert_split_parity(Q, case, rows=None):
    ix, gpu_idx, _, st, bits = run(Q, case, Q.SPLIT_ON)
    ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True, rows=rows)
    assert err == 0 and st == 0, (err, st, bits)
    vis = visible_counts(case, oracle)
    exact, checked, fails = check(gpu_idx, ora_idx, ora_scores, vis, case.sparse_count, rows=rows)
    assert not fails, fails[:5]
    worst = check_scores(ix.score_lines().cpu().numpy(), ora_scores, vis, rows=rows)
    assert worst <= 1.0, worst
    return ix, gpu_idx, ora_scores, vis


SPLIT = [
    # units of one or two tiles, k = 64: every unit selects; ragged rows around 4096
    ("k64_ragged", dict(batch=6, s1=1, seq_lens_k=[30000, 12345, 4097, 4096, 8191, 300], block_size=64,
                        sparse_count=64, sparse_mode=3)),
    # k = 1 and rows shorter than a tile
    ("k1", dict(batch=4, s1=1, seq_lens_k=[20000, 129, 1, 7000], block_size=16, sparse_count=1,
                sparse_mode=0)),
    # k above some units' length: those keep every key (tiles that point at the score line)
    ("k300_mixed", dict(batch=3, s1=1, seq_lens_k=[40000, 700, 90], block_size=128, sparse_count=300,
                        sparse_mode=3)),
    # fp8, fp32 scales, compressed causal keys
    ("fp8_c4_k100", dict(batch=3, s1=1, qk_dtype=W.FP8, scale_dtype=W.F32, seq_lens_k=[60000, 20001, 5],
                         block_size=32, sparse_count=100, sparse_mode=3, cmp_ratio=4)),
    # units of ~4.2k keys cut at aligned 4096-key boundaries, k = 512, merged candidates
    ("k512_chunks", dict(batch=16, s1=1, seq_lens_k=[60000 + 2731 * i for i in range(16)], block_size=64,
                         sparse_count=512, sparse_mode=0)),
    # k = 2048 with units of ~3.4k keys: rows of 32768 keys keep ~20k candidates (merged)
    ("k2048_merge", dict(batch=32, s1=1, seq_lens_k=[32768] * 32, block_size=64, sparse_count=2048,
                         sparse_mode=3)),
    # k = 2048, rows of 70000 keys: more candidates than the merge holds -> the score line
    ("k2048_fallback", dict(batch=20, s1=1, seq_lens_k=[70000] * 20, block_size=128, sparse_count=2048,
                            sparse_mode=0)),
]


@pytest.mark.parametrize("name,kw", SPLIT, ids=[s[0] for s in SPLIT])
def test_split_topk_matches_oracle(qli, name, kw):
    case = W.make_case(name, seed=zlib.crc32(name.encode()) % 1000, **kw)
    assert_split_parity(qli, case)


def test_split_candidates_hold_every_clear_winner(qli):
    """The split-local stage itself: every candidate's code is the score line's code at its index,
    the candidates come in index order, and every key whose oracle score is more than twice the row
    tolerance above the row's k-th is among the candidates (fewer than k keys of the row can then
    have a higher GPU score, so its chunk must keep it)."""
    case = W.make_case("cands", batch=8, s1=1, seq_lens_k=[50000, 33333, 20000, 9000, 4097, 4096, 100, 2],
                       block_size=64, sparse_count=256, sparse_mode=3, seed=71)
    ix, gpu_idx, ora_scores, vis = assert_split_parity(qli, case)
    code, idx, info = (t.cpu().numpy() for t in ix.split_candidates())
    import torch
    lines = ix.workspace.view(torch.uint8)[256:256 + case.rows * code.shape[1] * 4]
    lines = lines.view(torch.int32).view(case.rows, code.shape[1]).cpu().numpy()
    k = case.sparse_count
    selected_tiles = 0
    for r in range(case.rows):
        n = int(vis[r])
        if n == 0:
            continue
        cand = []
        for t in range((n + 127) // 128):
            w = int(info[r, t]) & 0xFFFFFFFF
            c = w & 0x7FFFFFFF
            assert c <= 128
            if w & 0x80000000:
                selected_tiles += 1
                ii = idx[r, 128 * t:128 * t + c].astype(np.int64)
                assert np.array_equal(code[r, 128 * t:128 * t + c], lines[r, ii])
                cand.extend(ii.tolist())
            else:
                assert c == min(128, n - 128 * t)             # a kept tile: all its visible keys
                cand.extend(range(128 * t, 128 * t + c))
        cand = np.asarray(cand)
        assert np.all(np.diff(cand) > 0)                      # index order, no repeats
        assert cand.min() >= 0 and cand.max() < n
        s = np.asarray(ora_scores[r][:n], dtype=np.float64)
        if n > k:
            kth = np.sort(s)[::-1][k - 1]
            winners = np.nonzero(s > kth + 2 * row_tau(ora_scores[r], n))[0]
            assert np.isin(winners, cand).all(), r
    assert selected_tiles > 0                                 # some chunks did select


def test_split_ties_resolve_by_index(qli):
    """Keys drawn from 5 distinct rows: every chunk's cut falls in a run of exact ties, resolved by
    index inside the chunk's selection and again in the merge."""
    case = W.make_case("split_ties", batch=4, s1=1, seq_lens_k=[20000, 9000, 4096, 33000], block_size=128,
                       sparse_count=64, sparse_mode=0, seed=72)
    rng = np.random.default_rng(72)
    pick = rng.integers(0, 5, size=case.key.shape[:2])
    protos = case.key[0, :5, 0].copy()
    case.key[:, :, 0] = protos[pick]
    case.k_scale[:] = np.float16(1.0)
    _, gpu_idx, _, st, _ = run(qli, case, qli.SPLIT_ON)
    ora_idx, _, _ = oracle.score_topk(case)
    assert st == 0
    assert np.array_equal(gpu_idx, ora_idx)


def test_split_all_equal_keys(qli):
    """Every score equal: each chunk keeps its lowest indices and the row its lowest k."""
    case = W.make_case("split_equal", batch=2, s1=1, seq_lens_k=[9000, 5000], block_size=64, sparse_count=100,
                       seed=73)
    case.key[:] = case.key[0, 0]
    case.k_scale[:] = case.k_scale[0, 0]
    _, gpu_idx, _, st, _ = run(qli, case, qli.SPLIT_ON)
    assert st == 0
    for r in range(2):
        assert gpu_idx[r].tolist() == list(range(100))


def test_split_values_and_same_indices_as_one_stage(qli):
    """return_value = 1 with the split-local selection: the same indices as the one-stage top-k and
    each index's score from the score line."""
    case = W.make_case("split_vals", batch=5, s1=1, seq_lens_k=[25000, 18000, 9000, 700, 40000], block_size=64,
                       sparse_count=128, sparse_mode=3, seed=74)
    ix, idx, vals, st, _ = run(qli, case, qli.SPLIT_ON, return_value=1)
    assert st == 0
    _, idx_off, vals_off, st2, _ = run(qli, case, qli.SPLIT_OFF, return_value=1)
    assert st2 == 0
    assert np.array_equal(idx, idx_off)
    assert np.array_equal(vals, vals_off)
    lines = ix.score_lines().cpu().numpy()
    for r in range(case.rows):
        live = idx[r] >= 0
        assert np.array_equal(vals[r][live], lines[r][idx[r][live]])
        assert np.isneginf(vals[r][~live]).all()


def test_split_request_ignored_for_query_groups(qli):
    """S1 > 1 (query groups of several tokens): the request is ignored and the result is the
    oracle's."""
    case = W.make_case("split_groups", batch=2, s1=3, seq_lens_k=[9000, 4000], block_size=64, sparse_count=64,
                       sparse_mode=3, seed=75)
    assert_split_parity(qli, case)


def test_split_plan_replay(qli):
    """The execution plan (one CUDA-graph replay per call) with the split-local selection gives the
    direct call's indices."""
    import torch
    case = W.make_case("split_plan", batch=6, s1=1, seq_lens_k=[30000, 20000, 10000, 5000, 4096, 1], block_size=64,
                       sparse_count=256, sparse_mode=3, seed=76)
    p = qli.make_problem(**W.problem_kwargs(case), split_topk=qli.SPLIT_ON)
    ix = qli.Indexer(p)
    d = W.to_device(case)
    ref = ix.run(**d).clone()
    plan = ix.plan(**d)
    ix.out.fill_(-7)
    plan.launch()
    torch.cuda.synchronize()
    assert ix.device_error()[0] == 0
    assert torch.equal(ix.out, ref)
    ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True)
    assert err == 0
    exact, checked, fails = check(ref.cpu().numpy(), ora_idx, ora_scores, visible_counts(case, oracle),
                                  case.sparse_count)
    assert not fails, fails[:5]
