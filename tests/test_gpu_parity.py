"""CUDA path vs the CPU oracle, element by element, through the C ABI (needs a GB300)."""
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from checker import check, check_scores, visible_counts

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


def run_gpu(Q, case, repeat=1):
    import torch
    p = Q.make_problem(**W.problem_kwargs(case))
    ix = Q.Indexer(p)
    d = W.to_device(case)
    for _ in range(repeat):
        out = ix.run(**d)
    torch.cuda.synchronize()
    st, bits = ix.device_error()
    return out.cpu().numpy(), ix.score_lines().cpu().numpy(), st, bits


def assert_parity(Q, case, rows=None, scores=True):
    gpu_idx, gpu_scores, st, bits = run_gpu(Q, case)
    ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True, rows=rows)
    assert err == 0 and st == 0, (err, st, bits)
    vis = visible_counts(case, oracle)
    exact, checked, fails = check(gpu_idx, ora_idx, ora_scores, vis, case.sparse_count, rows=rows)
    assert not fails, fails[:5]
    if scores:
        worst = check_scores(gpu_scores, ora_scores, vis, rows=rows)
        assert worst <= 1.0, worst
    return exact, checked


# ---------------------------------------------------------------------------- the named workloads

@pytest.mark.parametrize("name", ["tiny_decode", "page_decode"])
def test_small_workloads(qli, name):
    exact, checked = assert_parity(qli, W.WORKLOADS[name]())
    assert checked > 0


def test_long_decode_full_size(qli):
    case = W.long_decode()
    assert_parity(qli, case)


def test_fp8_compressed_decode_full_size(qli):
    case = W.fp8_compressed_decode()
    assert_parity(qli, case)


def test_long_context_decode_sampled_rows(qli):
    """The long-context decode timed beside the workloads (32 rows of 64k-128k keys, the top-k's
    cluster form) at full size, checked on 8 of its rows (the oracle on all 3 M pairs takes
    minutes)."""
    case = W.long_context_decode()
    assert_parity(qli, case, rows=[0, 3, 7, 12, 18, 23, 27, 31])


def test_varlen_prefill_sampled_rows(qli):
    case = W.varlen_prefill()
    rng = np.random.default_rng(0)
    cum = np.concatenate([[0], case.seq_lens_q])
    rows = set(rng.choice(case.rows, 48, replace=False).tolist())
    for b in range(case.batch):                       # each sequence's first, k-th and last rows
        rows |= {int(cum[b]), int(min(cum[b] + 2047, cum[b + 1] - 1)), int(cum[b + 1] - 1)}
    assert_parity(qli, case, rows=sorted(rows))


# ---------------------------------------------------------------------------- seeded small shapes

SMALL = [
    # (name, kwargs)
    ("bs16_c1_m0", dict(batch=2, s1=1, seq_lens_k=[300, 17], block_size=16, sparse_count=64)),
    ("bs32_c2_m3", dict(batch=3, s1=3, seq_lens_k=[257, 1, 640], block_size=32, sparse_count=7,
                        sparse_mode=3, cmp_ratio=2)),
    ("bs64_c4_m3", dict(batch=2, s1=2, seq_lens_k=[1000, 129], block_size=64, sparse_count=100,
                        sparse_mode=3, cmp_ratio=4)),
    ("bs128_c8", dict(batch=2, s1=4, seq_lens_k=[4096, 385], block_size=128, sparse_count=512,
                      sparse_mode=3, cmp_ratio=8)),
    ("bs256_c16", dict(batch=1, s1=2, seq_lens_k=[8000], block_size=256, sparse_count=2048,
                       sparse_mode=0, cmp_ratio=16)),
    ("bs1024_c128", dict(batch=2, s1=1, seq_lens_k=[70000, 129], block_size=1024,
                         sparse_count=33, sparse_mode=3, cmp_ratio=128)),
    ("bs48_odd", dict(batch=2, s1=3, seq_lens_k=[700, 95], block_size=48, sparse_count=64,
                      sparse_mode=3)),
    ("bs80_c32", dict(batch=2, s1=1, seq_lens_k=[9000, 33], block_size=80, sparse_count=64,
                      sparse_mode=3, cmp_ratio=32)),
    ("sq_gt_sk", dict(batch=2, s1=4, seq_lens_k=[2, 130], block_size=16, sparse_count=16,
                      sparse_mode=3)),
    ("k1", dict(batch=2, s1=2, seq_lens_k=[500, 4000], block_size=64, sparse_count=1,
                sparse_mode=3)),
    ("sk0", dict(batch=3, s1=1, seq_lens_k=[0, 128, 127], block_size=64, sparse_count=8)),
    ("qlens", dict(batch=3, s1=4, q_lens=[4, 0, 1], seq_lens_k=[600, 600, 129], block_size=64,
                   sparse_count=200, sparse_mode=3)),
    ("fp8_f32", dict(batch=2, s1=2, qk_dtype=W.FP8, scale_dtype=W.F32, seq_lens_k=[3000, 257],
                     block_size=128, sparse_count=256, sparse_mode=3, cmp_ratio=4)),
    ("fp8_f16", dict(batch=2, s1=1, qk_dtype=W.FP8, scale_dtype=W.F16, seq_lens_k=[1500, 64],
                     block_size=32, sparse_count=100)),
    ("int8_f32", dict(batch=2, s1=1, scale_dtype=W.F32, seq_lens_k=[1500, 64], block_size=32,
                      sparse_count=100)),
    ("tnd_mixed", dict(layout_q="TND", q_lens=[5, 1, 0, 9], seq_lens_k=[300, 40, 10, 600],
                       block_size=32, sparse_count=64, sparse_mode=3)),
    ("tnd_mode0", dict(layout_q="TND", q_lens=[3, 2], seq_lens_k=[200, 1000], block_size=64,
                       sparse_count=128, sparse_mode=0, cmp_ratio=2)),
    ("k_ge_n", dict(batch=2, s1=2, seq_lens_k=[200, 2048], block_size=128, sparse_count=2048,
                    sparse_mode=3)),
    ("identity_table", dict(batch=3, s1=2, seq_lens_k=[513, 1, 256], block_size=128,
                            sparse_count=300, permute=False)),
    # 32 batches x 2 query groups = 64 groups (the metadata's one-warp path, both halves), empty
    # batches and sequences without keys
    ("groups64", dict(batch=32, s1=4, q_lens=[(i * 7) % 5 for i in range(32)],
                      seq_lens_k=[0 if i % 6 == 2 else 97 * i + 3 for i in range(32)], block_size=64,
                      sparse_count=96, sparse_mode=3)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[s[0] for s in SMALL])
def test_small_shapes(qli, name, kw):
    case = W.make_case(name, seed=zlib.crc32(name.encode()) % 1000, **kw)
    assert_parity(qli, case)


# ---------------------------------------------------------------------------- many rows per CTA
# Rows of at most 8192 keys and more rows than SMs: the two-per-SM top-k, each CTA taking every
# 304th row.  Consecutive rows of a CTA here alternate between long (> 4096 keys), mid, short and
# empty lines, so the next row's line is copied into either line buffer during a selection and
# into the row cache after one.
MANY = [
    ("many_k2048", dict(layout_q="TND", q_lens=[400, 400, 400, 400], seq_lens_k=[8000, 3000, 200, 6000],
                        block_size=128, sparse_count=2048, sparse_mode=3)),
    ("many_k64", dict(layout_q="TND", q_lens=[350, 1, 0, 600, 300], seq_lens_k=[8192, 4096, 50, 4000, 4500],
                      block_size=64, sparse_count=64, sparse_mode=3)),
    ("many_bsnd_k301", dict(batch=100, s1=4, seq_lens_k=[(i * 2654435761) % 8192 for i in range(100)],
                            block_size=64, sparse_count=301, sparse_mode=3)),
]


@pytest.mark.parametrize("name,kw", MANY, ids=[s[0] for s in MANY])
def test_many_rows_per_cta(qli, name, kw):
    case = W.make_case(name, seed=zlib.crc32(name.encode()) % 1000, **kw)
    assert case.rows > 2 * 152
    assert_parity(qli, case)


def test_negative_scales_and_weights(qli):
    case = W.make_case("neg", batch=2, s1=2, seq_lens_k=[700, 300], block_size=64,
                       sparse_count=100, sparse_mode=3, seed=5, scale_dtype=W.F32)
    rng = np.random.default_rng(1)
    case.q_scale *= np.where(rng.random(case.q_scale.shape) < 0.3, -1, 1).astype(np.float32)
    case.k_scale *= np.where(rng.random(case.k_scale.shape) < 0.3, -1, 1).astype(np.float32)
    case.weights *= np.where(rng.random(case.weights.shape) < 0.2, -1, 1).astype(np.float32)
    assert_parity(qli, case)


def test_int8_extremes_exact(qli):
    """All -128 / 127 codes: dots of +-2^21 and +-2^14 * 127 * ... must come out exact."""
    case = W.make_case("ext", batch=1, s1=1, seq_lens_k=[256], block_size=128, sparse_count=256,
                       seed=2, scale_dtype=W.F32)
    rng = np.random.default_rng(3)
    case.query[:] = np.where(rng.random(case.query.shape) < 0.5, -128, 127).astype(np.int8)
    case.key[:] = np.where(rng.random(case.key.shape) < 0.5, -128, 127).astype(np.int8)
    case.q_scale[:] = 1.0
    case.k_scale[:] = 1.0
    case.weights[:] = 0.0
    case.weights[0, 0, 0] = 1.0
    gpu_idx, gpu_scores, st, _ = run_gpu(qli, case)
    ora_idx, ora_scores, _ = oracle.score_topk(case, with_scores=True)
    assert st == 0
    assert np.array_equal(gpu_scores[0, :256], ora_scores[0, :256])   # integer dots, exact
    assert np.array_equal(gpu_idx, ora_idx)


def test_repeat_calls_same_result(qli):
    case = W.make_case("rep", batch=3, s1=2, seq_lens_k=[900, 5, 300], block_size=64,
                       sparse_count=64, sparse_mode=3, seed=8)
    a, _, _, _ = run_gpu(qli, case, repeat=1)
    b, _, _, _ = run_gpu(qli, case, repeat=3)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------- device-side faults

def test_bad_page_blanks_batch_and_reports(qli):
    case = W.make_case("badpage", batch=2, s1=1, seq_lens_k=[300, 300], block_size=64,
                       sparse_count=16, seed=4)
    case.block_table[1, 1] = case.num_blocks + 5
    gpu_idx, _, st, bits = run_gpu(qli, case)
    ora_idx, _, err = oracle.score_topk(case)
    assert err & oracle.ERR_PAGE
    assert st == 5 and bits & 2
    assert (gpu_idx[1] == -1).all()
    assert np.array_equal(gpu_idx, ora_idx)


def test_bad_page_in_long_rows_blanks_batch(qli):
    """Long rows (split over several CTAs when few rows share the GPU): a bad page in the last
    quarter of one batch's pages blanks that batch only."""
    case = W.make_case("badpage_long", batch=3, s1=1, seq_lens_k=[9000, 9000, 7000], block_size=64,
                       sparse_count=512, sparse_mode=3, seed=12)
    case.block_table[1, 130] = -7
    gpu_idx, _, st, bits = run_gpu(qli, case)
    ora_idx, _, err = oracle.score_topk(case)
    assert err & oracle.ERR_PAGE
    assert st == 5 and bits & 2
    assert (gpu_idx[1] == -1).all() and (gpu_idx[0] >= 0).all() and (gpu_idx[2] >= 0).all()
    assert np.array_equal(gpu_idx, ora_idx)


def test_bad_lengths_blank_batch_and_report(qli):
    case = W.make_case("badlen", batch=2, s1=2, q_lens=[2, 2], seq_lens_k=[300, 300],
                       block_size=64, sparse_count=16, seed=4)
    case.seq_lens_q = np.array([2, 3], np.int32)        # 3 > S1
    gpu_idx, _, st, bits = run_gpu(qli, case)
    ora_idx, _, err = oracle.score_topk(case)
    assert err & oracle.ERR_LENGTH
    assert st == 5 and bits & 1
    assert np.array_equal(gpu_idx, ora_idx)


# ---------------------------------------------------------------------------- top-k paths

def test_topk_all_equal_long_row(qli):
    """Every key identical: all scores tie, the sampled threshold keeps every key (more than the
    candidate buffer holds), so the exact fallback must pick the lowest indices."""
    case = W.make_case("ties", batch=1, s1=1, seq_lens_k=[6000], block_size=64, sparse_count=100,
                       seed=9)
    case.key[:] = case.key[0, 0]
    case.k_scale[:] = case.k_scale[0, 0]
    gpu_idx, _, st, _ = run_gpu(qli, case)
    assert st == 0
    assert gpu_idx[0].tolist() == list(range(100))


def test_topk_few_distinct_scores(qli):
    """Keys drawn from 7 distinct rows: long runs of exact ties around the k-th score."""
    case = W.make_case("few", batch=2, s1=1, seq_lens_k=[9000, 5000], block_size=128,
                       sparse_count=2048, sparse_mode=3, seed=10)
    rng = np.random.default_rng(10)
    pick = rng.integers(0, 7, size=case.key.shape[:2])
    protos = case.key[0, :7, 0].copy()
    case.key[:, :, 0] = protos[pick]
    case.k_scale[:] = np.float16(1.0)
    gpu_idx, _, st, _ = run_gpu(qli, case)
    ora_idx, _, _ = oracle.score_topk(case)
    assert st == 0
    assert np.array_equal(gpu_idx, ora_idx)     # exact ties resolve by index on both sides


@pytest.mark.parametrize("k", [40, 300, 512])
def test_topk_short_rows_with_ties(qli, k):
    """Rows of at most 512 keys (up to 256 keys each key's place is counted against the whole row), with keys drawn
    from 5 distinct rows so that runs of exact ties cross the k-th place; k below, inside and at
    or above the rows' lengths (then every key, in order, then -1)."""
    case = W.make_case("short_ties", batch=6, s1=2, seq_lens_k=[1, 2, 63, 256, 257, 512], block_size=64,
                       sparse_count=k, sparse_mode=3, seed=12)
    rng = np.random.default_rng(12)
    pick = rng.integers(0, 5, size=case.key.shape[:2])
    protos = case.key[0, :5, 0].copy()
    case.key[:, :, 0] = protos[pick]
    case.k_scale[:] = np.float16(1.0)
    gpu_idx, _, st, _ = run_gpu(qli, case)
    ora_idx, _, _ = oracle.score_topk(case)
    assert st == 0
    assert np.array_equal(gpu_idx, ora_idx)     # exact ties resolve by index on both sides


# ---------------------------------------------------------------------------- sparse_values

@pytest.mark.parametrize("name", ["page_decode", "fp8_compressed_decode", "long_decode"])
def test_sparse_values_are_the_indices_scores(qli, name):
    """return_value = 1: sparse_values holds each written index's score -- bit-equal to the kernel's
    own score line, within the row tolerance of the oracle's score -- and -inf beside -1."""
    import torch
    case = W.WORKLOADS[name]()
    p = qli.make_problem(**W.problem_kwargs(case), return_value=1)
    ix = qli.Indexer(p)
    d = W.to_device(case)
    idx = ix.run(**d).cpu().numpy()
    vals = ix.values.cpu().numpy()
    lines = ix.score_lines().cpu().numpy()
    torch.cuda.synchronize()
    assert ix.device_error()[0] == 0
    plain = qli.Indexer(qli.make_problem(**W.problem_kwargs(case)))
    assert np.array_equal(plain.run(**d).cpu().numpy(), idx)     # the indices do not change
    rows = range(idx.shape[0]) if idx.shape[0] <= 64 else range(0, idx.shape[0], 7)
    ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True, rows=list(rows))
    assert err == 0
    for r in rows:
        live = idx[r] >= 0
        assert np.isneginf(vals[r][~live]).all()
        assert np.array_equal(vals[r][live], lines[r][idx[r][live]])
        if not live.any():
            continue
        tau = 1e-5 * float(np.nanmax(ora_scores[r]))             # the row tolerance
        ref = ora_scores[r][idx[r][live]].astype(np.float64)
        assert np.all(np.abs(vals[r][live].astype(np.float64) - ref) <= tau), r


# ---------------------------------------------------------------------------- stride and mask rows

@pytest.mark.parametrize("kw,pad", [
    (dict(batch=3, s1=2, seq_lens_k=[700, 90, 1500], block_size=64, sparse_count=128, sparse_mode=3), 48),
    (dict(batch=2, s1=1, seq_lens_k=[5000, 333], block_size=16, sparse_count=512, sparse_mode=0), 4096),
    (dict(batch=2, s1=2, seq_lens_k=[9000, 4100], block_size=128, sparse_count=2048, sparse_mode=3,
          qk_dtype=W.FP8, scale_dtype=W.F32, cmp_ratio=4), 256),
])
def test_strided_key_pool_matches_oracle(qli, kw, pad):
    """README `stride` of key's first axis: pages `pad` junk elements apart, read by the 3-D
    tensor map with that page stride."""
    case = W.with_key_stride(W.make_case("strided", seed=31, **kw), pad, seed=7)
    assert case.key_stride == case.block_size * 128 + pad
    assert_parity(qli, case)


@pytest.mark.parametrize("kw", [
    dict(batch=3, s1=3, seq_lens_k=[4099, 1025, 37], block_size=64, sparse_count=256, sparse_mode=3,
         cmp_ratio=4),
    dict(layout_q="TND", q_lens=[5, 300, 64], seq_lens_k=[5, 300, 640], block_size=32, sparse_count=64,
         sparse_mode=3, cmp_ratio=8),
])
def test_complete_blocks_mask_matches_oracle(qli, kw):
    """The other reading of the causal rule under compression (only complete compressed blocks are
    visible: n = floor((p + 1) / cmp)) as a runtime flag, against the oracle's same switch."""
    import torch
    case = W.make_case("complete", seed=41, **kw)
    p = qli.make_problem(**W.problem_kwargs(case), mask_complete_blocks=1)
    ix = qli.Indexer(p)
    gpu_idx = ix.run(**W.to_device(case)).cpu().numpy()
    torch.cuda.synchronize()
    assert ix.device_error()[0] == 0
    ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True, complete_blocks_only=True)
    assert err == 0
    counts = visible_counts(case, oracle, complete_blocks_only=True)
    exact, checked, fails = check(gpu_idx, ora_idx, ora_scores, counts, case.sparse_count)
    assert not fails, fails[:5]
    # the flag changes the result for these shapes (some rows lose their partial block)
    ceil_idx, _, _ = oracle.score_topk(case)
    assert not np.array_equal(ceil_idx, ora_idx)


# ---------------------------------------------------------------------------- rows beyond the row cache

# The top-k keeps a row of up to 32768 scores in shared memory; longer rows take the path that
# samples and gathers from global memory.  These cases reach it with uncompressed keys.
LONG_ROWS = [
    ("long_m3", dict(batch=3, s1=1, seq_lens_k=[40000, 70000, 131072], block_size=128,
                     sparse_count=2048, sparse_mode=3)),
    ("long_m0_s2", dict(batch=2, s1=2, seq_lens_k=[33000, 65536], block_size=64,
                        sparse_count=2048, sparse_mode=0)),
    ("long_fp8_k777", dict(batch=2, s1=1, qk_dtype=W.FP8, scale_dtype=W.F32,
                           seq_lens_k=[50001, 32769], block_size=256, sparse_count=777,
                           sparse_mode=3)),
    # rows of every length in one problem: quarters of a cluster left empty, rows of at most 4096
    # keys (every key a candidate), a single key
    ("long_mixed", dict(batch=6, s1=1, seq_lens_k=[131072, 40001, 4096, 4097, 257, 1], block_size=64,
                        sparse_count=2048, sparse_mode=0)),
    ("long_mixed_k64", dict(batch=4, s1=1, seq_lens_k=[100000, 3, 70000, 33000], block_size=128,
                            sparse_count=64, sparse_mode=3)),
]


@pytest.mark.parametrize("name,kw", LONG_ROWS, ids=[s[0] for s in LONG_ROWS])
def test_rows_beyond_row_cache(qli, name, kw):
    case = W.make_case(name, seed=zlib.crc32(name.encode()) % 1000, **kw)
    assert case.max_seqlen_k > 32768
    assert_parity(qli, case)


def test_sparse_values_of_long_rows(qli):
    """return_value = 1 on rows beyond one CTA's row cache: each written index's score, read from
    the score line, and -inf beside -1."""
    import torch
    case = W.make_case("long_vals", batch=3, s1=1, seq_lens_k=[90000, 50000, 1000], block_size=64,
                       sparse_count=512, sparse_mode=3, seed=64)
    p = qli.make_problem(**W.problem_kwargs(case), return_value=1)
    ix = qli.Indexer(p)
    idx = ix.run(**W.to_device(case)).cpu().numpy()
    vals = ix.values.cpu().numpy()
    lines = ix.score_lines().cpu().numpy()
    torch.cuda.synchronize()
    assert ix.device_error()[0] == 0
    ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True)
    assert err == 0
    exact, checked, fails = check(idx, ora_idx, ora_scores, visible_counts(case, oracle), case.sparse_count)
    assert not fails, fails[:5]
    for r in range(case.rows):
        live = idx[r] >= 0
        assert np.array_equal(vals[r][live], lines[r][idx[r][live]])
        assert np.isneginf(vals[r][~live]).all()


def test_tnd_sequence_beyond_row_cache(qli):
    case = W.make_case("tnd_long", layout_q="TND", q_lens=[3, 2, 1], seq_lens_k=[40000, 5000, 36000],
                       block_size=128, sparse_count=2048, sparse_mode=3, seed=61)
    assert_parity(qli, case)


def test_all_equal_row_beyond_row_cache(qli):
    """Every key identical in rows of 40000 and 33000 keys: the sampled bound keeps every key, far
    more than the candidate buffer holds, so the exact selection must return the lowest indices."""
    case = W.make_case("ties_long", batch=2, s1=1, seq_lens_k=[40000, 33000], block_size=128,
                       sparse_count=2048, sparse_mode=0, seed=62)
    case.key[:] = case.key[0, 0]
    case.k_scale[:] = case.k_scale[0, 0]
    gpu_idx, _, st, _ = run_gpu(qli, case)
    assert st == 0
    for r in range(2):
        assert gpu_idx[r].tolist() == list(range(2048))
    ora_idx, _, _ = oracle.score_topk(case)
    assert np.array_equal(gpu_idx, ora_idx)


def test_few_distinct_scores_beyond_row_cache(qli):
    """Keys drawn from 5 distinct rows in a 60000-key row: long runs of exact ties at the cut."""
    case = W.make_case("few_long", batch=1, s1=1, seq_lens_k=[60000], block_size=128,
                       sparse_count=2048, sparse_mode=3, seed=63)
    rng = np.random.default_rng(63)
    pick = rng.integers(0, 5, size=case.key.shape[:2])
    protos = case.key[0, :5, 0].copy()
    case.key[:, :, 0] = protos[pick]
    case.k_scale[:] = np.float16(1.0)
    gpu_idx, _, st, _ = run_gpu(qli, case)
    ora_idx, _, _ = oracle.score_topk(case)
    assert st == 0
    assert np.array_equal(gpu_idx, ora_idx)
