"""Pins of the CPU oracle to things other than itself.

Each test ties one part of the oracle to the README's definition through a hand-worked value, a
closed form, a special case that reduces to a library routine, brute-force enumeration or an
invariant, so that a dropped term, a wrong sign, a wrong index or a transposed operand fails here.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as W
from cases import explicit_case, logical_keys

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_two_heads.json")


# ---------------------------------------------------------------------------- number formats

def test_half_to_float_matches_numpy_on_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(c)) for c in codes], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_decode_matches_torch_on_all_codes():
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


# ---------------------------------------------------------------------------- hand-worked values

def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("which", [0, 1])
@pytest.mark.parametrize("scale_dtype", [W.F16, W.F32])
def test_hand_worked_scores_and_topk(which, scale_dtype):
    g = _golden()
    c = g["cases"][which]
    for k, expect in c["topk"].items():
        case = explicit_case(q_rows=[g["q"]], keys=g["k"], q_scale=[g["q_scale"]],
                             k_scale=g["k_scale"], weights=[c["weights"]], sparse_count=int(k),
                             scale_dtype=scale_dtype)
        idx, scores, err = oracle.score_topk(case, with_scores=True, nthreads=1)
        assert err == 0
        assert idx[0].tolist() == expect
        assert scores[0, :3].tolist() == c["scores"]


def test_hand_worked_mask_counts():
    m = _golden()["mask"]
    dummy = explicit_case(q_rows=[{}], keys=[[0]], q_scale=[{}], k_scale=[0], weights=[{}],
                          sparse_mode=3, cmp_ratio=m["cmp_ratio"])
    sq, sk = m["rows"], m["seq_len_k"]
    got = [oracle.visible(dummy, sq, sk, r) for r in range(sq)]
    assert got == m["visible_started_blocks"]
    got = [oracle.visible(dummy, sq, sk, r, complete_blocks_only=True) for r in range(sq)]
    assert got == m["visible_complete_blocks"]
    dummy.sparse_mode = 0
    assert [oracle.visible(dummy, sq, sk, r) for r in range(sq)] == m["visible_mode0"]


# ---------------------------------------------------------------------------- closed forms

def test_int8_extreme_dot_is_exact():
    # every product (-128)(-128) = 2^14, 128 of them: 2^21, with unit scales and weight on head 0
    case = explicit_case(q_rows=[{0: [-128] * 128}], keys=[[-128] * 128, [127] * 128],
                         q_scale=[{0: 1.0}], k_scale=[1.0, 1.0], weights=[{0: 1.0}],
                         sparse_count=2)
    idx, scores, _ = oracle.score_topk(case, with_scores=True, nthreads=1)
    assert scores[0, 0] == 2.0 ** 21
    assert scores[0, 1] == 0.0  # 128 * (-128 * 127) < 0, removed by the ReLU
    assert idx[0].tolist() == [0, 1]


def test_single_dim_closed_form():
    # q_0 = alpha * e_0: dot with K_j is alpha * K_j[0]; score = relu(alpha * K_j[0] * sQ * sK) * W
    rng = np.random.default_rng(7)
    kv = rng.integers(-128, 128, size=40)
    alpha = 3
    case = explicit_case(q_rows=[{0: [alpha]}], keys=[[int(v)] for v in kv],
                         q_scale=[{0: 0.25}], k_scale=[2.0] * 40, weights=[{0: 1.0}],
                         sparse_count=40)
    idx, scores, _ = oracle.score_topk(case, with_scores=True, nthreads=1)
    expect = [max(0.0, 0.25 * 2.0 * alpha * int(v)) for v in kv]
    assert scores[0, :40].tolist() == expect
    order = sorted(range(40), key=lambda j: (-expect[j], j))
    assert idx[0].tolist() == order


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_one_hot_weight_reduces_to_matvec_argsort(seed):
    """W one-hot on head h0, unit scales: score_j = ReLU(K_j . q_h0), so the top-k is a sort of a
    matrix-vector product (numpy) through the block_table gather."""
    case = W.make_case("mv", batch=2, s1=1, seq_lens_k=[150, 77], block_size=16, sparse_count=50,
                       seed=seed)
    h0 = 5 + seed
    case.weights[:] = 0
    case.weights[:, :, h0] = 1
    case.q_scale[:] = 1
    case.k_scale[:] = 1
    idx, scores, _ = oracle.score_topk(case, with_scores=True, nthreads=2)
    for b in range(2):
        keys, _ = logical_keys(case, b)
        mv = keys.astype(np.int64) @ case.query[b, 0, h0].astype(np.int64)
        ref = np.maximum(mv, 0).astype(np.float64)
        n = len(ref)
        assert np.array_equal(scores[b, :n].astype(np.float64), ref)
        order = sorted(range(n), key=lambda j: (-ref[j], j))[:50]
        assert idx[b].tolist() == order


def test_e4m3_dot_matches_exact_rational_sum():
    rng = np.random.default_rng(11)
    case = W.make_case("fp8", batch=1, s1=1, qk_dtype=W.FP8, scale_dtype=W.F32,
                       seq_lens_k=[33], block_size=16, sparse_count=33, seed=3)
    case.weights[:] = 0
    case.weights[0, 0, 9] = 1
    case.q_scale[:] = 1
    case.k_scale[:] = 1
    idx, scores, _ = oracle.score_topk(case, with_scores=True, nthreads=1)
    keys, _ = logical_keys(case, 0)
    dec = {c: Fraction(oracle.e4m3_value(c)) for c in range(256) if c & 0x7F != 0x7F}
    q = case.query[0, 0, 9]
    for j in range(33):
        exact = sum(dec[int(a)] * dec[int(b)] for a, b in zip(q, keys[j]))
        want = np.float32(float(max(exact, 0)))  # one rounding of the exact sum
        assert scores[0, j] == want, j
    del rng


# ---------------------------------------------------------------------------- mask by enumeration

@pytest.mark.parametrize("cmp_ratio", [1, 2, 4, 8, 16, 32, 64, 128])
def test_visible_counts_by_enumeration(cmp_ratio):
    dummy = explicit_case(q_rows=[{}], keys=[[0]], q_scale=[{}], k_scale=[0], weights=[{}],
                          sparse_mode=3, cmp_ratio=cmp_ratio)
    for sk in range(0, 41):
        lc = -(-sk // cmp_ratio)
        # positions each compressed key covers, by listing them
        covers = [[t for t in range(sk) if t // cmp_ratio == j] for j in range(lc)]
        for sq in range(0, 6):
            for r in range(sq):
                p = sk - sq + r
                started = sum(1 for cov in covers if cov and cov[0] <= p)
                complete = sum(1 for j in range(lc) if (j + 1) * cmp_ratio - 1 <= p)
                dummy.sparse_mode = 3
                assert oracle.visible(dummy, sq, sk, r) == started
                assert oracle.visible(dummy, sq, sk, r, complete_blocks_only=True) == complete
                dummy.sparse_mode = 0
                assert oracle.visible(dummy, sq, sk, r) == lc
            dummy.sparse_mode = 3
            assert oracle.visible(dummy, sq, sk, sq) == 0  # dead row


@pytest.mark.parametrize("mode,cmp_ratio", [(0, 1), (3, 1), (3, 4), (3, 3), (0, 8)])
def test_output_is_visible_prefix_permutation(mode, cmp_ratio):
    """With k >= n every row outputs a permutation of 0..n-1 followed by -1s."""
    case = W.make_case("perm", batch=3, s1=5, q_lens=[5, 3, 0], seq_lens_k=[40, 9, 17],
                       block_size=16, sparse_count=64, sparse_mode=mode, cmp_ratio=cmp_ratio,
                       seed=4)
    idx, _, err = oracle.score_topk(case, nthreads=2)
    assert err == 0
    for b in range(3):
        sq, sk = int(case.seq_lens_q[b]), int(case.seq_lens_k[b])
        lc = -(-sk // cmp_ratio)
        for r in range(5):
            row = idx[b * 5 + r]
            if r >= sq:
                n = 0
            elif mode == 0:
                n = lc
            else:
                p = sk - sq + r
                n = min(lc, sum(1 for j in range(lc) if j * cmp_ratio <= p))
            assert sorted(row[:n].tolist()) == list(range(n))
            assert (row[n:] == -1).all()


# ---------------------------------------------------------------------------- invariants

def _small(seed=0, **kw):
    args = dict(batch=2, s1=3, seq_lens_k=[300, 130], block_size=32, sparse_count=37,
                sparse_mode=3, seed=seed)
    args.update(kw)
    return W.make_case("inv", **args)


def test_scores_nonnegative_when_weights_nonnegative():
    case = _small(1)
    _, scores, _ = oracle.score_topk(case, with_scores=True)
    s = scores[~np.isnan(scores)]
    assert s.size > 0 and (s >= 0).all() and (s > 0).any()


@pytest.mark.parametrize("what", ["weights", "k_scale"])
def test_power_of_two_scaling_doubles_scores_and_keeps_order(what):
    case = _small(2)
    idx0, s0, _ = oracle.score_topk(case, with_scores=True)
    arr = getattr(case, what)
    setattr(case, what, (arr.astype(np.float32) * 2).astype(arr.dtype))
    idx1, s1, _ = oracle.score_topk(case, with_scores=True)
    assert np.array_equal(idx0, idx1)
    ok = ~np.isnan(s0)
    assert np.array_equal(s1[ok], s0[ok] * 2)


def test_page_permutation_leaves_output_unchanged():
    case = _small(3)
    idx0, _, _ = oracle.score_topk(case)
    rng = np.random.default_rng(99)
    perm = rng.permutation(case.num_blocks)          # new position of each old page
    key = np.empty_like(case.key)
    ks = np.empty_like(case.k_scale)
    key[perm] = case.key
    ks[perm] = case.k_scale
    table = np.where(case.block_table >= 0, perm[np.maximum(case.block_table, 0)], -1)
    case.key, case.k_scale, case.block_table = key, ks, table.astype(np.int32)
    idx1, _, _ = oracle.score_topk(case)
    assert np.array_equal(idx0, idx1)


@pytest.mark.parametrize("pad", [16, 4096])
def test_key_stride_only_moves_the_pages(pad):
    """README parameter table, `stride` of key's first axis: a pool whose pages sit `pad` junk
    elements apart gives exactly the contiguous pool's scores and indices (reading the junk, or a
    page at the contiguous offset, would change them)."""
    case = _small(5)
    idx0, s0, _ = oracle.score_topk(case, with_scores=True)
    strided = W.with_key_stride(case, pad, seed=pad)
    assert strided.key_stride == case.block_size * 128 + pad
    idx1, s1, _ = oracle.score_topk(strided, with_scores=True)
    assert np.array_equal(idx0, idx1)
    assert np.array_equal(s0, s1, equal_nan=True)


def test_duplicate_keys_tie_in_index_order():
    case = _small(4, batch=1, s1=1, seq_lens_k=[64], sparse_count=64, sparse_mode=0)
    case.key[:] = case.key[0, 0]          # every key identical
    case.k_scale[:] = case.k_scale[0, 0]
    idx, scores, _ = oracle.score_topk(case, with_scores=True)
    assert idx[0].tolist() == list(range(64))
    assert len(set(scores[0, :64].tolist())) == 1


def test_tnd_single_sequence_equals_bsnd():
    tnd = W.make_case("tnd", layout_q="TND", q_lens=[7], seq_lens_k=[200], block_size=32,
                      sparse_count=50, sparse_mode=3, seed=6)
    bsnd = W.Case(**{**tnd.__dict__, "layout_q": "BSND", "s1": 7, "total_q": 0,
                     "query": tnd.query.reshape(1, 7, 64, 128),
                     "weights": tnd.weights.reshape(1, 7, 64),
                     "q_scale": tnd.q_scale.reshape(1, 7, 64),
                     "seq_lens_q": np.array([7], np.int32)})
    a, _, _ = oracle.score_topk(tnd)
    b, _, _ = oracle.score_topk(bsnd)
    assert np.array_equal(a, b)


def test_tnd_rows_follow_prefix_sums():
    """TND batch b owns rows [cum[b-1], cum[b]); checked against per-sequence BSND runs."""
    lens = [3, 0, 5]
    tnd = W.make_case("tnd3", layout_q="TND", q_lens=lens, seq_lens_k=[50, 20, 70],
                      block_size=16, sparse_count=80, sparse_mode=3, seed=8)
    a, _, _ = oracle.score_topk(tnd)
    row = 0
    for b, L in enumerate(lens):
        if L == 0:
            continue
        sub = W.Case(**{**tnd.__dict__, "layout_q": "BSND", "batch": 1, "s1": L, "total_q": 0,
                        "query": tnd.query[row:row + L].reshape(1, L, 64, 128),
                        "weights": tnd.weights[row:row + L].reshape(1, L, 64),
                        "q_scale": tnd.q_scale[row:row + L].reshape(1, L, 64),
                        "seq_lens_q": None, "seq_lens_k": tnd.seq_lens_k[b:b + 1],
                        "block_table": tnd.block_table[b:b + 1]})
        s, _, _ = oracle.score_topk(sub)
        assert np.array_equal(a[row:row + L], s)
        row += L


# ---------------------------------------------------------------------------- error conventions

def test_bad_page_blanks_the_batch():
    case = _small(5)
    case.block_table[1, 2] = case.num_blocks + 3
    idx, _, err = oracle.score_topk(case)
    assert err & oracle.ERR_PAGE
    assert (idx[3:6] == -1).all()
    assert (idx[:3] != -1).any()


def test_bad_lengths_blank_the_batch():
    case = _small(6, q_lens=[3, 4])            # 4 > S1 = 3
    idx, _, err = oracle.score_topk(case)
    assert err & oracle.ERR_LENGTH
    assert (idx[3:6] == -1).all()
    case = _small(6)
    case.seq_lens_k = np.array([300, 10 ** 6], np.int32)   # beyond the block_table's capacity
    idx, _, err = oracle.score_topk(case)
    assert err & oracle.ERR_LENGTH and (idx[3:6] == -1).all()


def test_bad_tnd_prefix_sums_blank_every_row():
    case = W.make_case("tndbad", layout_q="TND", q_lens=[3, 4], seq_lens_k=[40, 40],
                       block_size=16, sparse_count=8, sparse_mode=3, seed=9)
    idx, _, err = oracle.score_topk(case)
    assert err == 0 and (idx != -1).any()
    case.seq_lens_q = np.array([5, 3], np.int32)     # decreasing
    idx, _, err = oracle.score_topk(case)
    assert err & oracle.ERR_LENGTH and (idx == -1).all()


def test_fast_int8_draw_has_the_readme_distribution():
    """The integer draw used for the long-context pool gives the distribution of the README-style
    truncated uniform draw: -127..126 at 1/255 each, 0 at 2/255, never -128 or 127."""
    rng = np.random.default_rng(5)
    n = 4_000_000
    fast = np.bincount(W._int8_like_readme_fast(rng, (n,)).astype(np.int16) + 128, minlength=256) / n
    slow = np.bincount(W._int8_like_readme(np.random.default_rng(6).uniform(-128, 127, n)).astype(np.int16) + 128,
                       minlength=256) / n
    expect = np.zeros(256)
    expect[1:255] = 1 / 255
    expect[128] = 2 / 255
    for h in (fast, slow):
        assert h[0] == 0 and h[255] == 0
        assert np.max(np.abs(h - expect)) < 6 * np.sqrt(2 / 255 / n)
