"""The work split written by qli_metadata, word by word against a host re-derivation of its
definition (needs a GB300).

Definition (the metadata call: the cores used and each core's start point): query groups of
group_tokens consecutive live rows per batch; a group's tiles are ceil(n / 128), n the visible keys
of its last row; live groups (at least one tile) are listed in batch and row order.  The split cuts
a sequence of T positions in which every live group occupies U virtual positions (its query load)
followed by its tiles; a record holds the position of the group's first tile.  Score CTA c of G
owns positions [T W(c) / W(G), T W(c + 1) / W(G)) and the live groups whose tiles that range
overlaps, where W(c) weighs the first G1 CTAs (the first to arrive on their SM) 12 and the others
11.  Groups hold one token when a sequence has one query token, else up to three."""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

MAGIC = 0x514C4932
# weights of the first-arriving score CTAs of an SM and of the others in the split (equal: the
# library's kSplitFirst and kSplitSecond)
FIRST, SECOND = 1, 1


def split_start(T, G, G1, c):
    def w(x):
        return x * FIRST if x <= G1 else G1 * FIRST + (x - G1) * SECOND
    return T * w(c) // w(G)


def group_tokens(case):
    """Query tokens per group: one for one query token per sequence, two for two or four, else up
    to three."""
    if case.layout_q == "BSND":
        if case.s1 <= 1:
            return 1
        return 2 if case.s1 in (2, 4) else min(case.s1, 3)
    return 3


@pytest.fixture(scope="module")
def qli():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_token_block_gb300 import build as B
    B.build()
    import sparse_attention_token_block_gb300 as Q
    return Q


def derive(case, G, G1, gt, U):
    """Header fields, batch entries, live group records and CTA ranges of the definition."""
    B = case.batch
    batches, records = [], []
    tnd = case.layout_q == "TND"
    lc_cap = case.max_blocks_per_seq * case.block_size
    bad_tnd = False
    err = 0
    raw = []
    for b in range(B):
        if not tnd:
            first = b * case.s1
            v = case.s1 if case.seq_lens_q is None else int(case.seq_lens_q[b])
            ok = 0 <= v <= case.s1
            sq = v if ok else 0
        else:
            lo = int(case.seq_lens_q[b - 1]) if b > 0 else 0
            hi = int(case.seq_lens_q[b])
            ok = lo >= 0 and hi >= lo and hi <= case.total_q
            bad_tnd |= not ok
            first = max(lo, 0)
            sq = hi - lo if ok else 0
        sk = int(case.seq_lens_k[b])
        ok = ok and 0 <= sk <= case.max_seqlen_k
        lc = -(-sk // case.cmp_ratio) if ok else 0
        ok = ok and lc <= lc_cap
        if not ok:
            err |= 1
        raw.append([sq, sk if ok else 0, lc, first, ok])
    gbase = 0
    T = 0
    for b, (sq, sk, lc, first, ok) in enumerate(raw):
        okb = ok and not bad_tnd
        groups = -(-sq // gt) if okb else 0
        batches.append([sq, sk, lc, first, int(okb), groups, gbase])
        for g in range(groups):
            r0 = g * gt
            rl = min(r0 + gt, sq) - 1
            n = oracle.visible(case, sq, sk, rl)
            tiles = -(-n // 128)
            if tiles:
                records.append([b, r0, first + r0, sq, sk, lc, T + U, tiles])
                T += U + tiles
        gbase += groups
    ctas = []
    starts = [rec[6] for rec in records]
    for c in range(G):
        t0, t1 = split_start(T, G, G1, c), split_start(T, G, G1, c + 1)
        if t1 <= t0:
            ctas.append((0, 0))
            continue
        first = max(i for i, s in enumerate(starts) if s - U <= t0)       # block holding t0
        end = max(first, next((i for i, s in enumerate(starts) if s >= t1), len(starts)))
        ctas.append((first, end))
    return dict(live=len(records), T=T, err=err, groups=gbase, batches=batches, records=records, ctas=ctas)


CASES = [
    ("tiny_decode", lambda: W.tiny_decode()),
    ("long_decode", lambda: W.long_decode()),
    ("fp8_compressed_decode", lambda: W.fp8_compressed_decode()),
    ("varlen_prefill", lambda: W.varlen_prefill()),
    ("tnd_empty_and_short", lambda: W.make_case("m1", layout_q="TND", q_lens=[5, 0, 9, 1, 30],
                                                seq_lens_k=[3, 40, 600, 0, 30], block_size=32,
                                                sparse_count=64, sparse_mode=3, seed=1)),
    ("bsnd_qlens", lambda: W.make_case("m2", batch=4, s1=4, q_lens=[4, 0, 1, 3],
                                       seq_lens_k=[600, 600, 129, 2], block_size=64,
                                       sparse_count=200, sparse_mode=3, seed=2)),
    ("bad_length", lambda: W.make_case("m3", batch=3, s1=2, q_lens=[2, 3, 1],
                                       seq_lens_k=[300, 300, 5000], block_size=64,
                                       sparse_count=16, seed=3)),
    # 24 batches of two query groups (48 groups: the one-warp path's second half of groups)
    ("page_decode", lambda: W.page_decode()),
    # 32 batches x 2 groups = 64 groups, empty batches and rows without keys on both halves
    ("two_halves", lambda: W.make_case("m5", batch=32, s1=4, q_lens=[(i * 7) % 5 for i in range(32)],
                                       seq_lens_k=[0 if i % 6 == 2 else 50 * i + 3 for i in range(32)],
                                       block_size=32, sparse_count=64, sparse_mode=3, seed=5)),
    # 17 batches x 2 groups = 34 groups: two past the first half
    ("just_over_half", lambda: W.make_case("m6", batch=17, s1=4, seq_lens_k=[300 + 17 * i for i in range(17)],
                                           block_size=64, sparse_count=32, sparse_mode=0, seed=6)),
    # 31 batches of at most one row: rows without keys, batches without rows between live ones
    ("small_gaps", lambda: W.make_case("m4", batch=31, s1=1, q_lens=[(i % 3 > 0) * 1 for i in range(31)],
                                       seq_lens_k=[0 if i % 4 == 1 else 40 * i + 7 for i in range(31)],
                                       block_size=32, sparse_count=64, sparse_mode=3, seed=4)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_metadata_matches_definition(qli, name, make):
    import torch
    case = make()
    if name == "bad_length":
        case.seq_lens_q = np.array([2, 3, 1], np.int32)      # 3 > S1: batch 1 invalid
    p = qli.make_problem(**W.problem_kwargs(case))
    meta = torch.full((qli.metadata_words(p),), -7, dtype=torch.int32, device="cuda")
    d = W.to_device(case)
    qli.check(qli.metadata(p, d["seq_lens_q"], d["seq_lens_k"], meta), "metadata")
    m = meta.cpu().numpy()
    G, G1, U = int(m[1]), int(m[9]), int(m[10])
    assert m[0] == MAGIC and 1 <= G <= 1024 and 1 <= G1 <= G and U == 2
    ref = derive(case, G, G1, group_tokens(case), U)
    assert int(m[2]) == ref["live"] and int(m[3]) == ref["T"]
    assert int(m[4]) == ref["err"] and int(m[5]) == case.batch and int(m[6]) == case.rows
    assert int(m[7]) == ref["groups"]
    B = case.batch
    be = m[16:16 + 8 * B].reshape(B, 8)[:, :7]
    assert np.array_equal(be, np.array(ref["batches"], dtype=np.int64).reshape(B, 7))
    cta_off = 16 + 8 * B
    ctas = m[cta_off:cta_off + 2 * G].reshape(G, 2)
    assert [tuple(map(int, x)) for x in ctas] == ref["ctas"]
    rec_off = (cta_off + 2 * 1024 + 3) & ~3
    recs = m[rec_off:rec_off + 8 * ref["live"]].reshape(-1, 8)
    assert np.array_equal(recs, np.array(ref["records"], dtype=np.int64).reshape(-1, 8))
    # every live group's tiles are covered exactly once by the CTAs' (group, tile range) units,
    # each unit holds at least one tile, and no virtual position is covered
    cover = np.zeros(ref["T"], np.int64)
    for c in range(G):
        t0, t1 = split_start(ref["T"], G, G1, c), split_start(ref["T"], G, G1, c + 1)
        f, e = ctas[c]
        for g in range(f, e):
            tb, tn = recs[g][6], recs[g][7]
            lo, hi = max(t0, tb), min(t1, tb + tn)
            assert hi > lo
            cover[lo:hi] += 1
    real = np.zeros(ref["T"], bool)
    for r in recs:
        real[r[6]:r[6] + r[7]] = True
    assert (cover[real] == 1).all() and (cover[~real] == 0).all()
