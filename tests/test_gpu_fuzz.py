"""Seeded random shapes, CUDA path vs the CPU oracle through the C ABI (needs a GB300).

Each case draws its shape from a fixed seed: layout (BSND with S1 1..4, or TND with 1..6
sequences), per-sequence query and key lengths (empty, one token, ragged around the 128-key tiles,
up to ~9k keys), block_size (16..256, not only powers of two), cmp_ratio 1..16, mask mode 0 or 3,
k 1..2048, int8 or e4m3 codes, fp16 or fp32 scales, a random or identity block_table, and for some
cases a query count above the SMs, so that every score and top-k build is reached.  Indices must
match the oracle's (ties within each row's tolerance), the scores within it."""
import numpy as np
import pytest

import oracle
import workloads as W
from checker import check, check_scores, visible_counts

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module")
def qli():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_token_block_gb300 import build as B
    B.build()
    import sparse_attention_token_block_gb300 as Q
    return Q


def draw_shape(seed):
    """The kwargs of workloads.make_case for fuzz case `seed` (sizes kept so that the oracle takes
    a second or two)."""
    rng = np.random.default_rng(1000 + seed)
    kw = {}

    def k_len():
        r = rng.random()
        if r < 0.08:
            return 0
        if r < 0.16:
            return int(rng.integers(1, 4))
        if r < 0.4:
            return int(128 * rng.integers(1, 20) + rng.integers(-1, 2))
        return int(rng.integers(4, 9000))

    if rng.random() < 0.5:
        B = int(rng.integers(1, 40))
        s1 = int(rng.integers(1, 5))
        kw.update(layout_q="BSND", batch=B, s1=s1)
        if rng.random() < 0.4:
            kw["q_lens"] = [int(rng.integers(0, s1 + 1)) for _ in range(B)]
        kw["seq_lens_k"] = [k_len() for _ in range(B)]
    else:
        B = int(rng.integers(1, 7))
        kw.update(layout_q="TND", q_lens=[int(rng.integers(0, 130)) for _ in range(B)])
        kw["seq_lens_k"] = [k_len() for _ in range(B)]
    kw["block_size"] = int(rng.choice([16, 32, 48, 64, 80, 128, 256]))
    kw["cmp_ratio"] = int(rng.choice([1, 1, 1, 2, 4, 16]))
    kw["sparse_mode"] = int(rng.choice([0, 3]))
    kw["sparse_count"] = int(rng.choice([1, 7, 64, 300, 512, 2048]))
    kw["qk_dtype"] = W.FP8 if rng.random() < 0.3 else W.INT8
    kw["scale_dtype"] = W.F32 if rng.random() < 0.3 else W.F16
    kw["permute"] = bool(rng.random() < 0.8)
    return kw


@pytest.mark.parametrize("seed", range(N_CASES))
def test_fuzz_shape_matches_oracle(qli, seed):
    import torch
    kw = draw_shape(seed)
    case = W.make_case("fuzz%d" % seed, seed=seed, **kw)
    p = qli.make_problem(**W.problem_kwargs(case))
    ix = qli.Indexer(p)
    d = W.to_device(case)
    gpu = ix.run(**d).cpu().numpy()
    lines = ix.score_lines().cpu().numpy()
    torch.cuda.synchronize()
    st, bits = ix.device_error()
    ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True)
    assert err == 0 and st == 0, (kw, err, st, bits)
    vis = visible_counts(case, oracle)
    exact, checked, fails = check(gpu, ora_idx, ora_scores, vis, case.sparse_count)
    assert not fails, (kw, fails[:3])
    if case.rows:
        assert check_scores(lines, ora_scores, vis) <= 1.0, kw
