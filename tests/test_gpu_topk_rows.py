"""The persistent two-per-SM top-k with hundreds of rows per CTA, against the CPU oracle (needs a
GB300).  Its CTAs work out the places of their rows in chunks of 512 rows (one row per thread) and
copy each next row's line during the current row's output; the testing build of the library caps
its grid (include/qli_testing.h) so that a problem of a few thousand rows crosses those chunk
boundaries.  Run in a child process: the testing build must be the first library the process
loads."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, %(root)r)
sys.path.insert(0, %(tests)r)
import numpy as np
import torch
import oracle
import workloads as W
import sparse_attention_token_block_gb300 as Q
from checker import check, visible_counts
Q.use_testing_library()
Q.lib.qli_testing_set_topk_ctas(%(ctas)d)
case = W.make_case("rows_per_cta", layout_q="TND", q_lens=%(q_lens)r, seq_lens_k=%(k_lens)r, block_size=64,
                   sparse_count=%(k)d, sparse_mode=3, seed=%(seed)d)
p = Q.make_problem(**W.problem_kwargs(case))
ix = Q.Indexer(p)
d = W.to_device(case)
gpu = ix.run(**d).cpu().numpy()
st, bits = ix.device_error()
ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True)
vis = visible_counts(case, oracle)
exact, checked, fails = check(gpu, ora_idx, ora_scores, vis, case.sparse_count)
# the plan (graph replay, the top-k directly after the score kernel) gives the same indices
plan = ix.plan(**d)
ix.out.fill_(-7)
plan.launch()
torch.cuda.synchronize()
same = bool(np.array_equal(ix.out.cpu().numpy(), gpu))
print("RESULT", case.rows, st, err, len(fails), checked, same)
"""


@pytest.fixture(scope="module")
def built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_token_block_gb300 import build as B
    B.build()


CASES = [
    # 1800 rows over 2 CTAs: 900 rows each, one chunk boundary; short, mid and long lines mixed
    ("two_ctas", 2, [300, 700, 200, 600], [300, 5000, 8192, 3000], 128, 11),
    # 3 CTAs: rows 0, 3, 6, ... of each sequence; a chunk boundary inside each CTA's rows; k = 7
    ("three_ctas", 3, [513, 1030, 60], [600, 4100, 2000], 7, 12),
]


@pytest.mark.parametrize("name,ctas,q_lens,k_lens,k,seed", CASES, ids=[c[0] for c in CASES])
def test_many_rows_per_cta_matches_oracle(built, name, ctas, q_lens, k_lens, k, seed):
    src = CHILD % dict(root=ROOT, tests=os.path.join(ROOT, "tests"), ctas=ctas, q_lens=q_lens, k_lens=k_lens,
                       k=k, seed=seed)
    out = subprocess.run([sys.executable, "-c", src], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    res = [l for l in out.stdout.splitlines() if l.startswith("RESULT")][0].split()
    rows, st, err, nfails, checked, same = int(res[1]), int(res[2]), int(res[3]), int(res[4]), int(res[5]), res[6]
    assert rows > 2 * 152 and rows // ctas > 512
    assert st == 0 and err == 0
    assert nfails == 0 and checked > 0
    assert same == "True"
