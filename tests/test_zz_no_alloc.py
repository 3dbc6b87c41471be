"""qli_score_topk_static, the entry point for callers that cannot allocate device memory.

It must give what qli_score_topk gives with a caller-provided workspace, on two calls in a row
(the library's scratch array keeps the first call's contents when the second starts), whether
this file runs alone in a fresh process or after the rest of the suite.  It sits in a file of its
own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as W
from checker import check, visible_counts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_token_block_gb300 import build as B
    B.build()
    import sparse_attention_token_block_gb300 as Q
    return Q


def _via_workspace(Q, p, d):
    import torch
    ix = Q.Indexer(p)
    out = ix.run(**d)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ix.meta


def test_static_scratch_matches_workspace_path_twice(Q):
    import torch
    cases = [
        W.make_case("static_a", batch=4, s1=2, seq_lens_k=[3000, 17, 900, 2048], block_size=64,
                    sparse_count=256, sparse_mode=3, seed=21),
        W.make_case("static_b", batch=3, s1=1, qk_dtype=W.FP8, scale_dtype=W.F32,
                    seq_lens_k=[5000, 640, 1], block_size=128, sparse_count=100, sparse_mode=3,
                    cmp_ratio=4, seed=22),
    ]
    for case in cases:
        p = Q.make_problem(**W.problem_kwargs(case))
        d = W.to_device(case)
        ref, meta = _via_workspace(Q, p, d)
        err = torch.full((1,), 0xFF, dtype=torch.int32, device="cuda")
        for _ in range(2):
            out = torch.full(ref.shape, -7, dtype=torch.int32, device="cuda")
            st = Q.lib.qli_score_topk_static(
                ctypes.byref(p), d["query"].data_ptr(), d["key"].data_ptr(),
                d["weights"].data_ptr(), d["q_scale"].data_ptr(), d["k_scale"].data_ptr(),
                None if d["seq_lens_q"] is None else d["seq_lens_q"].data_ptr(),
                d["seq_lens_k"].data_ptr(), d["block_table"].data_ptr(), meta.data_ptr(),
                meta.numel(), out.data_ptr(), err.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
            assert st == Q.QLI_OK, Q.status_string(st)
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            # same kernels on the same inputs: identical, which is within any tolerance
            assert np.array_equal(got, ref)
            assert int(err.item()) == 0
        # and the oracle's indices under the parity tests' tie-aware rule (row tolerance 1e-5 of
        # the row's largest score)
        ora_idx, ora_scores, ora_err = oracle.score_topk(case, with_scores=True)
        assert ora_err == 0
        _, checked, fails = check(got, ora_idx, ora_scores, visible_counts(case, oracle), case.sparse_count)
        assert checked == case.rows and not fails, fails[:3]


def test_static_scratch_rejects_oversized_problems(Q):
    p = Q.make_problem(batch=64, max_q_tokens=4, num_blocks=4096, block_size=128,
                       max_blocks_per_seq=512, sparse_count=2048, sparse_mode=3, cmp_ratio=1,
                       max_seqlen_q=4, max_seqlen_k=65536)
    assert Q.workspace_size(p) > 16 << 20
    st = Q.lib.qli_score_topk_static(ctypes.byref(p), *([None] * 9), 0, None, None, None)
    assert st == 3  # QLI_ERR_WORKSPACE_TOO_SMALL, before anything is enqueued
