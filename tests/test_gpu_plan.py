"""Execution plans (qli_plan_*): a captured call replays the same kernels on the captured buffers,
so its output equals a stream call's and follows in-place changes of the inputs (needs a GB300)."""
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


def _setup(Q, case):
    p = Q.make_problem(**W.problem_kwargs(case))
    return p, Q.Indexer(p), W.to_device(case)


@pytest.mark.parametrize("name", ["page_decode", "fp8_compressed_decode"])
def test_plan_matches_stream_call(qli, name):
    import torch
    case = W.WORKLOADS[name]()
    p, ix, d = _setup(qli, case)
    ref = ix.run(**d).clone()
    plan = ix.plan(**d)
    ix.out.fill_(-7)
    for _ in range(3):
        plan.launch()
    torch.cuda.synchronize()
    assert torch.equal(ix.out, ref)
    assert ix.device_error()[0] == 0
    plan.close()


def test_plan_reads_inputs_in_place(qli):
    """New key codes and weights written into the captured buffers are what the next replay scores."""
    import torch
    case = W.make_case("plan_inplace", batch=3, s1=2, seq_lens_k=[700, 90, 1500], block_size=64,
                       sparse_count=128, sparse_mode=3, seed=21)
    p, ix, d = _setup(qli, case)
    plan = ix.plan(**d)
    plan.launch()
    torch.cuda.synchronize()
    first = ix.out.cpu().numpy().copy()
    # change the inputs in place (same shapes and addresses), then replay
    rng = np.random.default_rng(5)
    case.key[:] = rng.integers(-128, 128, size=case.key.shape).astype(np.int8)
    case.weights[:] = (rng.uniform(0, 0.01, size=case.weights.shape)).astype(case.weights.dtype)
    d["key"].copy_(torch.from_numpy(np.ascontiguousarray(case.key.view(np.uint8))).to(d["key"].device))
    d["weights"].copy_(torch.from_numpy(np.ascontiguousarray(case.weights)).to(d["weights"].device))
    plan.launch()
    torch.cuda.synchronize()
    gpu_idx = ix.out.cpu().numpy()
    ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True)
    assert err == 0
    _, _, fails = check(gpu_idx, ora_idx, ora_scores, visible_counts(case, oracle), case.sparse_count)
    assert not fails, fails[:5]
    assert not np.array_equal(first, gpu_idx)
    plan.close()


def test_plan_without_metadata_uses_the_buffer(qli):
    import torch
    case = W.WORKLOADS["page_decode"]()
    p, ix, d = _setup(qli, case)
    ref = ix.run(**d).clone()             # writes the metadata buffer
    plan = ix.plan(**d, with_metadata=False)
    ix.out.zero_()
    plan.launch()
    torch.cuda.synchronize()
    assert torch.equal(ix.out, ref)
    plan.close()


def test_plan_rejects_bad_arguments_and_leaves_the_stream_usable(qli):
    import torch
    case = W.WORKLOADS["tiny_decode"]()
    p, ix, d = _setup(qli, case)
    st, h = qli.plan_create(p, True, d["query"], d["key"], d["weights"], d["q_scale"], d["k_scale"],
                            d["seq_lens_q"], d["seq_lens_k"], d["block_table"], ix.meta, ix.workspace,
                            None)
    assert qli.STATUS_NAMES[st] == "QLI_ERR_INVALID_ARG" and h is None
    out = ix.run(**d)                     # capture ended cleanly: ordinary calls still work
    torch.cuda.synchronize()
    assert (out[0, :64] >= 0).all()


def _poison_score_lines(ix):
    """Every score code in the workspace set to the largest value: a tile the score kernel skipped
    would then win its row's top-k."""
    import torch
    ix.workspace.view(torch.uint8)[256:].fill_(0xFF)


@pytest.mark.parametrize("name", ["tiny_decode", "page_decode", "long_decode", "fp8_compressed_decode",
                                  "varlen_prefill", "mixed"])
def test_plan_replay_rewrites_every_visible_score(qli, name):
    """A replay must score every visible key again: after the score lines were poisoned, it returns
    the stream call's indices and rewrites the same metadata."""
    import torch
    if name == "mixed":
        # empty batches, short query runs and rows that see no key, two tokens per query group
        case = W.make_case("mixed", batch=37, s1=3, q_lens=[(i * 7) % 4 for i in range(37)],
                           seq_lens_k=[0 if i % 5 == 0 else 64 + 97 * i for i in range(37)], block_size=64,
                           sparse_count=96, sparse_mode=3, seed=33)
    else:
        case = W.WORKLOADS[name]()
    p, ix, d = _setup(qli, case)
    ref = ix.run(**d).clone()
    meta_ref = ix.meta.clone()
    plan = ix.plan(**d)
    for _ in range(2):
        _poison_score_lines(ix)
        ix.out.fill_(-7)
        plan.launch()
        torch.cuda.synchronize()
        assert torch.equal(ix.out, ref)
        assert torch.equal(ix.meta, meta_ref)
        assert ix.device_error()[0] == 0
    plan.close()
