"""The upstream per-token-head quantizer and the paged key-cache write on the GPU (qli_quantize,
qli_quantize_keys) against the oracle: codes and scales bit-exact, the pool untouched outside the
written slots, bad positions and pages reported, and the whole chain (bfloat16 activations ->
codes -> indices) equal to the oracle's (needs a GB300)."""
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


def _bf16_dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _gpu_quantize(Q, bits, fp8, scale_f32):
    import torch
    x = _bf16_dev(bits)
    codes = torch.full(bits.shape, 0x5A, dtype=torch.uint8, device="cuda")
    scales = torch.full(bits.shape[:-1], -1, dtype=torch.float32 if scale_f32 else torch.float16, device="cuda")
    Q.check(Q.quantize(Q.FP8_E4M3 if fp8 else Q.INT8, Q.F32 if scale_f32 else Q.F16, x, codes, scales),
            "quantize")
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("scale_f32", [False, True])
@pytest.mark.parametrize("shape", [(1, 128), (1001, 128), (4, 3, 64, 128)])
def test_quantize_is_bit_exact(qli, fp8, scale_f32, shape):
    bits = W.bf16_vectors(shape, seed=11 + len(shape))
    codes, scales = _gpu_quantize(qli, bits, fp8, scale_f32)
    ref_codes, ref_scales = oracle.quantize(bits, fp8, scale_f32)
    assert np.array_equal(codes, ref_codes.view(np.uint8)), np.argwhere(codes != ref_codes.view(np.uint8))[:5]
    assert np.array_equal(scales.view(np.uint8), ref_scales.view(np.uint8))


def test_quantize_full_query_of_a_decode_step(qli):
    """The query of a 32-batch, 8-token step (16384 vectors, the size the indexer reads per call)."""
    bits = W.bf16_vectors((32, 8, 64, 128), seed=3)
    for fp8 in (False, True):
        codes, scales = _gpu_quantize(qli, bits, fp8, False)
        ref_codes, ref_scales = oracle.quantize(bits, fp8, False)
        assert np.array_equal(codes, ref_codes.view(np.uint8))
        assert np.array_equal(scales, ref_scales)


@pytest.mark.parametrize("fp8,scale_f32", [(False, False), (True, True)])
def test_quantize_at_the_prefill_size(qli, fp8, scale_f32):
    """The quantizer benchmark's query: a TND prefill of T = 15360 tokens x 64 heads (983040
    vectors, 252 MB of bfloat16), every code and scale compared."""
    bits = W.bf16_vectors((15360, 64, 128), seed=31)
    codes, scales = _gpu_quantize(qli, bits, fp8, scale_f32)
    ref_codes, ref_scales = oracle.quantize(bits, fp8, scale_f32)
    assert np.array_equal(codes, ref_codes.view(np.uint8))
    assert np.array_equal(scales.view(np.uint8), ref_scales.view(np.uint8))


def test_quantize_rejects_bad_arguments(qli):
    import torch
    x = _bf16_dev(W.bf16_vectors((2, 128), seed=1))
    codes = torch.empty((2, 128), dtype=torch.uint8, device="cuda")
    scales = torch.empty(2, dtype=torch.float16, device="cuda")
    lib = qli.lib
    st = qli._stream()
    bad = qli.STATUS_NAMES
    assert bad[lib.qli_quantize(7, qli.F16, x.data_ptr(), 2, codes.data_ptr(), scales.data_ptr(), st)] == \
        "QLI_ERR_INVALID_ARG"
    assert bad[lib.qli_quantize(qli.INT8, qli.F16, x.data_ptr(), -1, codes.data_ptr(), scales.data_ptr(), st)] == \
        "QLI_ERR_INVALID_ARG"
    assert bad[lib.qli_quantize(qli.INT8, qli.F16, x.data_ptr() + 2, 1, codes.data_ptr(), scales.data_ptr(), st)] == \
        "QLI_ERR_INVALID_ARG"
    assert bad[lib.qli_quantize(qli.INT8, qli.F16, x.data_ptr() + 8, 1, codes.data_ptr(), scales.data_ptr(), st)] == \
        "QLI_ERR_INVALID_ARG"                          # rows are read 16 bytes at a time
    assert lib.qli_quantize(qli.INT8, qli.F16, None, 0, None, None, st) == qli.QLI_OK


def _key_case(fp8, scale_f32, pad):
    case = W.make_case("kw", batch=3, s1=1, seq_lens_k=[700, 129, 1500], block_size=64, sparse_count=64,
                       qk_dtype=W.FP8 if fp8 else W.INT8, scale_dtype=W.F32 if scale_f32 else W.F16, seed=8)
    return W.with_key_stride(case, pad, seed=2) if pad else case


@pytest.mark.parametrize("fp8,scale_f32,pad", [(False, False, 0), (True, True, 0), (False, True, 48),
                                               (True, False, 16)])
def test_key_cache_write_matches_oracle(qli, fp8, scale_f32, pad):
    import torch
    case = _key_case(fp8, scale_f32, pad)
    p = qli.make_problem(**W.problem_kwargs(case))
    d = W.to_device(case)
    rng = np.random.default_rng(4)
    # the last key of every batch, plus distinct earlier positions scattered over the pages
    tok_b, tok_p = [], []
    for b, n in enumerate(case.seq_lens_k):
        pos = rng.choice(int(n) - 1, size=min(37, int(n) - 1), replace=False)
        tok_b += [b] * (len(pos) + 1)
        tok_p += list(pos) + [int(n) - 1]
    tok_b = np.array(tok_b, np.int32)
    tok_p = np.array(tok_p, np.int32)
    kb = W.bf16_vectors((len(tok_b), 128), seed=9)
    ws = torch.zeros(64, dtype=torch.int32, device="cuda")
    qli.check(qli.workspace_init(ws), "workspace_init")
    qli.check(qli.quantize_keys(p, _bf16_dev(kb), torch.from_numpy(tok_b).cuda(), torch.from_numpy(tok_p).cuda(),
                                d["block_table"], d["key"], d["k_scale"], ws), "quantize_keys")
    st, bits = qli.get_device_error(ws)
    assert st == qli.QLI_OK and bits == 0
    err = oracle.quantize_keys(case, kb, tok_b, tok_p)
    assert err == 0
    assert np.array_equal(d["key"].cpu().numpy(), case.key.view(np.uint8))
    assert np.array_equal(d["k_scale"].cpu().numpy().view(np.uint8), case.k_scale.view(np.uint8))


def test_key_cache_write_reports_and_skips_bad_tokens(qli):
    import torch
    case = _key_case(False, False, 0)
    case.block_table[1, 1] = case.num_blocks + 5          # a page outside the pool
    p = qli.make_problem(**W.problem_kwargs(case))
    d = W.to_device(case)
    tok_b = np.array([0, 3, -1, 1, 2], np.int32)          # batch 3 and -1 do not exist
    tok_p = np.array([699, 0, 0, 64 + 5, p.max_blocks_per_seq * 64], np.int32)  # last: past the table
    kb = W.bf16_vectors((5, 128), seed=10)
    ws = torch.zeros(64, dtype=torch.int32, device="cuda")
    qli.check(qli.workspace_init(ws), "workspace_init")
    qli.check(qli.quantize_keys(p, _bf16_dev(kb), torch.from_numpy(tok_b).cuda(), torch.from_numpy(tok_p).cuda(),
                                d["block_table"], d["key"], d["k_scale"], ws), "quantize_keys")
    st, bits = qli.get_device_error(ws)
    err = oracle.quantize_keys(case, kb, tok_b, tok_p)
    assert err == (oracle.ERR_LENGTH | oracle.ERR_PAGE)
    assert bits == err and qli.STATUS_NAMES[st] == "QLI_ERR_DEVICE_BAD_INPUT"
    assert np.array_equal(d["key"].cpu().numpy(), case.key.view(np.uint8))   # only token 0 landed
    assert np.array_equal(d["k_scale"].cpu().numpy().view(np.uint8), case.k_scale.view(np.uint8))


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_chain_from_bfloat16(qli, fp8):
    """One decode step from bfloat16 activations: quantize the query, write each batch's new key
    into the paged cache, then index; the same steps on the oracle give the same indices."""
    import torch
    case = W.make_case("chain", batch=4, s1=2, seq_lens_k=[3000, 1717, 260, 4097], block_size=128,
                       sparse_count=256, sparse_mode=3, qk_dtype=W.FP8 if fp8 else W.INT8, seed=12)
    p = qli.make_problem(**W.problem_kwargs(case))
    ix = qli.Indexer(p)
    d = W.to_device(case)
    q_bits = W.bf16_vectors(case.query.shape, seed=13)
    k_bits = W.bf16_vectors((case.batch, 128), seed=14, special=False)
    tok_b = np.arange(case.batch, dtype=np.int32)
    tok_p = (case.seq_lens_k - 1).astype(np.int32)
    # GPU: quantize into the indexer's own input tensors, then run it
    qli.check(qli.quantize(p.qk_dtype, p.scale_dtype, _bf16_dev(q_bits), d["query"], d["q_scale"]), "quantize")
    qli.check(qli.quantize_keys(p, _bf16_dev(k_bits), torch.from_numpy(tok_b).cuda(),
                                torch.from_numpy(tok_p).cuda(), d["block_table"], d["key"], d["k_scale"],
                                ix.workspace), "quantize_keys")
    gpu_idx = ix.run(**d).cpu().numpy()
    assert ix.device_error()[0] == qli.QLI_OK
    # oracle: the same steps on the host copy
    case.query, case.q_scale = oracle.quantize(q_bits, fp8, False)
    assert oracle.quantize_keys(case, k_bits, tok_b, tok_p) == 0
    ora_idx, ora_scores, err = oracle.score_topk(case, with_scores=True)
    assert err == 0
    _, _, fails = check(gpu_idx, ora_idx, ora_scores, visible_counts(case, oracle), case.sparse_count)
    assert not fails, fails[:5]
