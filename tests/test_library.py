"""Host-side checks of the C-ABI library that need no GPU: it loads, exports every symbol the
header declares, and rejects invalid problems synchronously."""
import ctypes
import re
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def Q():
    from sparse_attention_token_block_gb300 import build as B
    B.build()
    import sparse_attention_token_block_gb300 as Q
    return Q


def declared_symbols(header="qli.h"):
    text = open(os.path.join(ROOT, "include", header)).read()
    return sorted(set(re.findall(r"\b(qli_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(Q):
    names = declared_symbols()
    assert set(names) == set(Q.EXPORTS)
    for n in names:
        assert hasattr(Q.lib, n), n
    # the product library carries no test switch
    for n in declared_symbols("qli_testing.h"):
        assert not hasattr(Q.lib, n), n


def test_measurement_library_exports_its_symbol(Q):
    from sparse_attention_token_block_gb300 import build as B
    L = ctypes.CDLL(B.PEAK_LIB)
    for n in declared_symbols("qli_peak.h"):
        assert hasattr(L, n), n
    for n in declared_symbols("qli_peak.h"):
        assert not hasattr(Q.lib, n), n


def test_testing_build_exports_product_and_testing_symbols(Q):
    L = ctypes.CDLL(Q.TESTING_LIB_PATH)
    for n in declared_symbols() + declared_symbols("qli_testing.h"):
        assert hasattr(L, n), n


def _ok_problem(Q, **kw):
    args = dict(batch=2, max_q_tokens=1, num_blocks=8, block_size=64, max_blocks_per_seq=4,
                sparse_count=64, sparse_mode=3, cmp_ratio=1, max_seqlen_q=1, max_seqlen_k=256)
    args.update(kw)
    return Q.make_problem(**args)


def test_validate_accepts_readme_example(Q):
    p = _ok_problem(Q, batch=24, max_q_tokens=4, num_blocks=96, block_size=128,
                    max_blocks_per_seq=4, sparse_count=512, sparse_mode=0, max_seqlen_q=4,
                    max_seqlen_k=512)
    st, why = Q.validate(p)
    assert st == 0, why
    assert Q.metadata_words(p) >= 1024
    assert Q.workspace_size(p) >= 256 + 96 * 512 * 4


@pytest.mark.parametrize("field,value,status", [
    ("num_heads_q", 32, 1), ("num_heads_k", 2, 1), ("head_dim", 64, 1), ("block_size", 24, 1),
    ("block_size", 2048, 1), ("sparse_count", 0, 1), ("sparse_count", 2049, 1),
    ("sparse_mode", 1, 1), ("cmp_ratio", 3, 1), ("cmp_ratio", 256, 1), ("query_quant_mode", 1, 1),
    ("key_quant_mode", 1, 1), ("pre_tokens", 5, 1), ("next_tokens", 0, 1), ("qk_dtype", 2, 1),
    ("scale_dtype", 7, 1), ("layout_q", 2, 1), ("max_blocks_per_seq", 3, 1),
    ("return_value", 2, 1), ("num_blocks", 0, 1), ("batch", -1, 1), ("split_topk", 3, 1),
    ("split_topk", -1, 1),
])
def test_validate_rejects(Q, field, value, status):
    p = _ok_problem(Q)
    setattr(p, field, value)
    st, why = Q.validate(p)
    assert st == status, (field, why)
    assert Q.metadata_words(p) == 0 and Q.workspace_size(p) == 0


def test_split_topk_workspace_and_auto_rule(Q):
    """The two-stage top-k needs two more [rows, ld] lines and one word per tile in the
    workspace; it runs only on request (AUTO keeps one stage), and a request for it is ignored when
    S1 > 1."""
    kw = dict(batch=4, max_q_tokens=1, num_blocks=600, block_size=64, max_blocks_per_seq=150,
              max_seqlen_q=1, max_seqlen_k=9000)
    rows, ld = 4, 9088
    lines = 256 + rows * ld * 4
    split = lines + 2 * rows * ld * 4 + rows * (ld // 128) * 4
    size = lambda **o: Q.workspace_size(_ok_problem(Q, **dict(kw, **o)))
    for k in (1, 64, 512, 2048):
        assert size(sparse_count=k, split_topk=Q.SPLIT_OFF) == lines
        assert size(sparse_count=k, split_topk=Q.SPLIT_AUTO) == lines
        assert size(sparse_count=k, split_topk=Q.SPLIT_ON) == split
    # query groups of several tokens: one stage whatever is asked
    assert size(sparse_count=64, max_q_tokens=2, max_seqlen_q=2, split_topk=Q.SPLIT_ON) == 256 + 2 * (lines - 256)


def test_invalid_calls_enqueue_nothing(Q):
    # rejected before any CUDA call, so these work without a GPU
    p = _ok_problem(Q)
    p.sparse_count = 0
    assert Q.lib.qli_metadata(ctypes.byref(p), None, None, None, 0, None) == 1
    assert Q.lib.qli_score_topk(ctypes.byref(p), *([None] * 9), 0, None, 0, None, None, None) == 1
    p = _ok_problem(Q)
    assert Q.lib.qli_metadata(ctypes.byref(p), None, None, None, 0, None) == 1      # no buffer
    assert Q.lib.qli_metadata(ctypes.byref(p), None, None, 16, 10, None) == 3       # too small
    assert Q.lib.qli_score_topk(ctypes.byref(p), *([None] * 9), 0, None, 0, None, None,
                                None) == 3
    # sparse_values must be given exactly when return_value = 1
    assert Q.lib.qli_score_topk(ctypes.byref(p), *([None] * 9), 1 << 20, None, 1 << 30, None,
                                1024, None) == 1
    p.return_value = 1
    assert Q.lib.qli_score_topk(ctypes.byref(p), *([None] * 9), 1 << 20, None, 1 << 30, None,
                                None, None) == 1
    assert Q.lib.qli_topk(ctypes.byref(p), None, None, 1 << 20, None, 1 << 30, None, None, None) == 1
    assert Q.status_string(6) == "device wait timed out"
    assert Q.version() >= 100


def test_quantizer_and_gather_reject_bad_arguments(Q):
    # qli_quantize / qli_quantize_keys / qli_gather_kv check their arguments before any CUDA call;
    # the pointers below are aligned dummies that the rejected calls never dereference
    A = 1 << 20                                        # a 16-byte aligned stand-in address
    L = Q.lib
    assert L.qli_quantize(2, Q.F16, A, 1, A, A, None) == 1                 # qk dtype
    assert L.qli_quantize(Q.INT8, 5, A, 1, A, A, None) == 1                # scale dtype
    assert L.qli_quantize(Q.INT8, Q.F16, A, -1, A, A, None) == 1           # count
    assert L.qli_quantize(Q.INT8, Q.F16, A, 1 << 37, A, A, None) == 1      # grid limit
    assert L.qli_quantize(Q.INT8, Q.F16, None, 1, A, A, None) == 1
    assert L.qli_quantize(Q.INT8, Q.F16, A + 8, 1, A, A, None) == 1        # 16-byte rows
    assert L.qli_quantize(Q.INT8, Q.F16, A, 1, A + 4, A, None) == 1        # 8-byte codes
    assert L.qli_quantize(Q.INT8, Q.F32, A, 1, A, A + 2, None) == 1        # fp32 scales
    assert L.qli_quantize(Q.INT8, Q.F16, None, 0, None, None, None) == 0   # nothing to do
    p = _ok_problem(Q)
    assert L.qli_quantize_keys(ctypes.byref(p), A, -1, A, A, A, A, A, None, 0, None) == 1
    assert L.qli_quantize_keys(ctypes.byref(p), A, 1, A, A, A, A, A, A + 16, 256, None) == 1  # workspace alignment
    assert L.qli_quantize_keys(ctypes.byref(p), A, 1, A, A, A, A, A, A, 64, None) == 1       # workspace size
    assert L.qli_quantize_keys(ctypes.byref(p), A, 1, None, A, A, A, A, None, 0, None) == 1
    assert L.qli_quantize_keys(ctypes.byref(p), A + 8, 1, A, A, A, A, A, None, 0, None) == 1
    assert L.qli_quantize_keys(ctypes.byref(p), A, 1, A, A, A, A + 8, A, None, 0, None) == 1  # key pool
    assert L.qli_quantize_keys(ctypes.byref(p), None, 0, None, None, None, None, None, None, 0, None) == 0
    bad = _ok_problem(Q)
    bad.head_dim = 64
    assert L.qli_quantize_keys(ctypes.byref(bad), A, 1, A, A, A, A, A, None, 0, None) == 1
    g = lambda *args: L.qli_gather_kv(ctypes.byref(p), *args)
    assert g(None, A, A, A, A, 24, 0, A, None, None, 0, None) == 1         # entry not a multiple of 16
    assert g(None, A, A, A, A, 0, 0, A, None, None, 0, None) == 1
    assert g(None, A, A, A, A, 65552, 0, A, None, None, 0, None) == 1      # above 64 KiB
    page = p.block_size * 64
    assert g(None, A, A, A, A, 64, page - 16, A, None, None, 0, None) == 1  # stride below a page
    assert g(None, A, A, A, A, 64, page + 8, A, None, None, 0, None) == 1   # stride not 16-aligned
    assert g(None, A, A, None, A, 64, 0, A, None, None, 0, None) == 1       # indices
    assert g(None, A, None, A, A, 64, 0, A, None, None, 0, None) == 1       # block_table
    assert g(None, A, A, A, A + 8, 64, 0, A, None, None, 0, None) == 1      # pool alignment
    assert g(None, A, A, A, A, 64, 0, A + 8, None, None, 0, None) == 1      # output alignment
    assert g(None, A, A, A, A, 64, 0, A, A + 2, None, 0, None) == 1         # counts alignment
    assert g(None, A, A, A, A, 64, 0, A, None, A, 16, None) == 1            # workspace size
    t = _ok_problem(Q)
    t.layout_q = Q.TND
    t.total_q_tokens = 8
    assert L.qli_gather_kv(ctypes.byref(t), None, A, A, A, A, 64, 0, A, None, None, 0, None) == 1  # TND prefix sums


def test_problem_struct_layout_matches_the_header(Q, tmp_path):
    """The binding's ctypes mirror of qli_problem has the header's size and field offsets (a C
    program built against include/qli.h prints them)."""
    import subprocess
    fields = [f[0] for f in Q.Problem._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stddef.h>\n#include <stdio.h>\n#include \"qli.h\"\nint main(void) {\n"
                   "  printf(\"%zu\\n\", sizeof(qli_problem));\n"
                   + "".join("  printf(\"%%zu\\n\", offsetof(qli_problem, %s));\n" % f for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert got[0] == ctypes.sizeof(Q.Problem)
    assert got[1:] == [getattr(Q.Problem, f).offset for f in fields]
