"""ctypes front end of the CPU oracle (``qli_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg use it.
The product path never imports this package.

``build()`` compiles the C file with the system C compiler; ``score_topk(case)`` runs the oracle on
a :class:`workloads.Case` and returns the indices (and optionally every visible key's fp32 score).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qli_oracle.c")
_LIB = os.path.join(_HERE, "libqli_oracle.so")
# a test may point the front end at another build of the oracle (a planted mistake)
_LIB_OVERRIDE = os.environ.get("QLI_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

ERR_LENGTH = 1
ERR_PAGE = 2


class Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "s1", "total_q", "layout_tnd", "qk_fp8", "scale_f32", "num_heads", "head_dim",
        "num_blocks", "block_size", "max_blocks_per_seq", "sparse_count", "sparse_mode",
        "cmp_ratio", "complete_blocks_only", "key_stride")]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libqli_oracle.so`` (plain C11, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-Wall",
                               "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if _LIB_OVERRIDE:
                L = ctypes.CDLL(_LIB_OVERRIDE)
            else:
                build()
                L = ctypes.CDLL(_LIB)
            L.qlio_half_to_float.restype = ctypes.c_float
            L.qlio_half_to_float.argtypes = [ctypes.c_uint16]
            L.qlio_e4m3_value.restype = ctypes.c_double
            L.qlio_e4m3_value.argtypes = [ctypes.c_uint8]
            L.qlio_visible.restype = ctypes.c_int64
            L.qlio_visible.argtypes = [ctypes.POINTER(Problem), ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int64]
            L.qlio_rows.restype = ctypes.c_int64
            L.qlio_rows.argtypes = [ctypes.POINTER(Problem)]
            vp = ctypes.c_void_p
            L.qlio_score_topk.restype = ctypes.c_int
            L.qlio_score_topk.argtypes = [ctypes.POINTER(Problem), vp, vp, vp, vp, vp, vp, vp, vp,
                                          vp, vp, ctypes.c_int64, vp, ctypes.c_int]
            L.qlio_quantize_vectors.restype = None
            L.qlio_quantize_vectors.argtypes = [ctypes.c_int, ctypes.c_int, vp, ctypes.c_int64, vp, vp]
            L.qlio_quantize_keys.restype = ctypes.c_int
            L.qlio_quantize_keys.argtypes = [ctypes.POINTER(Problem), vp, ctypes.c_int64, vp, vp, vp, vp, vp]
            L.qlio_gather_kv.restype = ctypes.c_int
            L.qlio_gather_kv.argtypes = [ctypes.POINTER(Problem), vp, vp, vp, vp, vp, ctypes.c_int64,
                                         ctypes.c_int64, vp, vp]
            _lib = L
    return _lib


def problem_of(case, complete_blocks_only: bool = False) -> Problem:
    return Problem(batch=case.batch, s1=case.s1, total_q=case.total_q,
                   layout_tnd=1 if case.layout_q == "TND" else 0,
                   qk_fp8=0 if case.qk_dtype == "int8" else 1,
                   scale_f32=1 if case.scale_dtype == "f32" else 0,
                   num_heads=case.query.shape[-2], head_dim=case.query.shape[-1],
                   num_blocks=case.num_blocks, block_size=case.block_size,
                   max_blocks_per_seq=case.max_blocks_per_seq, sparse_count=case.sparse_count,
                   sparse_mode=case.sparse_mode, cmp_ratio=case.cmp_ratio,
                   complete_blocks_only=1 if complete_blocks_only else 0,
                   key_stride=getattr(case, "key_stride", 0))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def half_to_float(code: int) -> float:
    return lib().qlio_half_to_float(code)


def e4m3_value(code: int) -> float:
    return lib().qlio_e4m3_value(code)


def visible(case, sq: int, sk: int, r: int, complete_blocks_only: bool = False) -> int:
    p = problem_of(case, complete_blocks_only)
    return lib().qlio_visible(ctypes.byref(p), sq, sk, r)


def max_compressed_len(case) -> int:
    if case.batch == 0:
        return 0
    return int(-(-int(max(0, case.seq_lens_k.max())) // case.cmp_ratio))


def score_topk(case, with_scores: bool = False, nthreads: int | None = None,
               complete_blocks_only: bool = False, rows=None):
    """Run the oracle.  Returns ``(indices[rows, k] int32, scores or None, error_mask)``.

    ``scores`` (when requested) is float32 ``[rows, max Lc]`` holding each visible key's fp32 score
    and NaN elsewhere.  ``rows`` (optional iterable of row numbers) limits the work to those rows;
    every other output row is -1.
    """
    L = lib()
    p = problem_of(case, complete_blocks_only)
    rows_total = int(L.qlio_rows(ctypes.byref(p)))
    k = case.sparse_count
    out = np.empty((max(rows_total, 0), k), dtype=np.int32)
    ld = max(1, max_compressed_len(case))
    scores = np.full((max(rows_total, 0), ld), np.nan, dtype=np.float32) if with_scores else None
    arrs = [np.ascontiguousarray(a) for a in (case.query, case.key, case.weights, case.q_scale,
                                               case.k_scale)]
    slq = None if case.seq_lens_q is None else np.ascontiguousarray(case.seq_lens_q, np.int32)
    slk = np.ascontiguousarray(case.seq_lens_k, np.int32)
    bt = np.ascontiguousarray(case.block_table, np.int32)
    mask = None
    if rows is not None:
        mask = np.zeros(max(rows_total, 1), dtype=np.uint8)
        mask[np.asarray(list(rows), dtype=np.int64)] = 1
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    err = L.qlio_score_topk(ctypes.byref(p), *[_ptr(a) for a in arrs], _ptr(slq), _ptr(slk),
                            _ptr(bt), _ptr(out), _ptr(scores), ld, _ptr(mask), int(nthreads))
    return out, scores, int(err)


# ------------------------------------------------------------------------------------ quantizer

def quantize(x_bf16: np.ndarray, fp8: bool, scale_f32: bool):
    """Per-(token, head) quantization of ``x_bf16`` (uint16 bfloat16 bits, [..., 128]): returns
    ``(codes [..., 128] (int8, or uint8 e4m3 codes), scales [...] (float16 or float32))``."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    n = x.size // 128
    codes = np.empty(x.shape, dtype=np.uint8 if fp8 else np.int8)
    scales = np.empty(x.shape[:-1], dtype=np.float32 if scale_f32 else np.float16)
    lib().qlio_quantize_vectors(1 if fp8 else 0, 1 if scale_f32 else 0, _ptr(x), n, _ptr(codes), _ptr(scales))
    return codes, scales


def quantize_keys(case, key_bf16: np.ndarray, token_batch, token_pos):
    """The paged key-cache write of ``key_bf16`` ([tokens, 128] bfloat16 bits) into ``case.key``
    and ``case.k_scale`` (in place) at the (batch, compressed position) of each token; returns the
    error mask."""
    p = problem_of(case)
    kb = np.ascontiguousarray(key_bf16, dtype=np.uint16)
    tb = np.ascontiguousarray(token_batch, dtype=np.int32)
    tp = np.ascontiguousarray(token_pos, dtype=np.int32)
    return lib().qlio_quantize_keys(ctypes.byref(p), _ptr(kb), len(tb), _ptr(tb), _ptr(tp),
                                    _ptr(case.block_table), _ptr(case.key), _ptr(case.k_scale))


# ------------------------------------------------------------------------------ downstream gather

def gather_kv(case, sparse_indices, kv, entry_bytes: int, kv_stride: int = 0, use_seq_lens_k: bool = True):
    """The sparse-attention gather: for every row and selected index, the KV entry at that
    compressed position of the row's batch through ``case.block_table``.  ``kv`` is the pool as
    bytes ([num_blocks, page bytes]); returns ``(out uint8 [rows, k, entry_bytes], counts int32
    [rows], error_mask)``."""
    p = problem_of(case)
    rows = int(lib().qlio_rows(ctypes.byref(p)))
    k = case.sparse_count
    idx = np.ascontiguousarray(sparse_indices, dtype=np.int32).reshape(rows, k)
    pool = np.ascontiguousarray(kv).view(np.uint8)
    out = np.full((rows, k, entry_bytes), 0xA5, dtype=np.uint8)   # every byte is written
    counts = np.empty(max(rows, 1), dtype=np.int32)[:rows]
    slq = None if case.seq_lens_q is None else np.ascontiguousarray(case.seq_lens_q, np.int32)
    slk = np.ascontiguousarray(case.seq_lens_k, np.int32) if use_seq_lens_k else None
    bt = np.ascontiguousarray(case.block_table, np.int32)
    err = lib().qlio_gather_kv(ctypes.byref(p), _ptr(slq), _ptr(slk), _ptr(bt), _ptr(idx), _ptr(pool),
                               int(entry_bytes), int(kv_stride), _ptr(out), _ptr(counts))
    return out, counts, int(err)
