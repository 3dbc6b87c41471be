"""Thin Python binding of ``libqli.so``, the GB300 quantized lightning indexer.

Every function here only marshals arguments to the C ABI declared in ``include/qli.h`` (same
names without the ``qli_`` prefix); all computation runs in the library's CUDA kernels.  Tensors
are torch CUDA tensors; the current torch stream is passed to the library.  The shared library is
loaded on first use; if it has not been built, that first use raises ImportError: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqli.so")
# the testing build (include/qli_testing.h): the same library plus a failure-detection switch;
# only the failure-detection tests select it, with use_testing_library() before the first call
TESTING_LIB_PATH = os.path.join(_HERE, "libqli_testing.so")
_lib_path = LIB_PATH

QLI_OK = 0
STATUS_NAMES = {0: "QLI_OK", 1: "QLI_ERR_INVALID_ARG", 2: "QLI_ERR_UNSUPPORTED",
                3: "QLI_ERR_WORKSPACE_TOO_SMALL", 4: "QLI_ERR_CUDA", 5: "QLI_ERR_DEVICE_BAD_INPUT",
                6: "QLI_ERR_DEVICE_TIMEOUT", 7: "QLI_ERR_NO_DEVICE"}
INT8, FP8_E4M3 = 0, 1
F16, F32 = 0, 1
BSND, TND = 0, 1
SPLIT_AUTO, SPLIT_ON, SPLIT_OFF = 0, 1, 2       # qli_split_topk
INT64_MAX = (1 << 63) - 1

# symbols include/qli.h declares
EXPORTS = ("qli_problem_init", "qli_validate", "qli_metadata_words", "qli_workspace_size",
           "qli_metadata", "qli_score_topk", "qli_score", "qli_topk", "qli_score_topk_static",
           "qli_workspace_init", "qli_get_device_error",
           "qli_plan_create", "qli_plan_launch", "qli_plan_destroy",
           "qli_quantize", "qli_quantize_keys", "qli_gather_kv",
           "qli_status_string", "qli_version")


class QliError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s: %s (%d)" % (what, STATUS_NAMES.get(status, "?"), status))


class Problem(ctypes.Structure):
    """Mirror of ``qli_problem``."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "max_q_tokens", "total_q_tokens", "num_heads_q", "num_heads_k", "head_dim",
        "qk_dtype", "scale_dtype", "layout_q", "num_blocks", "block_size", "max_blocks_per_seq",
        "sparse_count", "sparse_mode", "cmp_ratio", "query_quant_mode", "key_quant_mode",
        "return_value")] + [("pre_tokens", ctypes.c_int64), ("next_tokens", ctypes.c_int64),
                            ("max_seqlen_q", ctypes.c_int32), ("max_seqlen_k", ctypes.c_int32),
                            ("key_stride", ctypes.c_int32), ("mask_complete_blocks", ctypes.c_int32),
                            ("split_topk", ctypes.c_int32)]


def _load():
    if not os.path.exists(_lib_path):
        raise ImportError("%s is not built (run __graft_entry__.build() or "
                          "python sparse_attention_token_block_gb300/build.py)" % os.path.basename(_lib_path))
    L = ctypes.CDLL(_lib_path)
    if _lib_path == TESTING_LIB_PATH:
        L.qli_testing_set_stall.argtypes = [ctypes.c_int]
        L.qli_testing_set_stall.restype = None
        L.qli_testing_set_topk_ctas.argtypes = [ctypes.c_int]
        L.qli_testing_set_topk_ctas.restype = None
    vp, sz, i32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
    P = ctypes.POINTER(Problem)
    L.qli_problem_init.argtypes = [P]
    L.qli_problem_init.restype = None
    L.qli_validate.argtypes = [P, ctypes.POINTER(ctypes.c_char_p)]
    L.qli_validate.restype = ctypes.c_int
    L.qli_metadata_words.argtypes = [P]
    L.qli_metadata_words.restype = sz
    L.qli_workspace_size.argtypes = [P]
    L.qli_workspace_size.restype = sz
    L.qli_metadata.argtypes = [P, i32p, i32p, i32p, sz, vp]
    L.qli_metadata.restype = ctypes.c_int
    L.qli_score_topk.argtypes = [P, vp, vp, vp, vp, vp, i32p, i32p, i32p, i32p, sz, vp, sz, i32p,
                                 vp, vp]
    L.qli_score_topk.restype = ctypes.c_int
    L.qli_score.argtypes = [P, vp, vp, vp, vp, vp, i32p, i32p, i32p, i32p, sz, vp, sz, vp]
    L.qli_score.restype = ctypes.c_int
    L.qli_topk.argtypes = [P, i32p, i32p, sz, vp, sz, i32p, vp, vp]
    L.qli_topk.restype = ctypes.c_int
    L.qli_score_topk_static.argtypes = [P, vp, vp, vp, vp, vp, i32p, i32p, i32p, i32p, sz, i32p,
                                        vp, vp]
    L.qli_score_topk_static.restype = ctypes.c_int
    L.qli_workspace_init.argtypes = [vp, sz, vp]
    L.qli_workspace_init.restype = ctypes.c_int
    L.qli_get_device_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    L.qli_get_device_error.restype = ctypes.c_int
    L.qli_status_string.argtypes = [ctypes.c_int]
    L.qli_status_string.restype = ctypes.c_char_p
    L.qli_version.argtypes = []
    L.qli_version.restype = ctypes.c_int
    L.qli_plan_create.argtypes = [P, ctypes.c_int, vp, vp, vp, vp, vp, i32p, i32p, i32p, i32p, sz, vp,
                                  sz, i32p, vp, ctypes.POINTER(ctypes.c_void_p)]
    L.qli_plan_create.restype = ctypes.c_int
    L.qli_plan_launch.argtypes = [vp, vp]
    L.qli_plan_launch.restype = ctypes.c_int
    L.qli_plan_destroy.argtypes = [vp]
    L.qli_plan_destroy.restype = None
    L.qli_quantize.argtypes = [ctypes.c_int32, ctypes.c_int32, vp, ctypes.c_int64, vp, vp, vp]
    L.qli_quantize.restype = ctypes.c_int
    L.qli_quantize_keys.argtypes = [P, vp, ctypes.c_int64, i32p, i32p, i32p, vp, vp, vp, sz, vp]
    L.qli_quantize_keys.restype = ctypes.c_int
    L.qli_gather_kv.argtypes = [P, i32p, i32p, i32p, i32p, vp, ctypes.c_int64, ctypes.c_int64, vp, i32p, vp, sz,
                                vp]
    L.qli_gather_kv.restype = ctypes.c_int
    return L


_lib_handle = None


def use_testing_library():
    """Load the testing build (libqli_testing.so) instead of the product library.  Must be called
    before the first call into the library in this process."""
    global _lib_path
    if _lib_handle is not None and _lib_path != TESTING_LIB_PATH:
        raise RuntimeError("the product library is already loaded in this process")
    _lib_path = TESTING_LIB_PATH


def _get_lib():
    global _lib_handle
    if _lib_handle is None:
        _lib_handle = _load()
    return _lib_handle


def __getattr__(name):
    if name == "lib":
        return _get_lib()
    raise AttributeError(name)


# ------------------------------------------------------------------------------------ marshalling
def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def problem_init() -> Problem:
    p = Problem()
    _get_lib().qli_problem_init(ctypes.byref(p))
    return p


def validate(p: Problem):
    why = ctypes.c_char_p()
    st = _get_lib().qli_validate(ctypes.byref(p), ctypes.byref(why))
    return st, why.value.decode() if why.value else ""


def metadata_words(p: Problem) -> int:
    return int(_get_lib().qli_metadata_words(ctypes.byref(p)))


def workspace_size(p: Problem) -> int:
    return int(_get_lib().qli_workspace_size(ctypes.byref(p)))


def metadata(p: Problem, seq_lens_q, seq_lens_k, meta, stream=None) -> int:
    return _get_lib().qli_metadata(ctypes.byref(p), _ptr(seq_lens_q), _ptr(seq_lens_k), _ptr(meta),
                            meta.numel() if meta is not None else 0, _stream(stream))


def score_topk(p: Problem, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k,
               block_table, meta, workspace, sparse_indices, sparse_values=None, stream=None) -> int:
    return _get_lib().qli_score_topk(ctypes.byref(p), _ptr(query), _ptr(key), _ptr(weights),
                              _ptr(q_scale), _ptr(k_scale), _ptr(seq_lens_q), _ptr(seq_lens_k),
                              _ptr(block_table), _ptr(meta), meta.numel(), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(sparse_indices),
                              _ptr(sparse_values), _stream(stream))


def score(p: Problem, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k, block_table,
          meta, workspace, stream=None) -> int:
    return _get_lib().qli_score(ctypes.byref(p), _ptr(query), _ptr(key), _ptr(weights),
                                _ptr(q_scale), _ptr(k_scale), _ptr(seq_lens_q), _ptr(seq_lens_k),
                                _ptr(block_table), _ptr(meta), meta.numel(), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))


def topk(p: Problem, block_table, meta, workspace, sparse_indices, sparse_values=None, stream=None) -> int:
    return _get_lib().qli_topk(ctypes.byref(p), _ptr(block_table), _ptr(meta), meta.numel(),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _ptr(sparse_indices), _ptr(sparse_values), _stream(stream))


def score_topk_static(p: Problem, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k,
                      block_table, meta, sparse_indices, device_error=None, stream=None) -> int:
    """qli_score_topk_static: no workspace argument; the library's own fixed scratch is used."""
    return _get_lib().qli_score_topk_static(
        ctypes.byref(p), _ptr(query), _ptr(key), _ptr(weights), _ptr(q_scale), _ptr(k_scale),
        _ptr(seq_lens_q), _ptr(seq_lens_k), _ptr(block_table), _ptr(meta), meta.numel(),
        _ptr(sparse_indices), _ptr(device_error), _stream(stream))


def plan_create(p: Problem, with_metadata, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k,
                block_table, meta, workspace, sparse_indices, sparse_values=None):
    """qli_plan_create: returns (status, plan handle or None)."""
    h = ctypes.c_void_p(None)
    st = _get_lib().qli_plan_create(
        ctypes.byref(p), 1 if with_metadata else 0, _ptr(query), _ptr(key), _ptr(weights), _ptr(q_scale),
        _ptr(k_scale), _ptr(seq_lens_q), _ptr(seq_lens_k), _ptr(block_table), _ptr(meta), meta.numel(),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(sparse_indices),
        _ptr(sparse_values), ctypes.byref(h))
    return st, (h.value if st == QLI_OK else None)


def plan_launch(plan, stream=None) -> int:
    return _get_lib().qli_plan_launch(plan, _stream(stream))


def plan_destroy(plan) -> None:
    _get_lib().qli_plan_destroy(plan)


def quantize(qk_dtype, scale_dtype, x, codes, scales, stream=None) -> int:
    """qli_quantize: ``x`` bfloat16 [..., 128] -> ``codes`` (int8 / uint8 e4m3 bytes, same shape)
    and ``scales`` ([...], float16 or float32)."""
    return _get_lib().qli_quantize(qk_dtype, scale_dtype, _ptr(x), x.numel() // 128, _ptr(codes),
                                   _ptr(scales), _stream(stream))


def quantize_keys(p: Problem, key_bf16, token_batch, token_pos, block_table, key, k_scale,
                  workspace=None, stream=None) -> int:
    """qli_quantize_keys: write ``key_bf16`` ([tokens, 128] bfloat16) into the paged pool ``key``
    and ``k_scale`` at each token's (batch, compressed position)."""
    return _get_lib().qli_quantize_keys(
        ctypes.byref(p), _ptr(key_bf16), token_batch.numel(), _ptr(token_batch), _ptr(token_pos),
        _ptr(block_table), _ptr(key), _ptr(k_scale), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream))


def gather_kv(p: Problem, seq_lens_q, seq_lens_k, block_table, sparse_indices, kv, entry_bytes, out,
              counts=None, kv_stride=0, workspace=None, stream=None) -> int:
    """qli_gather_kv: ``out`` [rows, sparse_count, entry_bytes] (uint8) receives the KV entries the
    indices select through the block_table; ``counts`` (optional int32 [rows]) the entries copied."""
    return _get_lib().qli_gather_kv(
        ctypes.byref(p), _ptr(seq_lens_q), _ptr(seq_lens_k), _ptr(block_table), _ptr(sparse_indices), _ptr(kv),
        int(entry_bytes), int(kv_stride), _ptr(out), _ptr(counts), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream))


def workspace_init(workspace, stream=None) -> int:
    return _get_lib().qli_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))


def get_device_error(workspace, stream=None):
    bits = ctypes.c_uint32(0)
    st = _get_lib().qli_get_device_error(_ptr(workspace), _stream(stream), ctypes.byref(bits))
    return st, int(bits.value)


def status_string(st: int) -> str:
    return _get_lib().qli_status_string(st).decode()


def version() -> int:
    return _get_lib().qli_version()


def check(st: int, what: str = "qli"):
    if st != QLI_OK:
        raise QliError(st, what)


# ------------------------------------------------------------------------------------ convenience
def make_problem(*, batch, layout_q=BSND, max_q_tokens=0, total_q_tokens=0, qk_dtype=INT8,
                 scale_dtype=F16, num_blocks, block_size, max_blocks_per_seq, sparse_count,
                 sparse_mode, cmp_ratio, max_seqlen_q, max_seqlen_k, return_value=0, key_stride=0,
                 mask_complete_blocks=0, split_topk=0) -> Problem:
    p = problem_init()
    p.batch = batch
    p.layout_q = layout_q
    p.max_q_tokens = max_q_tokens
    p.total_q_tokens = total_q_tokens
    p.qk_dtype = qk_dtype
    p.scale_dtype = scale_dtype
    p.num_blocks = num_blocks
    p.block_size = block_size
    p.max_blocks_per_seq = max_blocks_per_seq
    p.sparse_count = sparse_count
    p.sparse_mode = sparse_mode
    p.cmp_ratio = cmp_ratio
    p.max_seqlen_q = max_seqlen_q
    p.max_seqlen_k = max_seqlen_k
    p.return_value = return_value
    p.key_stride = key_stride
    p.mask_complete_blocks = mask_complete_blocks
    p.split_topk = split_topk
    return p


class Indexer:
    """Owns the metadata, workspace and output buffers of one problem shape.

    ``run`` enqueues qli_metadata (when ``refresh_metadata``) and qli_score_topk on the current
    stream and returns the int32 ``sparse_indices`` tensor ([rows, sparse_count]).
    """

    def __init__(self, p: Problem, device="cuda"):
        import torch
        st, why = validate(p)
        if st != QLI_OK:
            raise QliError(st, "problem: " + why)
        self.p = p
        self.meta = torch.zeros(metadata_words(p), dtype=torch.int32, device=device)
        nbytes = workspace_size(p)
        self.workspace = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device=device)
        check(workspace_init(self.workspace), "workspace_init")
        rows = p.batch * p.max_q_tokens if p.layout_q == BSND else p.total_q_tokens
        self.rows = rows
        self.out = torch.empty((rows, p.sparse_count), dtype=torch.int32, device=device)
        # the indices' scores (README return_value), when the problem asks for them
        self.values = (torch.empty((rows, p.sparse_count), dtype=torch.float32, device=device)
                       if p.return_value else None)

    def run(self, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k, block_table,
            refresh_metadata=True, out=None):
        if refresh_metadata:
            check(metadata(self.p, seq_lens_q, seq_lens_k, self.meta), "metadata")
        o = self.out if out is None else out
        check(score_topk(self.p, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k,
                         block_table, self.meta, self.workspace, o, self.values), "score_topk")
        return o

    def plan(self, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k, block_table,
             with_metadata=True, out=None):
        """A ``Plan`` replaying this call on these tensors (their addresses are captured)."""
        o = self.out if out is None else out
        st, h = plan_create(self.p, with_metadata, query, key, weights, q_scale, k_scale, seq_lens_q,
                            seq_lens_k, block_table, self.meta, self.workspace, o, self.values)
        check(st, "plan_create")
        # the captured tensors stay referenced as long as the plan lives
        return Plan(h, (query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k, block_table,
                        self.meta, self.workspace, o, self.values))

    def device_error(self):
        return get_device_error(self.workspace)

    def score_lines(self):
        """The last call's per-row ordered score codes decoded to float32 ([rows, ld]); entries of
        keys that were not visible hold stale values.  Debug/test aid."""
        import torch
        lc = -(-self.p.max_seqlen_k // self.p.cmp_ratio)
        ld = max(128, -(-lc // 128) * 128)
        codes = self.workspace.view(torch.uint8)[256:256 + self.rows * ld * 4].view(torch.int32)
        codes = codes.view(self.rows, ld).to(torch.int64) & 0xFFFFFFFF
        neg = codes < 0x80000000
        bits = torch.where(neg, (~codes) & 0xFFFFFFFF, codes & 0x7FFFFFFF)
        return bits.to(torch.int32).view(torch.float32).reshape(self.rows, ld)

    def split_candidates(self):
        """With the split-local selection on: the last call's candidate codes and key indices
        ([rows, ld] int32 each, valid where the tile words say) and tile words ([rows, ld / 128]
        int32: count of the tile's candidates, top bit set when they are in the candidate lines
        rather than the score line).  Debug/test aid."""
        import torch
        lc = -(-self.p.max_seqlen_k // self.p.cmp_ratio)
        ld = max(128, -(-lc // 128) * 128)
        line = self.rows * ld * 4
        ws = self.workspace.view(torch.uint8)
        o = 256 + line
        code = ws[o:o + line].view(torch.int32).view(self.rows, ld)
        idx = ws[o + line:o + 2 * line].view(torch.int32).view(self.rows, ld)
        info = ws[o + 2 * line:o + 2 * line + line // 128].view(torch.int32).view(self.rows, ld // 128)
        return code, idx, info


class Plan:
    """One indexer call captured as a CUDA graph (qli_plan_*); ``launch`` replays it on the current
    stream.  Holds references to the captured tensors."""

    def __init__(self, handle, keep):
        self._h = handle
        self._keep = keep

    def launch(self, stream=None):
        check(plan_launch(self._h, stream), "plan_launch")

    def close(self):
        if self._h is not None:
            plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
