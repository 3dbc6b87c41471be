"""Seeded synthetic inputs for the quantized lightning indexer.

This module only draws random inputs and lays them out in the documented
shapes; it holds none of the indexer's arithmetic, so both the CPU oracle and
the CUDA path can be fed from it.

Shapes and value distributions follow the Ascend ``VllmQuantLightningIndexer``
README (single-operator call example and parameter table):

* query   BSND ``[B, S1, 64, 128]`` or TND ``[T, 64, 128]``, int8 or fp8-e4m3
* key     PA_BSND pool ``[num_blocks, block_size, 1, 128]``
* k_scale ``[num_blocks, block_size, 1]``; q_scale / weights ``[..., 64]``
* block_table ``[B, max_blocks_per_seq]`` int32

int8 values are drawn the way the README's example does: a float64 uniform on
[-128, 127) converted to int8 by truncation toward zero.  fp8 values are a
float normal times 4 cast to ``float8_e4m3fn`` (round to nearest even);
codes that decode to NaN are never produced at these magnitudes.

The key pool is sized for the number of compressed keys each batch holds,
``ceil(S_k / cmp_ratio)``: the fifth workload spells that length out.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

NUM_HEADS_Q = 64
NUM_HEADS_K = 1
HEAD_DIM = 128

INT8 = "int8"
FP8 = "fp8_e4m3"
F16 = "f16"
F32 = "f32"


@dataclasses.dataclass
class Case:
    """One indexer invocation: every input array (numpy, host) and the attributes."""

    name: str
    layout_q: str                 # "BSND" or "TND"
    qk_dtype: str                 # INT8 or FP8 (FP8 arrays hold the raw e4m3 codes as uint8)
    scale_dtype: str              # F16 or F32 (weights, q_scale and k_scale share it)
    batch: int
    s1: int                       # BSND query rows per batch (0 for TND)
    total_q: int                  # TND rows T (0 for BSND)
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    sparse_count: int
    sparse_mode: int
    cmp_ratio: int
    query: np.ndarray             # int8 / uint8 codes
    key: np.ndarray               # int8 / uint8 codes
    weights: np.ndarray
    q_scale: np.ndarray
    k_scale: np.ndarray
    seq_lens_q: Optional[np.ndarray]  # int32 [B] (TND: prefix sums) or None
    seq_lens_k: np.ndarray        # int32 [B], original (uncompressed) key tokens
    block_table: np.ndarray       # int32 [B, max_blocks_per_seq]
    key_stride: int = 0           # elements between key pages (0: contiguous, block_size * 128)

    @property
    def rows(self) -> int:
        return self.batch * self.s1 if self.layout_q == "BSND" else self.total_q

    @property
    def max_seqlen_k(self) -> int:
        return int(self.seq_lens_k.max()) if self.batch else 0

    @property
    def max_seqlen_q(self) -> int:
        if self.layout_q == "BSND":
            return int(self.seq_lens_q.max()) if self.seq_lens_q is not None and self.batch else self.s1
        if self.batch == 0:
            return 0
        cum = np.concatenate([[0], self.seq_lens_q.astype(np.int64)])
        return int(np.diff(cum).max())


def _int8_like_readme(draw: np.ndarray) -> np.ndarray:
    # float -> int8 by truncation toward zero, as torch's .to(torch.int8) does
    return np.trunc(draw).astype(np.int8)


def _int8_like_readme_fast(rng, shape) -> np.ndarray:
    """The distribution of _int8_like_readme(U(-128, 127)) drawn as integers: -127 .. 126 with
    probability 1/255 each and 0 with 2/255 (the draws in (-1, 1) truncate to 0), i.e. a uniform
    draw over -127 .. 127 with 127 sent to 0 -- without a float array of the whole shape."""
    v = rng.integers(-127, 128, size=shape, dtype=np.int8)
    v[v == 127] = 0
    return v


def _fp8_codes(x: np.ndarray) -> np.ndarray:
    import torch  # the float8 cast is a library routine; only used here for input drawing

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    codes = t.view(torch.uint8).numpy().copy()
    assert not np.any((codes & 0x7F) == 0x7F), "NaN code drawn"
    return codes


def _scale_cast(x: np.ndarray, scale_dtype: str) -> np.ndarray:
    return x.astype(np.float16) if scale_dtype == F16 else x.astype(np.float32)


def _pages_for(seq_lens_k, cmp_ratio, block_size) -> List[int]:
    out = []
    for s in seq_lens_k:
        compressed = -(-int(s) // cmp_ratio)
        out.append(-(-compressed // block_size))
    return out


def paged_layout(seq_lens_k, cmp_ratio, block_size, rng, permute=True, extra_pages=0, width=None):
    """Allocate pages for each batch and build the block_table.

    Returns (num_blocks, block_table).  Pages are handed out as one seeded
    random permutation of the whole pool (or in order when ``permute`` is
    false); unused table slots hold -1.
    """
    pages = _pages_for(seq_lens_k, cmp_ratio, block_size)
    total = sum(pages) + extra_pages
    w = max(pages) if pages else 0
    if width is not None:
        w = max(w, width)
    w = max(w, 1)
    perm = rng.permutation(total).astype(np.int32) if permute else np.arange(total, dtype=np.int32)
    table = np.full((len(pages), w), -1, dtype=np.int32)
    pos = 0
    for b, p in enumerate(pages):
        table[b, :p] = perm[pos:pos + p]
        pos += p
    return max(total, 1), table


def make_case(name, *, layout_q="BSND", qk_dtype=INT8, scale_dtype=F16, batch=1, s1=1,
              q_lens=None, seq_lens_k=(256,), block_size=128, sparse_count=64, sparse_mode=0,
              cmp_ratio=1, seed=0, permute=True, pass_seq_lens_q=False, extra_pages=0,
              table_width=None, fast_draw=False) -> Case:
    """General seeded case.  ``fast_draw``: int8 codes by _int8_like_readme_fast (same distribution,
    another stream of draws; for pools of hundreds of MB).

    BSND: ``batch`` x ``s1`` query rows; ``q_lens`` (optional) gives
    actual_seq_lengths_query per batch.  TND: ``q_lens`` is the per-sequence
    query length list; the passed tensor holds its prefix sums.
    """
    rng = np.random.default_rng(seed)
    seq_lens_k = np.asarray(seq_lens_k, dtype=np.int32)
    B = len(seq_lens_k) if layout_q == "TND" else batch
    assert len(seq_lens_k) == B
    num_blocks, table = paged_layout(seq_lens_k, cmp_ratio, block_size, rng, permute,
                                     extra_pages, table_width)
    if layout_q == "BSND":
        rows_shape = (B, s1, NUM_HEADS_Q)
        if q_lens is not None:
            seq_lens_q = np.asarray(q_lens, dtype=np.int32)
        elif pass_seq_lens_q:
            seq_lens_q = np.full(B, s1, dtype=np.int32)
        else:
            seq_lens_q = None
        total_q = 0
    else:
        q_lens = np.asarray(q_lens, dtype=np.int64)
        seq_lens_q = np.cumsum(q_lens).astype(np.int32)
        total_q = int(seq_lens_q[-1]) if B else 0
        rows_shape = (total_q, NUM_HEADS_Q)
        s1 = 0
    q_shape = rows_shape + (HEAD_DIM,)
    k_shape = (num_blocks, block_size, NUM_HEADS_K, HEAD_DIM)
    if qk_dtype == INT8 and fast_draw:
        key = _int8_like_readme_fast(rng, k_shape)
        query = _int8_like_readme_fast(rng, q_shape)
    elif qk_dtype == INT8:
        key = _int8_like_readme(rng.uniform(-128, 127, k_shape))
        query = _int8_like_readme(rng.uniform(-128, 127, q_shape))
    else:
        key = _fp8_codes(rng.standard_normal(k_shape) * 4.0)
        query = _fp8_codes(rng.standard_normal(q_shape) * 4.0)
    k_scale = _scale_cast(rng.uniform(0, 10, (num_blocks, block_size, NUM_HEADS_K)), scale_dtype)
    q_scale = _scale_cast(rng.uniform(0, 10, rows_shape), scale_dtype)
    weights = _scale_cast(rng.uniform(0, 0.01, rows_shape), scale_dtype)
    return Case(name=name, layout_q=layout_q, qk_dtype=qk_dtype, scale_dtype=scale_dtype,
                batch=B, s1=s1, total_q=total_q, block_size=block_size, num_blocks=num_blocks,
                max_blocks_per_seq=table.shape[1], sparse_count=sparse_count,
                sparse_mode=sparse_mode, cmp_ratio=cmp_ratio, query=query, key=key,
                weights=weights, q_scale=q_scale, k_scale=k_scale, seq_lens_q=seq_lens_q,
                seq_lens_k=seq_lens_k, block_table=table)


# ----------------------------------------------------------------------------------------------
# The five named workloads
# ----------------------------------------------------------------------------------------------

def tiny_decode() -> Case:
    """B=1, one query token, S_k=256 in two 128-key pages, table [[0,1]], k=64, mode 0."""
    return make_case("tiny_decode", batch=1, s1=1, seq_lens_k=[256], block_size=128,
                     sparse_count=64, sparse_mode=0, cmp_ratio=1, seed=0, permute=False)


def page_decode() -> Case:
    """The README's single-operator example, drawn in its order from ``np.random.seed(0)``.

    B=24, S1=4, S_k=512 in 4 pages of 128 per batch, identity block_table,
    k=512, sparse_mode 0, cmp_ratio 1.
    """
    b, s1, s2, bs, n1, n2, d = 24, 4, 512, 128, NUM_HEADS_Q, NUM_HEADS_K, HEAD_DIM
    np.random.seed(0)
    mb = (s2 + bs - 1) // bs
    table = np.arange(b * mb, dtype=np.int32).reshape(b, -1)
    key = _int8_like_readme(np.random.uniform(-128, 127, (b * mb, bs, n2, d)))
    k_scale = np.random.uniform(0, 10, (b * mb, bs, n2)).astype(np.float16)
    query = _int8_like_readme(np.random.uniform(-128, 127, (b, s1, n1, d)))
    q_scale = np.random.uniform(0, 10, (b, s1, n1)).astype(np.float16)
    weights = np.random.uniform(0, 0.01, (b, s1, n1)).astype(np.float16)
    seq_lens_q = np.random.uniform(s1, s1, (b,)).astype(np.int32)
    seq_lens_k = np.random.uniform(s2, s2, (b,)).astype(np.int32)
    return Case(name="page_decode", layout_q="BSND", qk_dtype=INT8, scale_dtype=F16, batch=b,
                s1=s1, total_q=0, block_size=bs, num_blocks=b * mb, max_blocks_per_seq=mb,
                sparse_count=512, sparse_mode=0, cmp_ratio=1, query=query, key=key,
                weights=weights, q_scale=q_scale, k_scale=k_scale, seq_lens_q=seq_lens_q,
                seq_lens_k=seq_lens_k, block_table=table)


def long_decode(seed: int = 3, batch: int = 32) -> Case:
    """B=32, one query token each, S_k ~ U{8192..32768}, 64-key pages, k=2048, causal."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(8192, 32768, size=batch, endpoint=True).astype(np.int32)
    return make_case("long_decode", batch=batch, s1=1, seq_lens_k=lens, block_size=64,
                     sparse_count=2048, sparse_mode=3, cmp_ratio=1, seed=seed + 100,
                     permute=True, pass_seq_lens_q=True)


def long_context_decode(seed: int = 9, batch: int = 32) -> Case:
    """B=32, one query token each, S_k ~ U{65536..131072}, 64-key pages, k=2048, causal: rows longer
    than one top-k CTA's row cache (not one of the five workloads; timed beside them)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(65536, 131072, size=batch, endpoint=True).astype(np.int32)
    return make_case("long_context_decode", batch=batch, s1=1, seq_lens_k=lens, block_size=64,
                     sparse_count=2048, sparse_mode=3, cmp_ratio=1, seed=seed + 100,
                     permute=True, pass_seq_lens_q=True, fast_draw=True)


def fp8_compressed_decode(seed: int = 4, batch: int = 16) -> Case:
    """B=16, S1=2, fp8 q/k, S_k ~ U{16384..65536} compressed 4x, 128-key pages, fp32 scales."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(16384, 65536, size=batch, endpoint=True).astype(np.int32)
    return make_case("fp8_compressed_decode", batch=batch, s1=2, qk_dtype=FP8, scale_dtype=F32,
                     seq_lens_k=lens, block_size=128, sparse_count=2048, sparse_mode=3,
                     cmp_ratio=4, seed=seed + 100, permute=True, pass_seq_lens_q=True)


def varlen_prefill(seed: int = 5, lens=(1024, 2048, 4096, 8192)) -> Case:
    """TND prefill: sequences of the given lengths, key length = query length, causal."""
    return make_case("varlen_prefill", layout_q="TND", q_lens=list(lens), seq_lens_k=list(lens),
                     block_size=128, sparse_count=2048, sparse_mode=3, cmp_ratio=1, seed=seed,
                     permute=True)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "page_decode": page_decode,
    "long_decode": long_decode,
    "fp8_compressed_decode": fp8_compressed_decode,
    "varlen_prefill": varlen_prefill,
    "long_context_decode": long_context_decode,    # beside the five: rows beyond one CTA's cache
}


# ----------------------------------------------------------------------------------------------
# Unquantized activations (inputs of the upstream per-token-head quantizer)
# ----------------------------------------------------------------------------------------------

def bf16_vectors(shape, seed: int, special: bool = True) -> np.ndarray:
    """Seeded bfloat16 bit patterns (uint16) of ``shape`` (last axis 128): normal draws, each
    vector scaled by a log-uniform magnitude in [1e-3, 1e3] (activations whose range differs from
    token to token and head to head).  Values are truncated to bfloat16, so they are exact.

    With ``special`` the first vectors (as many as fit) are degenerate ones: all zero; magnitudes
    near 1e-38 (scales in the float subnormal range); magnitudes near 1e10 (scales beyond the
    float16 range); integers with one element 127 and the rest at k + 1/2 (every quotient an exact
    halfway case for int8 codes); one element 448 with the rest at midpoints of the e4m3 grid
    (halfway cases for e4m3 codes); and magnitudes near 1e30 mixed with signed zeros and -1e-40
    (zero and underflowing quotients, whose sign the e4m3 code keeps)."""
    rng = np.random.default_rng(seed)
    shape = tuple(shape)
    assert shape[-1] == HEAD_DIM
    n = int(np.prod(shape[:-1]))
    mag = np.exp(rng.uniform(math.log(1e-3), math.log(1e3), size=(n, 1)))
    x = (rng.normal(0.0, 1.0, size=(n, HEAD_DIM)) * mag).astype(np.float32)
    if special:
        extra = []
        extra.append(np.zeros(HEAD_DIM, np.float32))
        extra.append((rng.normal(0.0, 1.0, HEAD_DIM) * 1e-38).astype(np.float32))
        extra.append((rng.normal(0.0, 1.0, HEAD_DIM) * 1e10).astype(np.float32))
        halves = rng.integers(-127, 127, size=HEAD_DIM) + 0.5
        halves[rng.integers(0, HEAD_DIM)] = 127.0 * (1 if rng.integers(0, 2) else -1)
        extra.append(halves.astype(np.float32))
        # e4m3 grid below 448: exponents 2^-6 .. 2^8 with 3 mantissa bits; midpoints between neighbours
        grid = np.array(sorted({m / 8.0 * 2.0 ** e for e in range(-6, 9) for m in range(8, 16)} |
                               {m / 8.0 * 2.0 ** -6 for m in range(0, 8)}))
        grid = grid[grid <= 448.0]
        mids = (grid[:-1] + grid[1:]) / 2.0
        pick = mids[rng.integers(0, len(mids), size=HEAD_DIM)] * rng.choice([-1.0, 1.0], size=HEAD_DIM)
        pick[rng.integers(0, HEAD_DIM)] = 448.0
        extra.append(pick.astype(np.float32))
        # signed zeros, and tiny negative elements beside a huge maximum (their quotients underflow)
        sz = (rng.normal(0.0, 1.0, HEAD_DIM) * 1e30).astype(np.float32)
        sz[::4] = -0.0
        sz[1::8] = 0.0
        sz[2::16] = -1e-40
        extra.append(sz)
        m = min(len(extra), n)
        x[:m] = np.stack(extra[:m])
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    return bits.reshape(shape)


# ----------------------------------------------------------------------------------------------
# The attention's KV cache (input of the downstream gather)
# ----------------------------------------------------------------------------------------------

def kv_pool(case: Case, entry_bytes: int, pad: int = 0, seed: int = 0) -> np.ndarray:
    """Random bytes standing for the attention's paged KV cache of ``case``: the same pages as the
    key pool (``case.num_blocks`` pages of ``case.block_size`` entries, addressed by the same
    block_table), ``entry_bytes`` per entry, ``pad`` junk bytes after every page.  Returns uint8
    [num_blocks, block_size * entry_bytes + pad]."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=(case.num_blocks, case.block_size * entry_bytes + pad), dtype=np.uint8)


def random_indices(case: Case, seed: int, frac_pad: float = 0.2) -> np.ndarray:
    """Seeded stand-ins for an indexer's output: per row, distinct compressed positions of the
    row's batch in random order (up to sparse_count of them, a random share of up to ``frac_pad``
    left out), then -1 padding.  int32 [rows, sparse_count]."""
    rng = np.random.default_rng(seed)
    rows, k = case.rows, case.sparse_count
    lc = -(-case.seq_lens_k.astype(np.int64) // case.cmp_ratio)
    if case.layout_q == "BSND":
        b = np.arange(rows) // max(case.s1, 1)
    else:
        b = np.searchsorted(case.seq_lens_q, np.arange(rows), side="right")
    idx = np.full((rows, k), -1, np.int32)
    for r in range(rows):
        if b[r] >= case.batch:
            continue
        n = int(min(k, lc[b[r]]))
        m = int(n * (1 - frac_pad * rng.random()))
        idx[r, :m] = rng.choice(int(lc[b[r]]), size=m, replace=False)
    return idx


# ----------------------------------------------------------------------------------------------
# Marshalling for the CUDA library (torch device tensors and the problem attributes)
# ----------------------------------------------------------------------------------------------

def with_key_stride(case: Case, pad: int, seed: int = 0) -> Case:
    """The same case with its key pool laid out with ``pad`` junk elements after every page, so the
    stride of the pool's first axis is block_size * 128 + pad (the indexer's ``stride`` attribute).
    ``key`` becomes the strided buffer, [num_blocks, block_size * 128 + pad]."""
    nb, page = case.num_blocks, case.block_size * HEAD_DIM
    stride = page + pad
    rng = np.random.default_rng(seed)
    buf = rng.integers(0, 256, size=(nb, stride)).astype(np.uint8).view(case.key.dtype)
    buf[:, :page] = case.key.reshape(nb, page)
    return dataclasses.replace(case, key=buf, key_stride=stride)


def problem_kwargs(case: Case) -> dict:
    """Attributes of ``case`` as keyword arguments of the binding's ``make_problem``."""
    return dict(batch=case.batch, layout_q=0 if case.layout_q == "BSND" else 1,
                max_q_tokens=case.s1, total_q_tokens=case.total_q,
                qk_dtype=0 if case.qk_dtype == INT8 else 1,
                scale_dtype=0 if case.scale_dtype == F16 else 1, num_blocks=case.num_blocks,
                block_size=case.block_size, max_blocks_per_seq=case.max_blocks_per_seq,
                sparse_count=case.sparse_count, sparse_mode=case.sparse_mode,
                cmp_ratio=case.cmp_ratio, max_seqlen_q=case.max_seqlen_q,
                max_seqlen_k=case.max_seqlen_k, key_stride=case.key_stride)


def to_device(case: Case, device="cuda") -> dict:
    """Copy every input array of ``case`` to ``device`` as a torch tensor (codes keep their bytes)."""
    import torch

    def t(a, dtype=None):
        if a is None:
            return None
        x = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            x = x.view(dtype)
        return x.to(device)

    return dict(query=t(case.query.view(np.uint8)), key=t(case.key.view(np.uint8)),
                weights=t(case.weights), q_scale=t(case.q_scale), k_scale=t(case.k_scale),
                seq_lens_q=t(case.seq_lens_q), seq_lens_k=t(case.seq_lens_k),
                block_table=t(case.block_table))
