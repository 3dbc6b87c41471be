"""Benchmark of the quantized lightning indexer on one or more GB300s.

A step is one pass of the whole hot path over one batch of synthetic input: the work split
(qli_metadata), the scoring kernel (qli_score: paged key gather, tensor-core Q.K^T, fused
dequant/ReLU/head-sum/mask epilogue) and the top-k (qli_topk).  The default workload is the
long-context decode: 32 sequences, one query token each, 64 int8 heads of dim 128, key lengths
uniform in [8192, 32768] in 64-key pages under a random block_table, sparse_count 2048, causal.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events on the launching
stream with an L2 flush (a 512 MB write, then a read of it) between steps, outside the events;
barrier + synchronize around the timed region; the maximum over ranks.  A timed step replays the
library's execution plan (the three launches captured once as a CUDA graph, qli_plan_*), as a
serving loop with fixed buffers runs them; ``--no-graph`` times plain stream launches instead, and
the line also reports that time.  A further pass of up to 50 steps puts events between the three
kernels, for the per-stage times and the scoring kernel's roofline.  SM clocks and throttle
reasons are sampled with nvidia-smi over ~1.5 s of identical untimed load steps ending where the
timed steps begin, and through the timed steps.  Printed: one JSON line.

``--impl reference`` times the CPU oracle instead (the reference arm): the plain C implementation
run on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

OPS_PER_PAIR = 2 * 64 * 128          # 64 heads x 128-dim dot, multiply + add
METRIC = "indexer GOPS (algorithmic: 16384 ops per visible query-key pair)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "score_kernel_long_decode.md")
SCORE_SOURCES = ["qli_score.cuh", "qli_ptx.cuh", "qli_internal.cuh"]
QUANT_PROFILE = os.path.join(ROOT, "profiles", "quantize_kernel_prefill.md")
QUANT_SOURCES = ["qli_quant.cu", "qli_ptx.cuh", "qli_internal.cuh"]
GATHER_PROFILE = os.path.join(ROOT, "profiles", "gather_kernel_long_decode.md")
GATHER_SOURCES = ["qli_gather.cu", "qli_ptx.cuh", "qli_internal.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_decode", choices=sorted(W.WORKLOADS))
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling)")
    ap.add_argument("--flush-mb", type=int, default=512)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time stream launches instead of the captured execution plan")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true", help="skip the clock-sampling load window")
    ap.add_argument("--op", default="indexer", choices=["indexer", "quantize", "gather", "mma"],
                    help="indexer: the indexer step (default); quantize: the upstream quantizer; "
                         "gather: the downstream sparse-attention gather; mma: the rate of the score "
                         "kernel's tensor-core instruction form (libqli_peak.so)")
    ap.add_argument("--entry-bytes", type=int, default=512, help="KV entry size of --op gather")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload timings of the other configurations")
    return ap.parse_args()


def make_workload(name, batch, rank):
    fn = W.WORKLOADS[name]
    if name == "long_decode":
        return fn(seed=3 + 1000 * rank, batch=batch or 32)
    if name == "fp8_compressed_decode":
        return fn(seed=4 + 1000 * rank, batch=batch or 16)
    if name == "long_context_decode":
        return fn(seed=9 + 1000 * rank, batch=batch or 32)
    return fn()


def visible_pairs(case):
    """Visible (query row, compressed key) pairs of the workload: Lc = ceil(S_k / cmp_ratio) keys
    per sequence; under sparse_mode 3 row r of Sq sees min(Lc, ceil((S_k - Sq + r + 1) / cmp))."""
    c = case.cmp_ratio
    total = 0
    lo = 0
    for b in range(case.batch):
        sk = int(case.seq_lens_k[b])
        if case.layout_q == "BSND":
            sq = case.s1 if case.seq_lens_q is None else int(case.seq_lens_q[b])
        else:
            hi = int(case.seq_lens_q[b])
            sq, lo = hi - lo, hi
        lc = -(-sk // c)
        for r in range(sq):
            if case.sparse_mode == 0:
                total += lc
            else:
                pos = sk - sq + r
                total += 0 if pos < 0 else min(lc, -(-(pos + 1) // c))
    return total


def workload_stats(case):
    """Visible pairs, keys read (once per sequence) and algorithmic bytes of the scoring stage."""
    pairs = visible_pairs(case)
    esz = 2 if case.scale_dtype == W.F16 else 4
    lc = [-(-int(s) // case.cmp_ratio) for s in case.seq_lens_k]
    keys = int(sum(lc))
    pages = int(sum(-(-x // case.block_size) for x in lc))
    rows = case.rows
    score_bytes = keys * (128 + esz) + rows * 64 * (128 + 2 * esz) + pages * 4
    total_bytes = score_bytes + rows * case.sparse_count * 4 + case.batch * 8
    return dict(pairs=pairs, keys=keys, rows=rows, score_bytes=score_bytes,
                total_bytes=total_bytes)


def max_over_ranks(x, dist, device):
    """The largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gops(pairs_per_rank, steps, world, total_ms):
    """Algorithmic GOPS of the whole job: every rank scores its own workload (weak scaling), the
    time is the slowest rank's."""
    return pairs_per_rank * OPS_PER_PAIR * steps * world / (total_ms * 1e-3) / 1e9


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense 16-bit tensor-core peak (TFLOP/s): the measured bf16 burst figure (the score kernel is
    timed alone between events; its kind::f16 MMAs run at the bf16 rate)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def recorded_traffic(profile=PROFILE_TRAFFIC, sources=SCORE_SOURCES):
    """Per-launch DRAM bytes of a kernel from its committed ncu summary, if that summary was taken
    on the current kernel source (else None)."""
    try:
        text = open(profile).read()
    except OSError:
        return None, None
    h = hashlib.sha256()
    for s in sources:
        with open(os.path.join(ROOT, "sparse_attention_token_block_gb300", "csrc", s), "rb") as f:
            h.update(f.read())
    sha = h.hexdigest()[:16]
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha") != sha:
        return None, sha
    try:
        return float(vals["traffic_bytes_per_launch"]), sha
    except (KeyError, ValueError):
        return None, sha


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx),
                "samples": len(sm), "reasons": sorted(reasons)}


def cpu_baseline(case, budget_s=15.0):
    """Time the oracle (as it stands) on a bounded sample of the workload: whole sequences, as
    many as fit in about ``budget_s`` of wall time on the host cores."""
    import oracle
    nthreads = os.cpu_count() or 1
    oracle.build()
    if case.layout_q != "BSND":
        take, sub = case.batch, case
    else:
        t0 = time.perf_counter()
        oracle.score_topk(subcase(case, [0]), nthreads=nthreads)
        one = max(time.perf_counter() - t0, 1e-3)
        take = int(max(1, min(case.batch, budget_s / one)))
        sub = subcase(case, list(range(take)))
    t0 = time.perf_counter()
    oracle.score_topk(sub, nthreads=nthreads)
    dt = time.perf_counter() - t0
    pairs = visible_pairs(sub)
    return {"value": pairs * OPS_PER_PAIR / dt / 1e9, "unit": "GOPS", "cores": nthreads,
            "kind": "oracle", "seconds": dt,
            "sample": "%d of %d sequences of the workload (%d visible pairs); full oracle: exact "
                      "dots, fp32 scaling and head sum, stable sort" % (take, case.batch, pairs)}


def subcase(case, batches):
    """The workload restricted to some of its sequences (BSND decode workloads)."""
    b = np.asarray(batches, dtype=np.int64)
    rows = case.query[b]
    return W.Case(**{**case.__dict__, "batch": len(b), "query": rows, "weights": case.weights[b],
                     "q_scale": case.q_scale[b],
                     "seq_lens_q": None if case.seq_lens_q is None else case.seq_lens_q[b],
                     "seq_lens_k": case.seq_lens_k[b], "block_table": case.block_table[b]})


def run_reference(args, rank, world):
    if rank != 0:
        return
    case = make_workload(args.workload, args.batch, 0)
    import oracle
    oracle.build()
    nthreads = os.cpu_count() or 1
    # each step scores whole sequences of the workload, as many as keep every host core busy (the
    # oracle runs its rows on all of them) while K + W steps stay within a few minutes
    take = None
    if case.layout_q == "BSND":
        t0 = time.perf_counter()
        oracle.score_topk(subcase(case, list(range(min(case.batch, nthreads)))), nthreads=nthreads)
        per_seq = max(time.perf_counter() - t0, 1e-3) / min(case.batch, nthreads)
        budget = 120.0 / max(1, args.steps + args.warmup)          # seconds of oracle work per step
        take = int(max(min(case.batch, nthreads), min(case.batch, budget / per_seq)))
    sub = subcase(case, list(range(take))) if take else case
    pairs = visible_pairs(sub)
    for _ in range(args.warmup):
        oracle.score_topk(sub, nthreads=nthreads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.score_topk(sub, nthreads=nthreads)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = pairs * OPS_PER_PAIR * args.steps / total / 1e9
    sample = ("%d of %d sequences per step (%d visible pairs)" % (take, case.batch, pairs)
              if take else "whole workload")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic", "config": config_of(case, args, world),
            "cpu_baseline": {"value": value, "unit": "GOPS", "cores": nthreads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def config_of(case, args, world):
    return {"workload": "%s: B=%d, S1=%d, %s q/k, %s scales, S_k %d..%d, block_size %d, "
                        "sparse_count %d, sparse_mode %d, cmp_ratio %d" % (
                            case.name, case.batch, case.s1 or 0, case.qk_dtype, case.scale_dtype,
                            int(case.seq_lens_k.min()), int(case.seq_lens_k.max()),
                            case.block_size, case.sparse_count, case.sparse_mode, case.cmp_ratio),
            "global_batch": case.batch * world, "parallelism": "independent sequences per rank",
            "l2": "flushed between timed steps (%d MB write, then read back; outside the events)" % (
                args.flush_mb if args is not None else 512)}


def quantize_bytes(nvec, tokens, esz):
    """Algorithmic bytes of one quantizer step: every query vector read as bfloat16 (256 B) and
    written as codes (128 B) plus its scale; every key the same plus its (batch, position) pair
    and the block_table entry it reads."""
    return nvec * (256 + 128 + esz) + tokens * (256 + 128 + esz + 8 + 4)


def run_quantize(args, rank, world, local):
    """The upstream quantizer on the TND prefill workload (4 sequences of 1024..8192 tokens,
    T = 15360): one step quantizes the query (T x 64 vectors, qli_quantize) and writes every
    token's key into the paged cache (T keys, qli_quantize_keys)."""
    import torch
    import sparse_attention_token_block_gb300 as Q
    from sparse_attention_token_block_gb300 import build as B

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    case = W.varlen_prefill(seed=5 + 1000 * rank)
    p = Q.make_problem(**W.problem_kwargs(case))
    esz = 2 if case.scale_dtype == W.F16 else 4
    q_bits = W.bf16_vectors(case.query.shape, seed=31 + rank)
    k_bits = W.bf16_vectors((int(case.seq_lens_k.sum()), 128), seed=32 + rank, special=False)
    tok_b = np.repeat(np.arange(case.batch, dtype=np.int32), case.seq_lens_k)
    tok_p = np.concatenate([np.arange(n, dtype=np.int32) for n in case.seq_lens_k])
    d = W.to_device(case, dev)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    xq, xk = bf(q_bits), bf(k_bits)
    tb, tp = torch.from_numpy(tok_b).to(dev), torch.from_numpy(tok_p).to(dev)
    ws = torch.zeros(64, dtype=torch.int32, device=dev)
    Q.check(Q.workspace_init(ws), "workspace_init")
    flush = torch.empty(args.flush_mb * (1 << 20) // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        Q.check(Q.quantize(p.qk_dtype, p.scale_dtype, xq, d["query"], d["q_scale"]), "quantize")
        if ev:
            ev[1].record(stream)
        Q.check(Q.quantize_keys(p, xk, tb, tp, d["block_table"], d["key"], d["k_scale"], ws), "quantize_keys")
        if ev:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        torch.amax(flush, dim=0, out=sink)
        step()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    if not args.no_clocks:
        clocks.start()
    t_end = time.perf_counter() + (0 if args.no_clocks else 1.5)
    while time.perf_counter() < t_end:
        for _ in range(10):
            step()
        torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i)
        torch.amax(flush, dim=0, out=sink)
        step(evs[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    st, bits = Q.get_device_error(ws)
    Q.check(st, "device error (bits %d)" % bits)
    nvec, tokens = q_bits.size // 128, len(tok_b)
    q_ms = [e[0].elapsed_time(e[1]) for e in evs]
    k_ms = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms = max_over_ranks(sum(q_ms) + sum(k_ms), None, dev)
    nbytes = quantize_bytes(nvec, tokens, esz)
    value = nbytes * args.steps * world / (total_ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    q_avg = statistics.mean(q_ms)
    achieved = quantize_bytes(nvec, 0, esz) / (q_avg * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        take = 32768
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 5.0:
            oracle.quantize(q_bits.reshape(-1, 128)[:take], case.qk_dtype == W.FP8, esz == 4)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": quantize_bytes(take, 0, esz) * reps / dt / 1e9, "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": "%d query vectors, %d passes" % (take, reps)}
    line = {
        "metric": "quantizer GB/s (algorithmic bytes: bfloat16 in, codes and scales out)", "value": value,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 -> " + ("int8" if case.qk_dtype == W.INT8 else "fp8_e4m3"), "data": "synthetic",
        "config": {"workload": "query quantization and key-cache write of a TND prefill: T=%d tokens "
                               "(%s), 64 heads of 128, %s scales, key pages of %d" % (
                                   tokens, "+".join(str(int(x)) for x in case.seq_lens_k), case.scale_dtype,
                                   case.block_size),
                   "l2": "flushed between timed steps (%d MB write, then read back; outside the events)"
                         % args.flush_mb},
        "stage_us": {"quantize_query": 1e3 * q_avg, "quantize_keys": 1e3 * statistics.mean(k_ms)},
        "roofline": {"kernel": "quantize_vectors_kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": quantize_bytes(nvec, 0, esz),
                     "traffic": recorded_traffic(QUANT_PROFILE, QUANT_SOURCES)[0]},
        "clocks": clk,
        "gpu_launches": 2 * args.steps,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line))


def run_gather(args, rank, world, local):
    """The downstream sparse-attention gather on the long-context decode: the indexer's output
    (32 rows x 2048 indices, computed once) selects KV entries of ``--entry-bytes`` bytes from a
    paged KV cache that shares the key pool's block_table; one step is one qli_gather_kv."""
    import torch
    import sparse_attention_token_block_gb300 as Q
    from sparse_attention_token_block_gb300 import build as B

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    case = make_workload(args.workload, args.batch, rank)
    p = Q.make_problem(**W.problem_kwargs(case))
    ix = Q.Indexer(p, device=dev)
    d = W.to_device(case, dev)
    idx = ix.run(**d).clone()
    E = args.entry_bytes
    pool = torch.from_numpy(W.kv_pool(case, E, 0, seed=17 + rank)).to(dev)
    out = torch.empty((case.rows, case.sparse_count, E), dtype=torch.uint8, device=dev)
    counts = torch.empty(case.rows, dtype=torch.int32, device=dev)
    flush = torch.empty(args.flush_mb * (1 << 20) // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        Q.check(Q.gather_kv(p, d["seq_lens_q"], d["seq_lens_k"], d["block_table"], idx, pool, E, out, counts,
                            0, ix.workspace), "gather_kv")

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        torch.amax(flush, dim=0, out=sink)
        step()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    if not args.no_clocks:
        clocks.start()
    t_end = time.perf_counter() + (0 if args.no_clocks else 1.5)
    while time.perf_counter() < t_end:
        for _ in range(20):
            step()
        torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i)
        torch.amax(flush, dim=0, out=sink)
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    st, bits = ix.device_error()
    Q.check(st, "device error (bits %d)" % bits)
    valid = int((idx >= 0).sum().item())
    entries = case.rows * case.sparse_count
    nbytes = valid * E + entries * E + entries * 4 + case.rows * 4
    ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = sum(ms)
    avg = statistics.mean(ms)
    value = nbytes * args.steps * world / (total_ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        h_idx, h_pool = idx.cpu().numpy(), pool.cpu().numpy()
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 5.0:
            oracle.gather_kv(case, h_idx, h_pool, E)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": nbytes * reps / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "the whole gather, %d passes" % reps}
    line = {
        "metric": "sparse-attention gather GB/s (algorithmic bytes: selected entries read, all entries written)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bytes", "data": "synthetic",
        "config": {"workload": "gather after the %s indexer: %d rows x %d indices (%d valid), %d-byte KV entries "
                               "through a %d-entry-page block_table" % (case.name, case.rows, case.sparse_count,
                                                                       valid, E, case.block_size),
                   "l2": "flushed between timed steps (%d MB write, then read back; outside the events)"
                         % args.flush_mb},
        "us_per_call": 1e3 * avg,
        "roofline": {"kernel": "gather_kernel", "bound": "hbm", "achieved": nbytes / (avg * 1e-3) / 1e9,
                     "peak": peak, "unit": "GB/s", "frac": nbytes / (avg * 1e-3) / 1e9 / peak,
                     "peak_source": peak_kind, "algorithmic_bytes_per_launch": nbytes,
                     # the committed capture is of the default line (long decode, 512-byte entries)
                     "traffic": (recorded_traffic(GATHER_PROFILE, GATHER_SOURCES)[0]
                                 if (E, args.workload, args.batch) == (512, "long_decode", 0) else None)},
        "clocks": clk,
        "gpu_launches": args.steps,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line))


def score_roofline(stats, score_us, traffic=None):
    """Roofline of the scoring kernel for one workload: its algorithmic bytes per launch over the
    event-timed duration against the measured copy peak -- or, above the ridge point of the two
    measured peaks (algorithmic ops per byte), its algorithmic ops against the dense bf16 peak."""
    peak, peak_kind = peaks()
    tpeak, tpeak_kind = tensor_peak()
    ops_launch = stats["pairs"] * OPS_PER_PAIR
    if ops_launch / max(stats["score_bytes"], 1) > tpeak * 1e12 / (peak * 1e9):
        t_achieved = ops_launch / (score_us * 1e-6) / 1e12
        return {"kernel": "score_kernel", "bound": "tensor", "achieved": t_achieved, "peak": tpeak,
                "unit": "TFLOP/s", "frac": t_achieved / tpeak, "peak_source": tpeak_kind,
                "algorithmic_ops_per_launch": ops_launch, "traffic": traffic}
    achieved = stats["score_bytes"] / (score_us * 1e-6) / 1e9
    return {"kernel": "score_kernel", "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": peak_kind,
            "algorithmic_bytes_per_launch": stats["score_bytes"], "traffic": traffic}


def time_workload(Q, case, dev, flush_l2, steps, warmup, split_topk=0):
    """One workload's indexer call timed like the headline step (the execution plan replayed, L2
    flushed between calls, events on the launching stream), plus a pass with events between the
    three kernels for the per-stage times.  Returns the workload's summary for the JSON line.
    ``split_topk``: the problem's qli_split_topk (the two-stage top-k when ON)."""
    import torch
    stream = torch.cuda.current_stream(dev)
    stats = workload_stats(case)
    p = Q.make_problem(**W.problem_kwargs(case), split_topk=split_topk)
    ix = Q.Indexer(p, device=dev)
    d = W.to_device(case, dev)
    plan = ix.plan(**d)
    for _ in range(max(3, warmup)):
        flush_l2(1)
        plan.launch()
    torch.cuda.synchronize()
    Q.check(ix.device_error()[0], "device error (%s)" % case.name)
    pairs_ev = []
    for i in range(steps):
        flush_l2(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        plan.launch()
        b.record(stream)
        pairs_ev.append((a, b))
    sev = []
    for i in range(steps):
        flush_l2(i)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        Q.check(Q.metadata(p, d["seq_lens_q"], d["seq_lens_k"], ix.meta), "metadata")
        e[1].record(stream)
        Q.check(Q.score(p, d["query"], d["key"], d["weights"], d["q_scale"], d["k_scale"], d["seq_lens_q"],
                        d["seq_lens_k"], d["block_table"], ix.meta, ix.workspace), "score")
        e[2].record(stream)
        Q.check(Q.topk(p, d["block_table"], ix.meta, ix.workspace, ix.out), "topk")
        e[3].record(stream)
        sev.append(e)
    torch.cuda.synchronize()
    Q.check(ix.device_error()[0], "device error (%s)" % case.name)
    plan.close()
    us = statistics.mean(a.elapsed_time(b) for a, b in pairs_ev) * 1e3
    stage = {"metadata": 1e3 * statistics.mean(e[0].elapsed_time(e[1]) for e in sev),
             "score": 1e3 * statistics.mean(e[1].elapsed_time(e[2]) for e in sev),
             "topk": 1e3 * statistics.mean(e[2].elapsed_time(e[3]) for e in sev)}
    peak, _ = peaks()
    return {"config": config_of(case, None, 1)["workload"] + (", two-stage top-k" if split_topk else ""),
            "steps": steps,
            "us_per_call": us, "gops": stats["pairs"] * OPS_PER_PAIR / (us * 1e-6) / 1e9,
            "keys_scored_per_s": stats["pairs"] / (us * 1e-6), "stage_us": stage,
            "call_hbm_frac": stats["total_bytes"] / (us * 1e-6) / 1e9 / peak,
            "roofline": score_roofline(stats, stage["score"])}


def run_mma(args, rank, world, local):
    """Rate of tcgen05.mma kind::f16 (K 16, fp32 accumulators in tensor memory): M 128 with A from
    tensor memory -- the score kernel's form -- or from shared memory, M 64 with A from shared
    memory; N 64 .. 256; MMAs issued back to back by one warp per CTA into one accumulator or
    cycled over several independent ones; one or two CTAs per SM.  Prints one JSON line."""
    import ctypes
    import torch
    from sparse_attention_token_block_gb300 import build as B
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    L = ctypes.CDLL(B.PEAK_LIB)
    L.qli_peak_mma_f16.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p] * 4
    L.qli_peak_mma_f16.restype = ctypes.c_int
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(2 * sms, dtype=torch.int64, device=dev)
    ns = torch.zeros(2 * sms, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    tpeak, tkind = tensor_peak()
    iters = 8192
    # (A from tensor memory, M, N, accumulators, CTAs per SM)
    shapes = [(1, 128, n, 1, 1) for n in (64, 128, 192, 256)] + [(0, 128, n, 1, 1) for n in (64, 128, 192, 256)]
    shapes += [(1, 128, 64, c, 1) for c in (2, 4, 6)] + [(1, 128, 128, c, 1) for c in (2, 3)]
    shapes += [(1, 128, 64, c, 2) for c in (1, 2)] + [(0, 128, 64, 4, 1)]
    shapes += [(0, 64, n, c, 1) for n in (64, 128) for c in (1, 2)] + [(0, 64, 256, 1, 1)]
    out = []
    for a_tmem, m, n, chains, per_sm in shapes:
        ctas = per_sm * sms
        best = None
        for _ in range(max(3, args.warmup)):
            assert L.qli_peak_mma_f16(a_tmem, m, n, chains, per_sm, iters, ctas, cyc.data_ptr(), ns.data_ptr(),
                                      err.data_ptr(), stream) == 0
            torch.cuda.synchronize()
            assert int(err.item()) == 0, "a bounded wait gave up"
            c = cyc[:ctas].cpu().numpy().astype(np.float64)
            t = ns[:ctas].cpu().numpy().astype(np.float64)
            flop = 2.0 * m * n * 16 * iters
            tf = ctas * flop / (t.max() * 1e-9) / 1e12
            if best is None or tf > best["tflops"]:
                best = {"a_operand": "tensor memory" if a_tmem else "shared memory", "m": m, "n": n,
                        "accumulators": chains, "ctas_per_sm": per_sm,
                        "tflops": tf, "frac_of_bf16_peak": tf / tpeak,
                        "cycles_per_mma_per_sm": float(np.median(c)) / (iters * per_sm),
                        "sm_mhz_implied": float(np.median(c / t * 1e3))}
        out.append(best)
    if rank == 0:
        print(json.dumps({"metric": "tcgen05.mma kind::f16 rate, K 16", "unit": "TFLOP/s",
                          "bf16_peak": tpeak, "bf16_peak_source": tkind, "sms": sms, "iters_per_cta": iters,
                          "results": out}))


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.op == "quantize":
        run_quantize(args, rank, world, local)
        return
    if args.op == "gather":
        run_gather(args, rank, world, local)
        return
    if args.op == "mma":
        run_mma(args, rank, world, local)
        return
    import torch
    import sparse_attention_token_block_gb300 as Q
    from sparse_attention_token_block_gb300 import build as B

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    case = make_workload(args.workload, args.batch, rank)
    stats = workload_stats(case)
    p = Q.make_problem(**W.problem_kwargs(case))
    ix = Q.Indexer(p, device=dev)
    d = W.to_device(case, dev)
    flush = torch.empty(args.flush_mb * (1 << 20) // 4, dtype=torch.int32, device=dev)
    flush_sink = torch.empty((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(v):
        # write a buffer larger than L2 (evicts every input), then read it back so that the
        # write-back of those dirty lines also happens before the next timed region
        flush.fill_(v)
        torch.amax(flush, dim=0, out=flush_sink)      # a reduction: reads, no large temporary

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        Q.check(Q.metadata(p, d["seq_lens_q"], d["seq_lens_k"], ix.meta), "metadata")
        if evs:
            evs[1].record(stream)
        Q.check(Q.score(p, d["query"], d["key"], d["weights"], d["q_scale"], d["k_scale"],
                        d["seq_lens_q"], d["seq_lens_k"], d["block_table"], ix.meta,
                        ix.workspace), "score")
        if evs:
            evs[2].record(stream)
        Q.check(Q.topk(p, d["block_table"], ix.meta, ix.workspace, ix.out), "topk")
        if evs:
            evs[3].record(stream)

    for _ in range(max(3, args.warmup)):
        flush_l2(1)
        step()
    torch.cuda.synchronize()
    st, bits = ix.device_error()
    Q.check(st, "device error after warm-up (bits %d)" % bits)
    # the timed step is the public execution plan (qli_plan_*): the same three launches captured
    # once as a CUDA graph and replayed, as a serving loop with fixed buffers runs them
    plan = None if args.no_graph else ix.plan(**d)
    run_step = step if plan is None else plan.launch
    if plan is not None:
        for _ in range(max(3, args.warmup)):
            flush_l2(1)
            run_step()
        torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    # nvidia-smi samples every 100 ms: keep the GPU on the same load for ~1.5 s of untimed steps
    # right before the timed ones so the samples describe the clocks the timed steps ran at
    clocks = Clocks(local)
    if not args.no_clocks:
        clocks.start()
    t_end = time.perf_counter() + (0 if args.no_clocks else 1.5)
    while time.perf_counter() < t_end:
        for _ in range(20):
            flush_l2(2)
            run_step()
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    # the timed steps: events only at step boundaries, so the three kernels may overlap their
    # launches (programmatic dependent launch) as they do in use
    for i in range(args.steps):
        flush_l2(i)
        evs[i][0].record(stream)
        run_step()
        evs[i][3].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    # the same steps launched one kernel at a time on the stream (no graph), for comparison
    sstream = []
    for i in range(max(3, min(args.steps, 50))):
        flush_l2(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        sstream.append((a, b))
    torch.cuda.synchronize()
    stream_us = sum(a.elapsed_time(b) for a, b in sstream) / len(sstream) * 1e3
    # a call that reuses the metadata (every call sharing the lengths, e.g. the other layers of a
    # step, needs it once): score + top-k only, as a plan without the metadata launch
    reuse_us = None
    if plan is not None:
        plan_nm = ix.plan(**d, with_metadata=False)
        rev = []
        for i in range(max(3, min(args.steps, 50))):
            flush_l2(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            plan_nm.launch()
            b.record(stream)
            rev.append((a, b))
        torch.cuda.synchronize()
        reuse_us = sum(a.elapsed_time(b) for a, b in rev) / len(rev) * 1e3
        plan_nm.close()
    # the same step also writing sparse_values (the README's return_value): a second indexer whose
    # problem asks for the values, replayed as a plan like the timed step
    values_us = None
    if plan is not None:
        pv = Q.make_problem(**W.problem_kwargs(case), return_value=1)
        ixv = Q.Indexer(pv, device=dev)
        planv = ixv.plan(**d)
        vev = []
        for i in range(max(3, min(args.steps, 50)) + 3):
            flush_l2(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            planv.launch()
            b.record(stream)
            vev.append((a, b))
        torch.cuda.synchronize()
        Q.check(ixv.device_error()[0], "device error with sparse_values")
        vev = vev[3:]
        values_us = sum(a.elapsed_time(b) for a, b in vev) / len(vev) * 1e3
        planv.close()
    # hot L2: the same plan replayed back to back without the flush (inputs partly L2-resident)
    hot_us = None
    if plan is not None:
        nhot = max(3, min(args.steps, 50))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(nhot):
            plan.launch()
        b.record(stream)
        torch.cuda.synchronize()
        hot_us = a.elapsed_time(b) / nhot * 1e3
    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    # per-stage pass (stage times and the score kernel's roofline): events between the kernels
    stage_steps = max(3, min(args.steps, 50))
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(stage_steps)]
    for i in range(stage_steps):
        flush_l2(i)
        step(sev[i])
    torch.cuda.synchronize()
    meta_ms = [e[0].elapsed_time(e[1]) for e in sev]
    score_ms = [e[1].elapsed_time(e[2]) for e in sev]
    topk_ms = [e[2].elapsed_time(e[3]) for e in sev]
    ops = stats["pairs"] * OPS_PER_PAIR * args.steps * world
    value = whole_job_gops(stats["pairs"], args.steps, world, total_ms)

    # end to end through the public call with host buffers: pinned host inputs copied in, the
    # indices copied out, every step
    e2e = None
    if not args.no_e2e:
        host = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in d.items()}
        out_h = torch.empty(ix.out.shape, dtype=torch.int32).pin_memory()
        dd = {k: (torch.empty_like(v) if v is not None else None) for k, v in d.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = out_h.numel() * 4

        e2e_plan = None if args.no_graph else ix.plan(**dd)

        def e2e_step():
            for k, v in host.items():
                if v is not None:
                    dd[k].copy_(v, non_blocking=True)
            if e2e_plan is None:
                out = ix.run(**dd)
            else:
                e2e_plan.launch()
                out = ix.out
            out_h.copy_(out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2(i)
            ev[i][0].record(stream)
            e2e_step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), dist, dev)
        e2e = {"value": ops / (e_ms * 1e-3) / 1e9, "unit": "GOPS", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / args.steps}

    st, bits = ix.device_error()
    Q.check(st, "device error after timing (bits %d)" % bits)
    if rank != 0:
        return
    peak, peak_kind = peaks()
    score_avg = sum(score_ms) / len(score_ms)
    # the committed score-kernel capture is of the long decode at its default size
    traffic = recorded_traffic()[0] if (args.workload, args.batch) == ("long_decode", 0) else None
    roofline = score_roofline(stats, score_avg * 1e3, traffic)
    # the other configurations, each timed the same way (fewer steps), for their own figures
    others = None
    if not args.no_workloads:
        others = {}
        for name in W.WORKLOADS:
            if name == args.workload:
                continue
            others[name] = time_workload(Q, make_workload(name, 0, rank), dev, flush_l2,
                                         max(3, min(args.steps, 30)), args.warmup)
        if args.workload == "long_decode":
            # the same call with the top-k in two stages (split-local selection in the score
            # kernel, then the merge): opt-in, measured beside the default
            others["long_decode_split_topk"] = time_workload(Q, case, dev, flush_l2, max(3, min(args.steps, 30)),
                                                             args.warmup, split_topk=Q.SPLIT_ON)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case)
    line = {
        "metric": METRIC, "value": value, "unit": "GOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8" if case.qk_dtype == W.INT8 else "fp8_e4m3",
        "data": "synthetic", "config": config_of(case, args, world),
        "keys_scored_per_s": stats["pairs"] * args.steps * world / (total_ms * 1e-3),
        "us_per_call": 1e3 * total_ms / args.steps,
        "launch": "stream launches" if args.no_graph else "execution plan (CUDA graph replay, qli_plan_launch)",
        "us_per_call_stream_launches": stream_us,
        "us_per_call_metadata_reused": reuse_us,
        "us_per_call_hot_l2": hot_us,
        "us_per_call_with_sparse_values": values_us,
        "stage_us": {"metadata": 1e3 * statistics.mean(meta_ms),
                     "score": 1e3 * score_avg, "topk": 1e3 * statistics.mean(topk_ms)},
        # the whole call's algorithmic bytes (scoring inputs, indices, lengths) over us_per_call
        "call_hbm_frac": stats["total_bytes"] / (total_ms / args.steps * 1e-3) / 1e9 / peak,
        "roofline": roofline,
        "workloads": others,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
