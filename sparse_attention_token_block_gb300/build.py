"""Build ``libqli.so`` (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel, then one link step makes the shared library next to
this file.  Re-running only rebuilds what changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libqli.so")
# the testing build: the same objects except the host API, compiled with QLI_TESTING (it adds the
# failure-detection test switch of include/qli_testing.h); the product library has no switch
TEST_LIB = os.path.join(HERE, "libqli_testing.so")
PEAK_LIB = os.path.join(HERE, "libqli_peak.so")
SOURCES = ["qli_api.cu", "qli_metadata.cu", "qli_score.cu", "qli_score_multi.cu", "qli_score_pair.cu", "qli_score_split.cu", "qli_topk.cu", "qli_topk_small.cu", "qli_topk_cluster.cu", "qli_noalloc.cu", "qli_plan.cu", "qli_quant.cu", "qli_gather.cu"]
HEADERS = ["qli_internal.cuh", "qli_ptx.cuh", "qli_score.cuh", "qli_topk.cuh"]
TEST_SOURCE = "qli_api.cu"
# the tensor-core rate micro-benchmark (include/qli_peak.h), a library of its own
PEAK_SOURCE = "qli_peak.cu"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc()))), "lib64")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                   "-I", os.path.join(ROOT, "include")] + list(extra)


def _newer(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(OBJ, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "qli.h")]
    hdrs.append(os.path.join(ROOT, "include", "qli_testing.h"))
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJ, src.replace(".cu", ".o"))
        if ptxas_info or _newer(o, [s] + hdrs):
            extra = ["-Xptxas", "-v"] if ptxas_info else []
            jobs.append((src, [nvcc(), "-c", s, "-o", o] + _flags(extra)))
    s = os.path.join(CSRC, PEAK_SOURCE)
    o_peak = os.path.join(OBJ, "qli_peak.o")
    if ptxas_info or _newer(o_peak, [s] + hdrs + [os.path.join(ROOT, "include", "qli_peak.h")]):
        jobs.append((PEAK_SOURCE, [nvcc(), "-c", s, "-o", o_peak] + _flags(["-Xptxas", "-v"] if ptxas_info else [])))
    s = os.path.join(CSRC, TEST_SOURCE)
    o_test = os.path.join(OBJ, TEST_SOURCE.replace(".cu", "_testing.o"))
    if _newer(o_test, [s] + hdrs):
        jobs.append((TEST_SOURCE + " (testing)", [nvcc(), "-c", s, "-o", o_test] + _flags(["-DQLI_TESTING"])))

    def run(job):
        name, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return name, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for name, r in ex.map(run, jobs):
                if verbose or ptxas_info or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError("nvcc failed on %s" % name)
    objs = [os.path.join(OBJ, s.replace(".cu", ".o")) for s in SOURCES]
    test_objs = [o_test if s == TEST_SOURCE else o for s, o in zip(SOURCES, objs)]
    peak_objs = [os.path.join(OBJ, "qli_peak.o")]
    for lib, parts in ((LIB, objs), (TEST_LIB, test_objs), (PEAK_LIB, peak_objs)):
        if _newer(lib, parts):
            tmp = lib + ".tmp%d" % os.getpid()
            cmd = [nvcc(), "-shared", "-o", tmp] + parts + ARCH + [
                "-cudart", "shared", "-Xlinker", "-rpath=" + cuda_lib_dir()]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
                raise RuntimeError("link of %s failed" % os.path.basename(lib))
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    build(verbose=True, ptxas_info="-v" in sys.argv)
    print(LIB)
