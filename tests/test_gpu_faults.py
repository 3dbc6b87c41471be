"""Failure detection on the GPU without a fault: every wait in the score kernel is bounded, so a
producer that issues nothing, or converters that consume nothing (the stall switch of the testing
build of the library, include/qli_testing.h), make the waits run out; the kernel must report
QLI_ERR_DEVICE_TIMEOUT through the workspace's error word, let the copies already in flight land
before its CTAs exit, and leave the CUDA context usable.  The product library has no such switch."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, %r)
import torch
import numpy as np
import workloads as W
import sparse_attention_token_block_gb300 as Q
Q.use_testing_library()
Q.lib.qli_testing_set_stall(%d)
case = W.make_case("stall", batch=2, s1=1, seq_lens_k=[700, 300], block_size=64, sparse_count=16, seed=1)
p = Q.make_problem(**W.problem_kwargs(case))
ix = Q.Indexer(p)
ix.run(**W.to_device(case))
st, bits = ix.device_error()
print("STATUS", st, bits)
x = torch.ones(1024, device="cuda").sum().item()     # the context still works
print("AFTER", x)
"""


def run_child(stall):
    out = subprocess.run([sys.executable, "-c", CHILD % (ROOT, stall)], capture_output=True,
                         text=True, timeout=120)
    return out


@pytest.fixture(scope="module")
def built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_token_block_gb300 import build as B
    B.build()


def test_stalled_producer_reports_timeout(built):
    out = run_child(1)
    assert out.returncode == 0, out.stderr[-2000:]
    status = [l for l in out.stdout.splitlines() if l.startswith("STATUS")][0].split()
    assert int(status[1]) == 6            # QLI_ERR_DEVICE_TIMEOUT
    assert int(status[2]) & 4             # timeout bit
    assert "AFTER 1024.0" in out.stdout


def test_stalled_converter_reports_timeout_after_copies_land(built):
    out = run_child(2)
    assert out.returncode == 0, out.stderr[-2000:]
    status = [l for l in out.stdout.splitlines() if l.startswith("STATUS")][0].split()
    assert int(status[1]) == 6            # QLI_ERR_DEVICE_TIMEOUT
    assert int(status[2]) & 4
    assert "AFTER 1024.0" in out.stdout


def test_normal_run_reports_no_error(built):
    out = run_child(0)
    assert out.returncode == 0, out.stderr[-2000:]
    status = [l for l in out.stdout.splitlines() if l.startswith("STATUS")][0].split()
    assert int(status[1]) == 0 and int(status[2]) == 0
