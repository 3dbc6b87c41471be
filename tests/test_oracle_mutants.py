"""The pins must catch plausible mistakes: each case plants one mistake in a copy of the oracle's
C source, builds it, and runs the pin suite of that part (tests/test_oracle.py for the indexer,
test_oracle_quant.py for the quantizer, test_oracle_gather.py for the gather) against it in a
subprocess; the suite has to fail."""
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qli_oracle.c")

MUTANTS = [
    ("drop_relu", "v = v > 0.0f ? v : 0.0f;    /* ReLU */", "v = v;"),
    ("scale_q_twice", "float a = sQ * sK;          /* ScaleQ @ ScaleK^T */", "float a = sQ * sQ;"),
    ("key_slot_shift", "int64_t slot = j % p->block_size;", "int64_t slot = (j + 1) % p->block_size;"),
    ("causal_floor", "n = (pos + 1 + p->cmp_ratio - 1) / p->cmp_ratio;", "n = (pos + 1) / p->cmp_ratio;"),
    ("ties_descending", "return (x->idx > y->idx) - (x->idx < y->idx);",
     "return (x->idx < y->idx) - (x->idx > y->idx);"),
    ("drop_weight", "float t = w * v;            /* (W @ 1) (.) ReLU(...) */", "float t = v;"),
    ("head_swap", "int64_t qoff = (row * p->num_heads + h) * (int64_t)p->head_dim;",
     "int64_t qoff = (row * p->num_heads + (h ^ 1)) * (int64_t)p->head_dim;"),
    ("e4m3_bias", "v = ldexp(8.0 + m, e - 10);", "v = ldexp(8.0 + m, e - 9);"),
    ("sort_ascending", "if (x->score > y->score) return -1;", "if (x->score > y->score) return 1;"),
    ("tnd_rows", "int32_t lo = b > 0 ? seq_lens_q[b - 1] : 0;", "int32_t lo = b > 1 ? seq_lens_q[b - 2] : 0;"),
    ("key_stride_ignored", "int64_t koff = page * page_stride + slot",
     "int64_t koff = page * (int64_t)p->block_size * p->head_dim + slot"),
    ("complete_blocks_ceil", "        n = (pos + 1) / p->cmp_ratio;\n", "        n = (pos + 1 + p->cmp_ratio - 1) / p->cmp_ratio;\n"),
]


E4M3_TIES = ("    double dl = v - qlio_e4m3_value(lo), dh = qlio_e4m3_value(hi) - v;\n"
             "    if (dl < dh) return lo;\n    if (dh < dl) return hi;\n    return (lo & 1) ? hi : lo;")

# (name, anchor, replacement, pin file)
MUTANTS_MORE = [
    ("quant_qmax_128", "const float qmax = qk_fp8 ? 448.0f : 127.0f;", "const float qmax = qk_fp8 ? 448.0f : 128.0f;",
     "test_oracle_quant.py"),
    ("quant_truncate", "float r = rintf(y);", "float r = truncf(y);", "test_oracle_quant.py"),
    ("quant_round_half_away", "float r = rintf(y);", "float r = roundf(y);", "test_oracle_quant.py"),
    ("quant_signed_max", "amax = fmaxf(amax, fabsf(x[d]));", "amax = fmaxf(amax, x[d]);", "test_oracle_quant.py"),
    ("quant_e4m3_ties_up", E4M3_TIES, E4M3_TIES.replace("return (lo & 1) ? hi : lo;", "return hi;"),
     "test_oracle_quant.py"),
    ("quant_e4m3_sign", "(signbit(y) ? 0x80 : 0)", "(y < 0.0f ? 0x80 : 0)", "test_oracle_quant.py"),
    ("quant_key_slot", "slot = pos % bs;", "slot = (pos + 1) % bs;", "test_oracle_quant.py"),
    ("quant_key_stride", "(uint8_t*)key_pool + page * stride + slot * 128",
     "(uint8_t*)key_pool + page * bs * 128 + slot * 128", "test_oracle_quant.py"),
    ("gather_slot", "page * stride + (j % bs) * entry_bytes", "page * stride + ((j + 1) % bs) * entry_bytes",
     "test_oracle_gather.py"),
    ("gather_no_zero_fill", "memset(dst, 0, (size_t)entry_bytes);", "(void)dst;", "test_oracle_gather.py"),
    ("gather_limit_inclusive", "if (j < 0 || j >= limit) {", "if (j < 0 || j > limit) {", "test_oracle_gather.py"),
    ("gather_row_batch", "        if (r < hi)\n", "        if (r <= hi)\n", "test_oracle_gather.py"),
    ("gather_counts_all", "counts[r] = copied;", "counts[r] = (int32_t)k;", "test_oracle_gather.py"),
]


@pytest.mark.parametrize("name,old,new,pins", MUTANTS_MORE, ids=[m[0] for m in MUTANTS_MORE])
def test_quantizer_and_gather_pins_catch_planted_mistake(name, old, new, pins, tmp_path):
    _run_mutant(name, old, new, pins, tmp_path)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    _run_mutant(name, old, new, "test_oracle.py", tmp_path)


def _run_mutant(name, old, new, pins, tmp_path):
    src = open(SRC).read()
    assert old in src, "mutation anchor missing: " + name
    mutant_c = tmp_path / ("mutant_%s.c" % name)
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / ("libmutant_%s.so" % name)
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC",
                           "-pthread", "-o", str(lib), str(mutant_c), "-lm"])
    env = dict(os.environ, QLI_ORACLE_LIB=str(lib))
    out = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", pins)],
                         env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode != 0, "planted mistake %s was not caught:\n%s" % (name, out.stdout[-1500:])
