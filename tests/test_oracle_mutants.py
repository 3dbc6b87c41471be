"""The pins must catch plausible mistakes: each case plants one mistake in a copy of the oracle's
C source, builds it, and runs the pin suite (tests/test_oracle.py) against it in a subprocess;
the suite has to fail."""
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
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = open(SRC).read()
    assert old in src, "mutation anchor missing: " + name
    mutant_c = tmp_path / ("mutant_%s.c" % name)
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / ("libmutant_%s.so" % name)
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC",
                           "-pthread", "-o", str(lib), str(mutant_c), "-lm"])
    env = dict(os.environ, QLI_ORACLE_LIB=str(lib))
    out = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle.py")],
                         env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode != 0, "planted mistake %s was not caught:\n%s" % (name, out.stdout[-1500:])
