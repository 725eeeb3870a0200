"""Planted mistakes in the oracle (CPU only).

Each case copies oracle/dsa_oracle.c, plants one plausible mistake in the
copy (a dropped term, a wrong sign, an operand or index mixed up, an order
reversed), builds it with gcc and runs the oracle's pins against it in a
child process (DSA_ORACLE_LIB points the oracle's loader at the copy).  The
pins must fail for every mistake, and pass for an unchanged copy built the
same way.  The mistakes are planted in the oracle, on the CPU; nothing here
touches the CUDA library.  Every mutation stays inside the buffers it reads,
so no copy can crash the child.
"""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "dsa_oracle.c")
PINS = ["tests/test_oracle.py", "tests/test_oracle_topk.py", "tests/test_oracle_oproj.py"]

MUTANTS = [
    ("scale dropped from the scores", "s[j] = sc * dot;", "s[j] = dot;"),
    ("sink left out of the denominator", "double L = exp(sk - m);", "double L = 0.0;"),
    ("exponent sign flipped", "const double w = exp(s[j] - m);", "const double w = exp(m - s[j]);"),
    ("value taken from q (operands mixed up)", "out[c] += w * load(kv, dtype, xoff + c);",
     "out[c] += w * load(q, dtype, qoff + c);"),
    ("neighbouring column in the score", "load(kv, dtype, xoff + d);", "load(kv, dtype, xoff + (d ^ 1));"),
    ("last selected key dropped", "const int K = n_sel[r];", "const int K = n_sel[r] > 0 ? n_sel[r] - 1 : 0;"),
    ("every decode row reads slot 0", "(size_t)(r / decode)", "(size_t)0"),
    ("output not normalised", "for (c = 0; c < DSA_D; ++c) out[c] /= L;", "(void)L;"),
    ("top-k: equal scores by larger position", "return (x->pos > y->pos) - (x->pos < y->pos);",
     "return (x->pos < y->pos) - (x->pos > y->pos);"),
    ("top-k: NaN before numbers", "if (xn != yn) return xn - yn;", "if (xn != yn) return yn - xn;"),
    ("top-k: picks listed by score, not position",
     "if (m > 1) qsort(out, (size_t)m, sizeof(int32_t), pos_cmp);", ""),
    ("top-k: one pick short", "const int m = ok ? (n < k ? n : k) : 0;",
     "const int m = ok ? (n < k ? n : k - 1) : 0;"),
    ("projection: weights transposed", "const double wv = widen_bf16(wk[n]);",
     "const double wv = widen_bf16(w[(size_t)n * (size_t)K + (size_t)k]);"),
    ("projection: signed products in the absolute sum", "if (ao) ao[n] += fabs(a) * fabs(wv);",
     "if (ao) ao[n] += a * wv;"),
]


def _build(tmp_path, name, text):
    src = tmp_path / (name + ".c")
    lib = tmp_path / (name + ".so")
    src.write_text(text)
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", "-I", os.path.dirname(SRC),
           str(src), "-o", str(lib), "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return str(lib)


def _pins(lib):
    env = dict(os.environ, DSA_ORACLE_LIB=lib, OMP_NUM_THREADS="4")
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_an_unchanged_copy_passes_the_pins(tmp_path):
    r = _pins(_build(tmp_path, "unchanged", open(SRC).read()))
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("what,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_a_planted_mistake_fails_a_pin(tmp_path, what, find, repl):
    text = open(SRC).read()
    assert text.count(find) == 1, "the mutation site must be unique: %r" % find
    r = _pins(_build(tmp_path, "mutant", text.replace(find, repl)))
    assert r.returncode != 0, "no pin caught: %s" % what
    assert "failed" in r.stdout or "error" in r.stdout.lower(), r.stdout[-2000:]
