"""Planted mistakes in the oracle must fail its pins.

Each case copies the oracle and its pin tests into a scratch directory,
plants one plausible mistake in the copy's source (a dropped term, a
transposed operand, a missing absolute value, a wrong index, a wrong exponent
bias, the wrong expert's weights, ties rounded away from even, a swapped
gate/up pair, a dropped SiLU factor, a wrong exponent sign, a wrong column
offset) and runs the pins on the copy in a child process: the run must fail.
The unchanged copy must pass, so a failure is the mistake's doing."""
import concurrent.futures
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C_SRC = "oracle/gemm_oracle.c"

# (name, file, [(old, new), ...]); every old text must occur in the file.
MUTATIONS = [
    ("dropped last k term", C_SRC, [("                d[j] += p;", "                d[j] += (k == K - 1) ? 0.0 : p;")]),
    ("transposed A", C_SRC, [("double a = decode(A[(long)i * lda + k], dtype);",
                              "double a = decode(A[(long)k * lda + i], dtype);")]),
    ("S without absolute value", C_SRC, [("                s[j] += fabs(p);", "                s[j] += p;")]),
    ("element index swapped", C_SRC, [("decode(B[(long)k * ldb + J[t]], dtype)",
                                       "decode(B[(long)k * ldb + I[t]], dtype)")]),
    ("fp16 exponent bias", C_SRC, [("exp - 25);", "exp - 24);")]),
    ("wrong expert weights", C_SRC, [("oracle_gemm_rows(A, Bs[g], dtype,", "oracle_gemm_rows(A, Bs[G - 1 - g], dtype,")]),
    ("ties away from zero", C_SRC, [("w += 0x7fffu + lsb;", "w += 0x8000u;")]),
    ("gate and up swapped", C_SRC, [("double g = gate[j];", "double g = up[j];"),
                                    ("h[j] = silu * up[j];", "h[j] = silu * gate[j];")]),
    ("sigmoid instead of silu", C_SRC, [("double silu = g / (1.0 + exp(-g));",
                                         "double silu = 1.0 / (1.0 + exp(-g));")]),
    ("exponent sign", C_SRC, [("double silu = g / (1.0 + exp(-g));", "double silu = g / (1.0 + exp(g));")]),
    ("up column offset", C_SRC, [("const double *up = gate + I;", "const double *up = gate + I - 1;")]),
    ("gate row stride", C_SRC, [("const double *gate = D + r * 2L * I;", "const double *gate = D + r * (long)I;")]),
]

COPY = ["oracle/__init__.py", C_SRC, "tests/conftest.py", "tests/test_oracle.py",
        "tests/test_oracle_swiglu.py", "blackwell_tensor_core_gb300/__init__.py",
        "blackwell_tensor_core_gb300/workloads.py"]


def _run_pins(workdir, edits):
    for rel in COPY:
        dst = os.path.join(workdir, rel)
        os.makedirs(os.path.dirname(dst), exist_ok=True)
        shutil.copyfile(os.path.join(ROOT, rel), dst)
    for rel, old, new in edits:
        path = os.path.join(workdir, rel)
        text = open(path).read()
        assert old in text, "mutation text not found in %s: %r" % (rel, old)
        open(path, "w").write(text.replace(old, new))
    env = dict(os.environ, OMP_NUM_THREADS="2", PYTHONDONTWRITEBYTECODE="1")
    env.pop("PYTHONPATH", None)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle.py", "tests/test_oracle_swiglu.py"],
                       cwd=workdir, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def test_planted_mistakes_fail_the_pins(tmp_path):
    jobs = [("unchanged", [])] + [(name, [(f, o, n) for o, n in subs]) for name, f, subs in MUTATIONS]
    with concurrent.futures.ThreadPoolExecutor(max_workers=4) as ex:
        futs = {name: ex.submit(_run_pins, str(tmp_path / ("m%02d" % i)), edits)
                for i, (name, edits) in enumerate(jobs)}
        results = {name: f.result() for name, f in futs.items()}
    rc, out = results.pop("unchanged")
    assert rc == 0, "the unchanged copy must pass its pins:\n" + out
    survivors = [name for name, (rc, _) in results.items() if rc == 0]
    assert not survivors, "planted mistakes not caught by any pin: %s" % survivors
