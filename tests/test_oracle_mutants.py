"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
the pins catch every one of them, while the unmodified source passes."""
import os
import subprocess
import sys

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_ref.c")

# (name, original text, planted mistake): each original occurs exactly once.
MUTANTS = [
    ("sigmoid sign", "return gmin / (1.0 + exp(-x));", "return gmin / (1.0 + exp(x));"),
    ("A instead of exp(A)", "const double x = exp(A_h) * z;", "const double x = A_h * z;"),
    ("gmin dropped", "return gmin / (1.0 + exp(-x));", "return -1.0 / (1.0 + exp(-x));"),
    ("erase sign", "b * k[i] * (v[j] - p[j])", "b * k[i] * (v[j] + p[j])"),
    ("beta dropped from write", "b * k[i] * (v[j] - p[j])", "k[i] * (v[j] - p[j])"),
    ("decay dropped", "S[(size_t)i * dv + j] *= a;", "(void)a;"),
    ("decay exponent sign", "const double a = exp(gate(gmin, A_h, z[i]));",
     "const double a = exp(-gate(gmin, A_h, z[i]));"),
    ("erase read with query", "p[j] += S[(size_t)i * dv + j] * k[i];",
     "p[j] += S[(size_t)i * dv + j] * q[i];"),
    ("erase read transposed", "p[j] += S[(size_t)i * dv + j] * k[i];",
     "p[j] += S[(size_t)j * dv + i] * k[i];"),
    ("output read with key", "o[j] += S[(size_t)i * dv + j] * q[i];",
     "o[j] += S[(size_t)i * dv + j] * k[i];"),
    ("write uses query", "b * k[i] * (v[j] - p[j])", "b * q[i] * (v[j] - p[j])"),
    ("initial state ignored", "if (S0) memcpy", "if (0) memcpy"),
    ("snapshot one token late", "n_done % chunk == 0", "n_done % chunk == 1"),
    ("gate of next channel", "z + xk,", "z + xk + (dk > 1),"),
]


_RUNNER = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
orc = oracle.Oracle({lib!r})
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(orc)
    except Exception:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
"""


def _failures(tmp_path, name, old, new):
    """Names of the pins that fail on the variant.  The pins run in a child
    process, since a planted indexing mistake may crash it; a crash counts as
    caught."""
    text = open(SRC).read()
    if old is not None:
        assert text.count(old) == 1, f"mutation anchor {old!r} must occur once"
        text = text.replace(old, new)
    src = tmp_path / "kda_ref_variant.c"
    src.write_text(text)
    lib = str(tmp_path / "libkda_ref_variant.so")
    oracle.build(force=True, src=str(src), out=lib)
    tests = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(tests), tests=tests, lib=lib)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         env=dict(os.environ, OMP_NUM_THREADS="2"), timeout=600)
    if res.returncode != 0:
        return ["<crashed>"]
    line = [l for l in res.stdout.splitlines() if l.startswith("FAILED:")][-1]
    return [x for x in line[len("FAILED:"):].split(",") if x]


def test_unmodified_copy_passes(tmp_path):
    assert _failures(tmp_path, "none", None, None) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    failed = _failures(tmp_path, name, old, new)
    assert failed, f"no pin catches the planted mistake '{name}'"


# Planted mistakes in the oracle's input pre-ops (a Python module: the variant
# is imported from a copy and the pre-op pins run against it in-process).
PRE_SRC = os.path.join(os.path.dirname(oracle.__file__), "preops.py")
PRE_MUTANTS = [
    ("norm without square root", "norm = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))",
     "norm = np.sum(x * x, axis=-1, keepdims=True)"),
    ("norm over the token axis", "np.sum(x * x, axis=-1, keepdims=True)",
     "np.sum(x * x, axis=0, keepdims=True)"),
    ("sigmoid branches swapped", "np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))",
     "np.where(x >= 0, e / (1.0 + e), 1.0 / (1.0 + e))"),
    ("sigmoid without abs", "e = np.exp(-np.abs(x))", "e = np.exp(-x)"),
    ("k left raw", "q, k = l2_normalize_rows(q), l2_normalize_rows(k)",
     "q, k = l2_normalize_rows(q), k"),
    ("q normalised by k", "q, k = l2_normalize_rows(q), l2_normalize_rows(k)",
     "q, k = q / np.linalg.norm(k, axis=-1, keepdims=True), l2_normalize_rows(k)"),
]


def _pre_failures(tmp_path, orc, old, new):
    import importlib.util

    import oracle_pins
    text = open(PRE_SRC).read()
    if old is not None:
        assert text.count(old) == 1, f"mutation anchor {old!r} must occur once"
        text = text.replace(old, new)
    path = tmp_path / "preops_variant.py"
    path.write_text(text)
    spec = importlib.util.spec_from_file_location("preops_variant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    failed = []
    for pin in oracle_pins.PREOP_PINS:
        try:
            pin(orc, pre=mod)
        except Exception:
            failed.append(pin.__name__)
    return failed


def test_unmodified_preops_pass(tmp_path, orc):
    assert _pre_failures(tmp_path, orc, None, None) == []


@pytest.mark.parametrize("name,old,new", PRE_MUTANTS, ids=[m[0] for m in PRE_MUTANTS])
def test_preop_mutant_is_caught(tmp_path, orc, name, old, new):
    assert _pre_failures(tmp_path, orc, old, new), f"no pin catches '{name}'"
