"""The pins have teeth: plant one plausible mistake at a time in a copy of the
oracle's C source (on the CPU, in a temporary directory), compile it, and
check that at least one pin of tests/oracle_pins.py rejects it."""
import os
import shutil
import tempfile

import pytest

import oracle
from tests import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, text to find, replacement, which occurrence (0-based))
MUTANTS = [
    ("dS_sign_dq", "double dS = p * (dP - x->D_all[i]);", "double dS = p * (x->D_all[i] - dP);", 0),
    ("dS_sign_dk", "double dS = p * (dP - x->D_all[i]);", "double dS = p * (x->D_all[i] - dP);", 1),
    ("dq_no_scale", "out[cc] += x->scale * dS * kj[cc];", "out[cc] += dS * kj[cc];", 0),
    ("dk_no_scale", "dk[cc] += x->scale * dS * qi[cc];", "dk[cc] += dS * qi[cc];", 0),
    ("dq_uses_v", "const double* kj = x->k + (size_t)j * d;", "const double* kj = x->v + (size_t)j * d;", 0),
    ("dv_uses_q", "dv[cc] += p * dOi[cc];", "dv[cc] += p * qi[cc];", 0),
    ("D_dropped", "x->D_all[i] = dot(x->dO + (size_t)i * x->d, o_row, x->d);", "x->D_all[i] = 0.0;", 0),
    ("causal_strict", "if (causal && j > i) return 0;", "if (causal && j >= i) return 0;", 0),
    ("causal_plus1", "if (causal && j > i) return 0;", "if (causal && j > i + 1) return 0;", 0),
    ("window_off_by_one", "(i - j >= window ||", "(i - j > window ||", 0),
    ("window_one_sided", "(!causal && j - i >= window)", "(0 && j - i >= window)", 0),
    ("lse_log2", "return m + log(l);", "return m + log2(l);", 0),
    ("no_max_subtract", "p[j] = visible(causal, window, i, j) ? exp(p[j] - m) : 0.0;",
     "p[j] = visible(causal, window, i, j) ? exp(p[j]) : 0.0; m = 0.0;", 0),
    ("no_normalise", "for (int j = 0; j < N; ++j) p[j] /= l;", "", 0),
    ("fwd_no_scale", "s[j] = scale * dot(q + (size_t)i * d, k + (size_t)j * d, d);",
     "s[j] = dot(q + (size_t)i * d, k + (size_t)j * d, d);", 0),
    ("online_no_acc_rescale", "for (int c = 0; c < d; ++c) acc[c] *= alpha;", "", 0),
    ("online_no_sum_rescale", "l *= alpha;", "", 0),
]


def _replace_nth(text, old, new, n):
    idx = -1
    for _ in range(n + 1):
        idx = text.find(old, idx + 1)
        assert idx >= 0, f"mutation site not found: {old!r} #{n}"
    return text[:idx] + new + text[idx + len(old):]


@pytest.fixture(scope="module")
def tmpdir_mut():
    d = tempfile.mkdtemp(prefix="oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new,n", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmpdir_mut, name, old, new, n):
    text = open(SRC).read()
    mutated = _replace_nth(text, old, new, n)
    src = os.path.join(tmpdir_mut, f"{name}.c")
    with open(src, "w") as f:
        f.write(mutated)
    lib = oracle.OracleLib(oracle.compile_source(src, os.path.join(tmpdir_mut, f"lib{name}.so")))
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, FloatingPointError, RuntimeError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
