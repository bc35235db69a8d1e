"""Host-side checks that need no GPU: the binding rejects operands on the
wrong or on several devices before any launch, the parity checker rejects
planted errors and excuses only output rounding, and bench.py refuses a
--gpus that the launch does not provide."""
import os
import subprocess
import sys
from types import SimpleNamespace

import numpy as np
import pytest

from tests.parity import TOL_O_MAX, check_fwd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _fake(dev, cuda=True):
    return SimpleNamespace(is_cuda=cuda, device=dev)


def test_device_of_rejects_mixed_and_host_operands():
    from exact_attention_67_gb300._lib import _device_of
    assert _device_of(_fake("cuda:1"), None, _fake("cuda:1")) == "cuda:1"
    with pytest.raises(ValueError, match="different devices"):
        _device_of(_fake("cuda:0"), _fake("cuda:1"))
    with pytest.raises(ValueError, match="CUDA"):
        _device_of(_fake("cuda:0"), _fake("cpu", cuda=False))


def _ref(shape=(2, 64, 16), seed=0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape) * 0.5, rng.standard_normal(shape[:-1])


def _bf16(x):
    """Round to bf16 (8 significant bits), nearest-even, in numpy."""
    x32 = np.asarray(x, np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


def test_check_fwd_accepts_rounded_exact_values_and_rejects_a_planted_error():
    o, lse = _ref()
    check_fwd(_bf16(o), lse.copy(), o, lse, "rounded")
    bad = _bf16(o)
    bad[1, 7, 3] += 1.5 * TOL_O_MAX
    with pytest.raises(AssertionError, match="over"):
        check_fwd(bad, lse.copy(), o, lse, "planted max")
    with pytest.raises(AssertionError):
        check_fwd(_bf16(o) + 2e-3, lse.copy(), o, lse, "planted mean")
    with pytest.raises(AssertionError):
        check_fwd(_bf16(o), lse + 2e-3, o, lse, "planted lse")


def test_check_fwd_excuses_only_rounding_at_large_magnitude():
    o, lse = _ref()
    o[0, 0, 0] = 4.39498          # bf16 neighbours 4.375 and 4.40625
    got = _bf16(o)
    assert abs(got[0, 0, 0] - o[0, 0, 0]) > TOL_O_MAX
    msg = check_fwd(got, lse.copy(), o, lse, "large")
    assert "1 element(s) excused" in msg
    got[0, 0, 0] = 4.375          # the other neighbour: more than half an ulp away
    with pytest.raises(AssertionError):
        check_fwd(got, lse.copy(), o, lse, "wrong neighbour")
    o[0, 0, 1] = 2.5              # half an ulp 0.0078 < 1e-2: never excused
    got = _bf16(o)
    got[0, 0, 1] += 0.0117
    with pytest.raises(AssertionError):
        check_fwd(got, lse.copy(), o, lse, "mid magnitude")


def _bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=e, timeout=600)


def test_bench_refuses_gpus_that_differ_from_world_size():
    r = _bench("--gpus", "4", "--steps", "1", env={"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode == 2
    assert "WORLD_SIZE=2" in r.stderr


def test_bench_gpus_2_without_gpus_fails_loudly():
    """Outside torchrun, --gpus 2 relaunches itself as two ranks; on a host
    without GPUs every rank fails, and so does the run."""
    import torch
    if torch.cuda.is_available() and torch.cuda.device_count() >= 2:
        pytest.skip("this host has GPUs: the relaunch would run for real")
    r = _bench("--gpus", "2", "--steps", "1", "--warmup", "3", "--no-cpu-baseline", "--no-e2e", "--no-clocks")
    assert r.returncode != 0
    assert "needs CUDA device" in (r.stdout + r.stderr)


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_for_hash", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_kernel_hash_ignores_comments_and_layout_but_not_code():
    """The DRAM-traffic entries of the bench line are tied to the code of the
    kernel they were captured on: editing a comment or re-indenting keeps
    them, any change of a token drops them."""
    b = _bench_module()
    src = ('// head\nint f(int x) {  /* block\n comment */ return x + 1;  // tail\n}\n'
           'const char* s = "a // not a comment /* nor this */";\nchar c = \'/\';\n')
    same = ('int f(int x)\n{\n    return x + 1;\n}  // another note\n'
            'const char* s = "a // not a comment /* nor this */";  /* x */ char c = \'/\';')
    assert b.code_tokens(src) == b.code_tokens(same)
    assert '"a // not a comment /* nor this */"' in b.code_tokens(src)
    for changed in (src.replace("x + 1", "x + 2"), src.replace("not a comment", "not a comment!"),
                    src.replace("'/'", "'*'")):
        assert b.code_tokens(changed) != b.code_tokens(src)
    # The escape inside a literal does not end it early.
    assert b.code_tokens('s = "q\\" // kept"; // dropped') == 's = "q\\" // kept";'
