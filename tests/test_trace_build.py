"""The timeline instrumentation (EXATTN_TRACE in ptx.cuh) is compiled out of
the library; this keeps the tracing build of every kernel file compiling.
Compile only (nvcc, no GPU)."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_67_gb300", "csrc")


@pytest.mark.parametrize("src", ["fwd.cu", "bwd.cu", "dq.cu"])
def test_tracing_build_compiles(src):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    with tempfile.TemporaryDirectory() as d:
        tu = os.path.join(d, "trace_tu.cu")
        with open(tu, "w") as f:
            f.write("#define EXATTN_TRACE\n"
                    "namespace exattn {\n"
                    "__device__ unsigned long long* g_exattn_trace;\n"
                    "__device__ int g_exattn_trace_cta;\n"
                    "}\n"
                    f'#include "{src}"\n')
        r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1", "-c",
                            "-I", CSRC, "-o", os.path.join(d, "trace_tu.o"), tu], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
