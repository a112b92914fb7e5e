"""The CTA-pair kernel variants against the oracle.

FS_TC_VARIANT selects, once per process, the tensor-core GEMM kernel the
library launches: the single-CTA kernel (default), the CTA-pair kernel for
every GEMM (pair), or for the forward down (pair_down) or gate/up (pair_up)
projections only.  Each variant reruns, in a child process, the oracle
comparisons of the grouped and shared expert GEMMs (bf16 and FP8) and of the
small FarSkip stacks: the same tolerances, the same seeded inputs.
"""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    "tests/test_gpu_kernels.py::test_grouped_swiglu",
    "tests/test_gpu_kernels.py::test_shared_expert",
    "tests/test_gpu_fp8.py::test_grouped_swiglu_fp8",
    "tests/test_gpu_fp8.py::test_shared_expert_fp8",
    "tests/test_gpu_stack.py::test_small_stack_wirings",
    "tests/test_gpu_fp8.py::test_small_stack_fp8",
]


@pytest.mark.gpu
@pytest.mark.parametrize("variant", ["pair", "pair_down", "pair_up"])
def test_kernel_variant_against_oracle(variant):
    env = dict(os.environ, FS_TC_VARIANT=variant)
    env.pop("FS_PARITY_LOG", None)
    cmd = [sys.executable, "-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider"]
    c = subprocess.run(cmd + ["--collect-only"] + CASES, capture_output=True, text=True, timeout=300, cwd=ROOT)
    n = re.search(r"(\d+) tests? collected", c.stdout)
    assert n, c.stdout[-2000:]
    r = subprocess.run(cmd + ["-x"] + CASES, capture_output=True, text=True, timeout=900, env=env, cwd=ROOT)
    tail = "\n".join((r.stdout + r.stderr).strip().splitlines()[-15:])
    assert r.returncode == 0, "FS_TC_VARIANT=%s:\n%s" % (variant, tail)
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and m.group(1) == n.group(1), tail      # every parametrised case of CASES ran
    print("FS_TC_VARIANT=%s: %s cases passed" % (variant, m.group(1)))
