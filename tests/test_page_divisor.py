"""Host check of the paged cache's page index (no GPU): the reciprocal the
library derives for a page size gives floor(row / page_tokens) exactly, for
every accepted page size up to 2^20 tokens and rows up to 2^31 - 1
(tests/c/page_divisor.cpp, compiled against the library's internal header)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_include():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda.h")):
            return os.path.join(cand, "include")
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
    return None


def test_page_index_reciprocal_is_exact(tmp_path):
    cxx = shutil.which(os.environ.get("CXX", "g++"))
    inc = _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("needs a C++ compiler and the CUDA headers")
    exe = str(tmp_path / "page_divisor")
    cmd = [cxx, "-std=c++17", "-O2", "-Wall", "-Werror", os.path.join(ROOT, "tests", "c", "page_divisor.cpp"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "int4_kv_cache_gb300", "csrc"), "-I", inc,
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("OK")
