"""The C ABI from plain C: tests/c/abi_example.c (quantize, decode, one fused
step, an argument error) compiled against include/tq.h, libtq.so and the
oracle library.  On the CPU it must compile and link; on a GB300 it must run
and agree with the oracle (codes bit for bit, outputs within 2e-3 / 1e-3)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_example.c")


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime.h")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return None


def _build_example(tmp_path):
    cc = shutil.which(os.environ.get("CC", "gcc"))
    cuda = _cuda_home()
    if cc is None or cuda is None:
        pytest.skip("needs a C compiler and the CUDA toolkit")
    import oracle.build as obuild
    from int4_kv_cache_gb300 import build

    tq_dir = os.path.dirname(build.build())
    oracle_dir = os.path.dirname(obuild.build())
    lib64 = os.path.join(cuda, "lib64")
    exe = str(tmp_path / "abi_example")
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", SRC, "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "oracle"), "-I", os.path.join(cuda, "include"),
           "-L", tq_dir, "-ltq", "-L", oracle_dir, "-ltq_oracle", "-L", lib64, "-lcudart", "-lm",
           f"-Wl,-rpath,{tq_dir}:{oracle_dir}:{lib64}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_abi_example_compiles_and_links(tmp_path):
    _build_example(tmp_path)


@pytest.mark.gpu
def test_c_abi_example_runs(tmp_path):
    from tests.gpu_helpers import need_gpu

    need_gpu()
    exe = _build_example(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("OK"), r.stdout
