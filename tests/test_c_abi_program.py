"""The C ABI from a plain C program (tests/c_abi_check.c): it compiles with
gcc against include/attn.h and links against libattn.so and the CUDA runtime
alone (CPU test); on a GPU it runs a causal GQA prefill and a split-KV decode
through the ABI and checks them against the oracle's C entry point."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
PKG = os.path.join(ROOT, "attention_forward_sm_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _compile(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    from attention_forward_sm_gb300 import _build
    import oracle
    _build.build()
    oracle.load()  # builds liboracle.so if stale
    exe = str(tmp_path / "c_abi_check")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c_abi_check.c"),
           "-o", exe, "-L", PKG, "-lattn", "-L", ORACLE, "-loracle",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{PKG}:{ORACLE}:{os.path.join(CUDA, 'lib64')}"]
    subprocess.run(cmd, check=True)
    return exe


def test_c_program_compiles_against_the_header(tmp_path):
    assert os.path.exists(_compile(tmp_path))


@pytest.mark.gpu
def test_c_program_runs_on_the_gpu(tmp_path):
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C ABI check passed" in r.stdout
