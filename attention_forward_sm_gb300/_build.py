"""Build libattn.so in-tree with nvcc for sm_103a (no torch extension, no cmake).

Each CUDA translation unit is compiled in parallel to an object file under
``_build/`` and the objects are linked into ``libattn.so`` next to this file
(the CUDA runtime is linked statically, so the library depends only on the
driver).  ``python -m attention_forward_sm_gb300._build`` runs it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libattn.so")
SOURCES = ["api.cu", "fwd_sm103a.cu", "decode_sm103a.cu", "decode_noalloc.cu", "decode_graph.cu",
           "decode_scratch.cu", "host_pipeline.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "attn.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, extra_flags=(), build_dir: str = BUILD) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    return obj, res.stderr


def build(force: bool = False, verbose: bool = False, lib: str = LIB, extra_flags=(),
          build_dir: str = BUILD) -> str:
    """Compile and link libattn.so (skipped when it is newer than every source).
    ``lib``, ``extra_flags`` and ``build_dir`` build a variant of the library
    elsewhere, e.g. the clock64 event-trace build (``-DATTN_TRACE``)."""
    if not force and lib == LIB and up_to_date():
        return lib
    os.makedirs(build_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda src: _compile(src, extra_flags, build_dir), SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *[o for o, _ in results], "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
