"""Clock64 event trace of the prefill kernel on a small case.

    python trace_case.py [d128|d64|fp8] [--units N]

Builds a trace variant of the library (``-DATTN_TRACE``, in
``attention_forward_sm_gb300/libattn_trace.so``; the product library is
untouched), runs one launch, reads the stamps of the first 16 CTAs' first
unit through ``attn_trace_copy`` and prints, per query tile, the softmax
pass (S ready -> P published, with its load / max / exponential / store
phases), the hand-off to the MMA warp, the time that warp takes to issue
the tile's P V and next Q K^T, the rest of the wait for the next S, and the
step period, averaged over the middle key tiles.  The pass is stamped by
the tile's first warp; P is complete when the slowest warp of the tile has
arrived, so the hand-off includes the spread between the tile's warps.  The trace stores
cost a little time, so its periods run slightly long; benchmark numbers
come from bench.py.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_forward_sm_gb300 import _build  # noqa: E402
from attention_forward_sm_gb300 import binding as attn  # noqa: E402
from attention_forward_sm_gb300 import workloads as W  # noqa: E402

CASES = {
    "d128": W.custom(4, 32, 32, 4096, 4096, 128, False, seed_index=900),
    "d64": W.custom(8, 32, 32, 4096, 4096, 64, False, seed_index=904),
    "fp8": W.custom(4, 32, 32, 4096, 4096, 128, False, seed_index=903),
}
EVENTS = 8      # softmax: S ready, S loaded, max, exponentials, P arrived; MMA: P taken, S issued; loader
CTAS = 16       # traced CTAs
KV = 64         # traced key tiles per unit


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(CASES), nargs="?", default="d128")
    args = ap.parse_args()
    w = CASES[args.case]
    lib_path = os.path.join(_build.PKG, "libattn_trace.so")
    _build.build(force=True, lib=lib_path, extra_flags=["-DATTN_TRACE"],
                 build_dir=os.path.join(_build.PKG, "_build_trace"))
    lib = attn.load(lib_path)
    lib.attn_trace_copy.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.attn_trace_copy.restype = ctypes.c_int
    if args.case == "fp8":
        q, k, _, v = W.make_inputs_fp8(w, "cuda")
        o = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    else:
        q, k, v = W.make_inputs(w, "cuda")
        o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device="cuda")
    sc = W.FP8_SCALES

    def call():
        if args.case == "fp8":
            attn.attn_fwd_fp8(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal,
                              w.scale, sc["q"], sc["k"], sc["v"])
        else:
            attn.attn_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, w.scale)

    for _ in range(4):
        call()
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    buf = np.zeros(CTAS * 1024, dtype=np.uint64)
    assert lib.attn_trace_copy(buf.ctypes.data, buf.size) == buf.size
    x = buf.astype(np.int64).reshape(CTAS, EVENTS, 2, KV)
    n_kv = min(KV, (w.Nk + 127) // 128)
    js = range(4, n_kv - 2)
    print(f"{args.case}: {w.label()}; cycles, mean over CTAs and key tiles {js.start}..{js.stop - 1}")
    for t in range(2):
        e = lambda ev, d=0: np.array([[x[c, ev, t, j + d] for j in js] for c in range(CTAS)], float)
        s_ready, s_ld, s_max, s_exp, p_arr = e(0), e(1), e(2), e(3), e(4)
        p_taken = e(5)           # the MMA warp took P of key tile j
        s_next = e(6, 1)         # it had issued S of key tile j + 1 (after P V of tile j)
        s_ready_next = e(0, 1)   # softmax saw S of key tile j + 1
        print(f"  tile {t}: pass {np.mean(p_arr - s_ready):6.0f} (load {np.mean(s_ld - s_ready):4.0f},"
              f" max {np.mean(s_max - s_ld):4.0f}, exp {np.mean(s_exp - s_max):4.0f},"
              f" store+arrive {np.mean(p_arr - s_exp):4.0f});"
              f" P -> MMA warp {np.mean(p_taken - p_arr):5.0f}; P V + next Q K^T issued in"
              f" {np.mean(s_next - p_taken):5.0f}; then S ready for the softmax after"
              f" {np.mean(s_ready_next - s_next):5.0f};"
              f" step period {np.mean(np.diff(e(4), axis=1)):6.0f}")


if __name__ == "__main__":
    main()
