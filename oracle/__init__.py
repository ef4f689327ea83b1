"""CPU fp64 attention oracle -- TEST INFRASTRUCTURE, not part of the product.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import this package.  It shares no code
with the CUDA library (``attention_forward_sm_gb300``) and imports nothing
from it; the library never imports this package.

The arithmetic lives in ``oracle.c`` (plain C, fp64, pthreads); this module
builds it with gcc and marshals numpy / torch arrays.  What it computes:

    s_j  = scale * <Q[b,h,i,:], K[b,h//G,j,:]>     for visible keys j
    LSE  = max_j s_j + ln sum_j exp(s_j - max)     (natural log)
    O    = sum_j softmax(s)_j * V[b,h//G,j,:]

with causal visibility j <= i (aligned at row 0).  This is the softmax
attention output that FlashAttention reaches without materialising the score
matrix ("FlashAttention-3 vs Triton Kernels", introduction), with the
lse-carrying recombination of key shards from the smzdm digest, section 5.

Every function is pinned by the CPU tests in ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force, a float64 textbook routine) and by
the mutation tests in ``tests/test_oracle_mutants.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile ``oracle.c`` into a shared library with gcc (no fast-math:
    the oracle keeps IEEE fp64 semantics).  Returns the library path."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", *extra_flags, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _needs_build(path: str) -> bool:
    return (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(_SRC)


def _bind(lib):
    i64, dbl, ip, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_int, ctypes.c_void_p
    common = [vp, vp, vp, i64, i64, i64, i64, i64, i64, ip, dbl, vp, i64]
    lib.oracle_attn_rows.argtypes = common + [vp, vp, ip]
    lib.oracle_attn_rows_online.argtypes = common + [i64, vp, vp, ip]
    lib.oracle_attn_rows_split.argtypes = common + [i64, vp, vp, ip]
    lib.oracle_attn_rows_partials.argtypes = common + [i64, vp, vp, ip]
    lib.oracle_combine.argtypes = [vp, vp, i64, i64, i64, vp, vp]
    lib.oracle_e4m3_to_bf16.argtypes = [vp, vp, i64]
    lib.oracle_e4m3_to_bf16.restype = ctypes.c_int
    for f in (lib.oracle_attn_rows, lib.oracle_attn_rows_online, lib.oracle_attn_rows_split,
              lib.oracle_attn_rows_partials, lib.oracle_combine):
        f.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building if stale) the oracle library.  With ``path`` given,
    load that file instead (used by the mutation tests)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build(_LIB_PATH):
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _as_bf16_bits(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> C-contiguous uint16 bit patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype != torch.bfloat16:
                raise TypeError("oracle inputs must be bf16")
            return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()
                                        .view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(x)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs must be bf16 tensors or uint16 bit arrays")
    return np.ascontiguousarray(a)


def _rows_array(rows, total):
    if rows is None:
        return np.arange(total, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


def _threads(nthreads):
    return int(nthreads) if nthreads else (os.cpu_count() or 1)


def _prep(q, k, v, B, Hq, Hkv, Nq, Nk, D, rows):
    qb, kb, vb = _as_bf16_bits(q), _as_bf16_bits(k), _as_bf16_bits(v)
    if qb.size != B * Hq * Nq * D or kb.size != B * Hkv * Nk * D or vb.size != B * Hkv * Nk * D:
        raise ValueError("tensor sizes do not match (B, Hq, Hkv, Nq, Nk, D)")
    r = _rows_array(rows, B * Hq * Nq)
    return qb, kb, vb, r


def attn_rows(q, k, v, B, Hq, Hkv, Nq, Nk, D, causal, scale, rows=None, *, mode="two_pass",
              block=64, nsplit=1, nthreads=None, lib=None):
    """O [len(rows), D] and LSE [len(rows)] in fp64 for the listed flat query
    rows ``(b*Hq + h)*Nq + i`` (all rows when ``rows`` is None).

    ``mode``: "two_pass" (the definition), "online" (blockwise running
    max / sum, ``block`` keys per step) or "split" (``nsplit`` key chunks
    recombined through their lse states)."""
    lib = lib or load()
    qb, kb, vb, r = _prep(q, k, v, B, Hq, Hkv, Nq, Nk, D, rows)
    o = np.zeros((r.size, D), dtype=np.float64)
    lse = np.zeros(r.size, dtype=np.float64)
    args = [qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, B, Hq, Hkv, Nq, Nk, D, int(causal),
            float(scale), r.ctypes.data, r.size]
    if mode == "two_pass":
        rc = lib.oracle_attn_rows(*args, o.ctypes.data, lse.ctypes.data, _threads(nthreads))
    elif mode == "online":
        rc = lib.oracle_attn_rows_online(*args, int(block), o.ctypes.data, lse.ctypes.data,
                                         _threads(nthreads))
    elif mode == "split":
        rc = lib.oracle_attn_rows_split(*args, int(nsplit), o.ctypes.data, lse.ctypes.data,
                                        _threads(nthreads))
    else:
        raise ValueError(mode)
    if rc != 0:
        raise RuntimeError(f"oracle failed with status {rc}")
    return o, lse


def partials(q, k, v, B, Hq, Hkv, Nq, Nk, D, causal, scale, nsplit, rows=None, *,
             nthreads=None, lib=None):
    """Per-chunk normalised partial outputs [rows, nsplit, D] and their lse
    [rows, nsplit] (-inf for an empty chunk), not yet combined."""
    lib = lib or load()
    qb, kb, vb, r = _prep(q, k, v, B, Hq, Hkv, Nq, Nk, D, rows)
    po = np.zeros((r.size, nsplit, D), dtype=np.float64)
    pl = np.zeros((r.size, nsplit), dtype=np.float64)
    rc = lib.oracle_attn_rows_partials(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, B, Hq, Hkv,
                                       Nq, Nk, D, int(causal), float(scale), r.ctypes.data, r.size,
                                       int(nsplit), po.ctypes.data, pl.ctypes.data,
                                       _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with status {rc}")
    return po, pl


def combine(part_o, part_lse, *, lib=None):
    """Log-sum-exp recombination of partial states (fp64)."""
    lib = lib or load()
    po = np.ascontiguousarray(part_o, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    nrows, nsplit, D = po.shape
    o = np.zeros((nrows, D), dtype=np.float64)
    lse = np.zeros(nrows, dtype=np.float64)
    rc = lib.oracle_combine(po.ctypes.data, pl.ctypes.data, nrows, nsplit, D, o.ctypes.data,
                            lse.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle combine failed with status {rc}")
    return o, lse


def decode(q, kcache, vcache, B, Hq, Hkv, Nk, D, scale=None, *, nthreads=None, lib=None):
    """Single-query decode: q [B,Hq,D], caches [B,Hkv,Nk,D]; all keys visible.
    Returns O [B*Hq, D] and LSE [B*Hq]."""
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    return attn_rows(q, kcache, vcache, B, Hq, Hkv, 1, Nk, D, False, scale, None,
                     nthreads=nthreads, lib=lib)


def e4m3_to_bf16(x, *, lib=None):
    """FP8 E4M3 codes (a uint8 / float8_e4m3fn tensor or uint8 array) -> the
    same values as a bf16 tensor (exact: every E4M3 value is a bf16 value).
    Raises on a NaN code."""
    import torch
    lib = lib or load()
    if isinstance(x, torch.Tensor):
        a = np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.uint8).numpy())
        shape = tuple(x.shape)
    else:
        a = np.ascontiguousarray(np.asarray(x, dtype=np.uint8))
        shape = a.shape
    out = np.zeros(a.size, dtype=np.uint16)
    if lib.oracle_e4m3_to_bf16(a.ctypes.data, out.ctypes.data, a.size) != 0:
        raise ValueError("NaN code in FP8 input")
    return torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).reshape(shape)


def attn_rows_fp8(q8, k8, v8, B, Hq, Hkv, Nq, Nk, D, causal, scale, q_scale, k_scale, v_scale,
                  rows=None, *, nthreads=None, lib=None):
    """Attention on FP8 E4M3 inputs with per-tensor dequantisation scales:
    the real operands are q_scale*Q8, k_scale*K8, v_scale*V8 (Q8, K8, V8 the
    decoded codes; V8 as [B, Hkv, Nk, D]).  Scores are
    scale * <q_scale Q8_i, k_scale K8_j> = (scale*q_scale*k_scale) <Q8_i, K8_j>,
    and O is linear in V, so this is the fp64 definition above on the decoded
    codes with the score scale folded and O multiplied by v_scale (LSE does
    not depend on V).  Returns O [rows, D], LSE [rows] in fp64."""
    lib = lib or load()
    qb, kb, vb = (e4m3_to_bf16(t, lib=lib) for t in (q8, k8, v8))
    o, lse = attn_rows(qb, kb, vb, B, Hq, Hkv, Nq, Nk, D, causal,
                       float(scale) * float(q_scale) * float(k_scale), rows,
                       nthreads=nthreads, lib=lib)
    return o * float(v_scale), lse
