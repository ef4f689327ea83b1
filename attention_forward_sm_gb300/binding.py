"""ctypes binding of libattn.so (include/attn.h).

Argument marshalling only: tensors become device pointers, the torch stream
becomes a ``cudaStream_t``; every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if the library is missing or
cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn.so")

ATTN_STATUS = {
    0: "ATTN_OK", -1: "ATTN_ERR_NULL", -2: "ATTN_ERR_ALIGN", -3: "ATTN_ERR_SHAPE",
    -4: "ATTN_ERR_DEVICE", -5: "ATTN_ERR_LAUNCH", -6: "ATTN_ERR_ALLOC", -7: "ATTN_ERR_TMA",
    -8: "ATTN_ERR_CUDA", -9: "ATTN_ERR_SCRATCH",
}
EXPORTED = ["attn_fwd", "attn_fwd_rows", "attn_fwd_fp8", "attn_fwd_host", "attn_fwd_host_workspace_bytes",
            "attn_decode_splitkv", "attn_decode_splitkv_noalloc",
            "attn_status_string", "attn_get_device_error", "attn_decode_workspace_bytes",
            "attn_selftest_wait_timeout", "attn_decode_splitkv_states", "attn_combine_states",
            "attn_decode_graph_create", "attn_decode_graph_launch", "attn_decode_graph_destroy"]
DEVERR_SELFTEST = 0x10
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def load(path: str = LIB_PATH):
    """Load libattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m attention_forward_sm_gb300._build`")
        lib = ctypes.CDLL(path)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
        lib.attn_fwd.restype = i
        lib.attn_fwd_rows.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp]
        lib.attn_fwd_rows.restype = i
        lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
        lib.attn_fwd_host.restype = i
        lib.attn_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.attn_fwd_host_workspace_bytes.restype = ctypes.c_longlong
        lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, f, f, f, vp]
        lib.attn_fwd_fp8.restype = i
        lib.attn_decode_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.attn_decode_splitkv.restype = i
        lib.attn_decode_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.attn_decode_splitkv_noalloc.restype = i
        lib.attn_status_string.argtypes = [i]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_get_device_error.argtypes = [vp]
        lib.attn_get_device_error.restype = i
        lib.attn_decode_splitkv_states.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.attn_decode_splitkv_states.restype = i
        lib.attn_combine_states.argtypes = [vp, vp, vp, vp, i, i, i, vp]
        lib.attn_combine_states.restype = i
        lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
        lib.attn_selftest_wait_timeout.restype = i
        lib.attn_decode_graph_create.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                                 ctypes.POINTER(vp)]
        lib.attn_decode_graph_create.restype = i
        lib.attn_decode_graph_launch.argtypes = [vp, vp]
        lib.attn_decode_graph_launch.restype = i
        lib.attn_decode_graph_destroy.argtypes = [vp]
        lib.attn_decode_graph_destroy.restype = i
        lib.attn_decode_workspace_bytes.argtypes = [i, i, i, i]
        lib.attn_decode_workspace_bytes.restype = ctypes.c_longlong
        _lib = lib
        return lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int):
    if rc != 0:
        msg = load().attn_status_string(rc).decode()
        raise AttnError(rc, msg)


# ----------------------------------------------------------------------------- C-ABI names


def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, causal, scale, stream=None) -> None:
    """``attn_fwd`` of include/attn.h: tensors (or raw device pointers), sizes,
    causal flag, scale, and a torch stream / raw handle (None = current)."""
    _check(load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                           int(Hkv), int(Nq), int(Nk), int(D), int(bool(causal)), float(scale),
                           _stream(stream)))


def attn_fwd_rows(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, causal, q_offset, scale,
                  stream=None) -> None:
    """``attn_fwd_rows`` of include/attn.h: ``attn_fwd`` for query rows
    q_offset .. q_offset+Nq-1 of a longer sequence (the causal mask uses the
    global row index)."""
    _check(load().attn_fwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                                int(Hkv), int(Nq), int(Nk), int(D), int(bool(causal)),
                                int(q_offset), float(scale), _stream(stream)))


def attn_fwd_host(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, causal, scale, stream=None) -> None:
    """``attn_fwd_host`` of include/attn.h: host (CPU, ideally pinned) tensors
    in and out; asynchronous on the stream."""
    _check(load().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                                int(Hkv), int(Nq), int(Nk), int(D), int(bool(causal)),
                                float(scale), _stream(stream)))


def attn_fwd_host_workspace_bytes(B, Hq, Hkv, Nq, Nk, D) -> int:
    return int(load().attn_fwd_host_workspace_bytes(int(B), int(Hq), int(Hkv), int(Nq), int(Nk),
                                                    int(D)))


def attn_fwd_fp8(q, k, vt, o, lse, B, Hq, Hkv, Nq, Nk, D, causal, scale, q_scale, k_scale,
                 v_scale, stream=None) -> None:
    """``attn_fwd_fp8`` of include/attn.h: e4m3 q, k and V transposed
    ([B, Hkv, D, Nk]), per-tensor dequantisation scales, bf16 o."""
    _check(load().attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(vt), _ptr(o), _ptr(lse), int(B), int(Hq),
                               int(Hkv), int(Nq), int(Nk), int(D), int(bool(causal)),
                               float(scale), float(q_scale), float(k_scale), float(v_scale),
                               _stream(stream)))


def attn_decode_splitkv(q, kcache, vcache, o, lse, B, Hq, Hkv, Nk, D, nsplit, stream=None) -> None:
    """``attn_decode_splitkv`` of include/attn.h."""
    _check(load().attn_decode_splitkv(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(o), _ptr(lse),
                                      int(B), int(Hq), int(Hkv), int(Nk), int(D), int(nsplit),
                                      _stream(stream)))


def attn_decode_splitkv_noalloc(q, kcache, vcache, o, lse, B, Hq, Hkv, Nk, D, nsplit,
                                stream=None) -> None:
    """``attn_decode_splitkv_noalloc`` of include/attn.h: the same decode for
    callers that cannot allocate device memory during the call; its scratch
    is a fixed 8 MiB device array shared by all calls on a device (order
    calls that could overlap on the GPU)."""
    _check(load().attn_decode_splitkv_noalloc(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(o),
                                              _ptr(lse), int(B), int(Hq), int(Hkv), int(Nk),
                                              int(D), int(nsplit), _stream(stream)))


def attn_status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def attn_get_device_error(stream=None) -> int:
    """Synchronise the stream, return and clear the device error word."""
    rc = load().attn_get_device_error(_stream(stream))
    if rc < 0:
        _check(rc)
    return rc


def attn_decode_splitkv_states(q, kcache, vcache, o_state, lse, B, Hq, Hkv, Nk, D, nsplit,
                               stream=None) -> None:
    """``attn_decode_splitkv_states`` of include/attn.h (fp32 state output)."""
    _check(load().attn_decode_splitkv_states(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(o_state),
                                             _ptr(lse), int(B), int(Hq), int(Hkv), int(Nk),
                                             int(D), int(nsplit), _stream(stream)))


def attn_combine_states(part_o, part_lse, o, lse, rows, nparts, D, stream=None) -> None:
    """``attn_combine_states`` of include/attn.h."""
    _check(load().attn_combine_states(_ptr(part_o), _ptr(part_lse), _ptr(o), _ptr(lse), int(rows),
                                      int(nparts), int(D), _stream(stream)))


def attn_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the bounded-wait self-test (a wait that is meant to run out)."""
    _check(load().attn_selftest_wait_timeout(int(limit_us), _stream(stream)))


def attn_decode_graph_create(q, kcache, vcache, o, lse, B, Hq, Hkv, Nk, D, nsplit) -> int:
    """``attn_decode_graph_create`` of include/attn.h; returns the handle (an
    integer).  The buffers are bound by address until the handle is
    destroyed: keep the tensors alive."""
    h = ctypes.c_void_p()
    _check(load().attn_decode_graph_create(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(o),
                                           _ptr(lse), int(B), int(Hq), int(Hkv), int(Nk), int(D),
                                           int(nsplit), ctypes.byref(h)))
    return int(h.value)


def attn_decode_graph_launch(handle: int, stream=None) -> None:
    """``attn_decode_graph_launch`` of include/attn.h: replay one decode step."""
    _check(load().attn_decode_graph_launch(handle or None, _stream(stream)))


def attn_decode_graph_destroy(handle: int) -> None:
    """``attn_decode_graph_destroy`` of include/attn.h."""
    _check(load().attn_decode_graph_destroy(handle or None))


def attn_decode_workspace_bytes(B, Hq, D, nsplit) -> int:
    return int(load().attn_decode_workspace_bytes(int(B), int(Hq), int(D), int(nsplit)))


# ----------------------------------------------------------------------------- tensor helpers


def _check_ranks(tensors: dict, ranks: dict):
    import torch
    for name, x in tensors.items():
        if not isinstance(x, torch.Tensor):
            raise TypeError(f"{name} must be a torch tensor")
        if x.dim() != ranks[name]:
            raise ValueError(f"{name} must have {ranks[name]} dimensions, got {x.dim()}")


def _check_inputs(tensors: dict, shapes: dict):
    """The helpers below pass raw pointers to the library, which cannot see
    dtypes or strides: check here that every input is a contiguous bf16 CUDA
    tensor, all on one device, with the expected ranks and matching sizes
    (``shapes`` maps a size name to the values the tensors give it)."""
    import torch
    dev = None
    for name, x in tensors.items():
        if x.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16, got {x.dtype}")
        if not x.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not x.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dev is None:
            dev = x.device
        elif x.device != dev:
            raise ValueError(f"{name} is on {x.device}, expected {dev}")
    for size, values in shapes.items():
        if len(set(values)) != 1:
            raise ValueError(f"inconsistent {size}: {values}")



def forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """O, LSE = attention(q [B,Hq,Nq,D], k/v [B,Hkv,Nk,D]) with outputs
    allocated by torch on q's device."""
    import torch
    _check_ranks({"q": q, "k": k, "v": v}, {"q": 4, "k": 4, "v": 4})  # [B, H, N, D]
    _check_inputs({"q": q, "k": k, "v": v},
                  {"B": (q.shape[0], k.shape[0], v.shape[0]), "D": (q.shape[3], k.shape[3], v.shape[3]),
                   "Hkv": (k.shape[1], v.shape[1]), "Nk": (k.shape[2], v.shape[2])})
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, causal, scale, stream)
    return o, lse


class DecodeGraph:
    """One decode step captured as a CUDA graph for fixed q / cache / output
    tensors (held here, so their addresses stay valid); ``replay()`` runs the
    step on the buffers' current contents."""

    def __init__(self, q, kcache, vcache, nsplit: int):
        import torch
        self.handle = 0
        _check_decode_inputs(q, kcache, vcache)
        B, Hq, D = q.shape
        Hkv, Nk = kcache.shape[1], kcache.shape[2]
        self.q, self.kcache, self.vcache = q, kcache, vcache
        self.o = torch.empty_like(q)
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
        self.handle = attn_decode_graph_create(q, kcache, vcache, self.o, self.lse, B, Hq, Hkv,
                                               Nk, D, nsplit)

    def replay(self, stream=None):
        attn_decode_graph_launch(self.handle, stream)
        return self.o, self.lse

    def close(self):
        if self.handle:
            h, self.handle = self.handle, 0
            attn_decode_graph_destroy(h)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _check_decode_inputs(q, kcache, vcache):
    # q [B, Hq, D], caches [B, Hkv, Nk, D]
    _check_ranks({"q": q, "kcache": kcache, "vcache": vcache}, {"q": 3, "kcache": 4, "vcache": 4})
    _check_inputs({"q": q, "kcache": kcache, "vcache": vcache},
                  {"B": (q.shape[0], kcache.shape[0], vcache.shape[0]),
                   "D": (q.shape[2], kcache.shape[3], vcache.shape[3]),
                   "Hkv": (kcache.shape[1], vcache.shape[1]), "Nk": (kcache.shape[2], vcache.shape[2])})


def decode(q, kcache, vcache, nsplit: int, stream=None):
    """O, LSE = split-KV decode(q [B,Hq,D], caches [B,Hkv,Nk,D])."""
    import torch
    _check_decode_inputs(q, kcache, vcache)
    B, Hq, D = q.shape
    Hkv, Nk = kcache.shape[1], kcache.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    attn_decode_splitkv(q, kcache, vcache, o, lse, B, Hq, Hkv, Nk, D, nsplit, stream)
    return o, lse
