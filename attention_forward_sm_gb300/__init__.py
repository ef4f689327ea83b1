"""GB300 (sm_103a) attention forward and split-KV decode.

The computation runs in ``libattn.so`` (hand-written CUDA, C ABI in
``include/attn.h``); this package is a thin ctypes binding plus the seeded
synthetic workloads used by the tests and the benchmark.

    from attention_forward_sm_gb300 import forward, decode
    o, lse = forward(q, k, v, causal=True)          # q [B,Hq,Nq,D] bf16 on cuda
    o, lse = decode(q1, kcache, vcache, nsplit=32)  # q1 [B,Hq,D]

Build the library with ``python -m attention_forward_sm_gb300._build``.
"""
from .binding import (AttnError, attn_decode_splitkv, attn_decode_workspace_bytes, attn_fwd,
                      attn_get_device_error, attn_status_string, decode, forward, load)

__all__ = ["AttnError", "attn_fwd", "attn_decode_splitkv", "attn_status_string",
           "attn_get_device_error", "attn_decode_workspace_bytes", "forward", "decode", "load"]
