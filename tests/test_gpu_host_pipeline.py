"""attn_fwd_host (operands in host memory, pipelined copies) on the GPU: its
results equal attn_fwd on device copies of the same inputs bit for bit, for
shapes cut into one or several (batch, KV-head block) units."""
import pytest
import torch

from attention_forward_sm_gb300 import binding as attn
from attention_forward_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    from attention_forward_sm_gb300 import _build
    _build.build()
    attn.load()
    assert torch.cuda.is_available(), "gpu tests need a CUDA device"


def device_reference(w, q, k, v):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device="cuda")
    attn.attn_fwd(qd, kd, vd, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, w.scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def host_call(w, q, k, v, pinned=True):
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, pin_memory=pinned)
    lse = torch.full((w.B, w.Hq, w.Nq), float("nan"), dtype=torch.float32, pin_memory=pinned)
    attn.attn_fwd_host(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, w.scale)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("shape", [
    (2, 4, 2, 300, 300, 128, True),       # one unit per batch element
    (3, 2, 2, 129, 77, 64, False),        # D = 64, ragged tails
    (1, 32, 8, 16384, 16384, 128, True),  # one batch element cut into 3 KV-head blocks
    (2, 16, 16, 4096, 4096, 128, False),  # 2 blocks per batch element
], ids=lambda s: "B{}Hq{}Hkv{}Nq{}Nk{}D{}{}".format(*s[:6], "c" if s[6] else ""))
def test_host_pipeline_matches_device_call(shape):
    B, Hq, Hkv, Nq, Nk, D, causal = shape
    w = W.custom(B, Hq, Hkv, Nq, Nk, D, causal, seed_index=1100 + Nq % 97)
    q, k, v = W.make_inputs(w, "cpu")
    o_ref, lse_ref = device_reference(w, q, k, v)
    o, lse = host_call(w, q, k, v)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert attn.attn_get_device_error() == 0


def test_host_pipeline_pageable_memory():
    w = W.custom(2, 4, 4, 256, 512, 128, False, seed_index=1150)
    q, k, v = W.make_inputs(w, "cpu")
    o_ref, lse_ref = device_reference(w, q, k, v)
    o, lse = host_call(w, q, k, v, pinned=False)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_host_pipeline_on_a_side_stream_and_repeated():
    w = W.custom(2, 8, 8, 1024, 1024, 128, True, seed_index=1160)
    q, k, v = (t.pin_memory() for t in W.make_inputs(w, "cpu"))
    o_ref, lse_ref = device_reference(w, q, k, v)
    s = torch.cuda.Stream()
    outs = []
    for _ in range(3):
        o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
        lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, pin_memory=True)
        attn.attn_fwd_host(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal,
                           w.scale, s)
        outs.append((o, lse))
    s.synchronize()
    for o, lse in outs:
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
