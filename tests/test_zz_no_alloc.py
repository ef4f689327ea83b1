"""attn_decode_splitkv_noalloc against attn_decode_splitkv, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device
memory while they run (memory reserved in full up front by their own
allocator, or no allocator calls allowed on a latency-critical path).  It
must give the same results as the allocating entry point, call after call,
even though every call reuses the same fixed scratch array.  This file is
collected last so that a failure here never hides another test's result.
"""
import numpy as np
import pytest
import torch

from attention_forward_sm_gb300 import binding as attn
from attention_forward_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_ABS, TOL_REL, TOL_MEAN, TOL_LSE = 2e-2, 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    from attention_forward_sm_gb300 import _build
    _build.build()
    attn.load()
    assert torch.cuda.is_available(), "gpu tests need a CUDA device"


def _close(o_a, l_a, o_b, l_b):
    a = o_a.float().cpu().numpy().astype(np.float64)
    b = o_b.float().cpu().numpy().astype(np.float64)
    err = np.abs(a - b)
    assert not ((err > TOL_ABS) & (err > TOL_REL * np.abs(b))).any(), err.max()
    assert err.mean() <= TOL_MEAN, err.mean()
    assert (l_a - l_b).abs().max().item() <= TOL_LSE


@pytest.mark.parametrize("case", ["decode", "ragged"])
def test_noalloc_matches_allocating_entry_point_twice(case):
    if case == "decode":
        w = W.WORKLOADS["decode"]  # B8 Hq32 Hkv8 Nk65536 D128 nsplit32: 4.2 MB of scratch
    else:
        w = W.custom(3, 12, 4, 1, 777, 64, False, seed_index=811, decode=True, nsplit=5)
    assert w.B * w.Hq * w.nsplit * (w.D + 1) * 4 <= attn.NOALLOC_SCRATCH_BYTES
    inputs = [W.make_inputs(w, "cuda"),
              W.make_inputs(W.custom(w.B, w.Hq, w.Hkv, 1, w.Nk, w.D, False, seed_index=w.seed + 1,
                                     decode=True, nsplit=w.nsplit), "cuda")]
    for q, k, v in inputs:  # two calls in a row; the second reuses the first's scratch
        o_ref = torch.empty_like(q)
        l_ref = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        attn.attn_decode_splitkv(q, k, v, o_ref, l_ref, w.B, w.Hq, w.Hkv, w.Nk, w.D, w.nsplit)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
        attn.attn_decode_splitkv_noalloc(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nk, w.D, w.nsplit)
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        _close(o, lse, o_ref, l_ref)
    assert attn.attn_get_device_error() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    q = torch.zeros(64, 64, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(64, 8, 64, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    # 64*64*64*(128+1)*4 bytes = 135 MB > 8 MiB
    with pytest.raises(attn.AttnError) as e:
        attn.attn_decode_splitkv_noalloc(q, kv, kv, o, lse, 64, 64, 8, 64, 128, 64)
    assert e.value.status == -9
    assert torch.count_nonzero(o).item() == 0
