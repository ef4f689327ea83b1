"""Failure detection without a GPU fault: a kernel whose pipeline wait can
never complete gives up after its time limit, reports it through the device
error word, and the CUDA context stays usable for the next call."""

import numpy as np
import pytest
import torch

import oracle
from attention_forward_sm_gb300 import binding as attn
from attention_forward_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    from attention_forward_sm_gb300 import _build
    _build.build()
    attn.load()
    assert torch.cuda.is_available(), "gpu tests need a CUDA device"


def test_wait_that_never_completes_is_reported_and_context_survives():
    assert attn.attn_get_device_error() == 0
    attn.attn_selftest_wait_timeout(2000)  # 2 ms limit on a barrier nothing arrives at
    word = attn.attn_get_device_error()    # synchronises the stream
    assert word == attn.DEVERR_SELFTEST
    assert attn.attn_get_device_error() == 0  # reading clears it
    # the context still runs real work correctly
    w = W.custom(1, 2, 2, 300, 300, 128, True, seed_index=77)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 300), dtype=torch.float32, device="cuda")
    attn.attn_fwd(q, k, v, o, lse, 1, 2, 2, 300, 300, 128, True, w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_rows(q.cpu(), k.cpu(), v.cpu(), 1, 2, 2, 300, 300, 128, True,
                                      float(np.float32(w.scale)))
    err = np.abs(o.float().cpu().numpy().reshape(o_ref.shape) - o_ref)
    assert err.max() < 2e-2 and err.mean() < 2e-3
    assert np.abs(lse.cpu().numpy().reshape(-1) - lse_ref).max() < 1e-3
    assert attn.attn_get_device_error() == 0


def test_selftest_rejects_bad_limit():
    with pytest.raises(attn.AttnError):
        attn.attn_selftest_wait_timeout(0)
