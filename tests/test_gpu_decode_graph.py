"""The decode step as a replayed CUDA graph (attn_decode_graph_*), on the GPU.

A replay runs the same two kernels as attn_decode_splitkv on the buffers'
contents at replay time, so its results are compared bit for bit with the
direct call, and with the oracle within the decode tolerance."""
import math

import numpy as np
import pytest
import torch

import oracle
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


def direct(q, k, v, nsplit):
    B, Hq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    attn.attn_decode_splitkv(q, k, v, o, lse, B, Hq, k.shape[1], k.shape[2], D, nsplit)
    return o, lse


def check_oracle(o, lse, q, k, v):
    B, Hq, D = q.shape
    o_ref, lse_ref = oracle.decode(q.cpu(), k.cpu(), v.cpu(), B, Hq, k.shape[1], k.shape[2], D,
                                   scale=float(np.float32(1.0 / math.sqrt(D))))
    o64 = o.float().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    err = np.abs(o64 - o_ref)
    assert not ((err > TOL_ABS) & (err > TOL_REL * np.abs(o_ref))).any()
    assert err.mean() <= TOL_MEAN
    dl = np.abs(lse.cpu().numpy().astype(np.float64).reshape(lse_ref.shape) - lse_ref).max()
    assert dl <= TOL_LSE


@pytest.mark.parametrize("shape", [(2, 8, 2, 3000, 128, 8), (1, 4, 4, 777, 64, 5),
                                   (1, 32, 8, 4096, 128, 16)],
                         ids=lambda s: "B{}Hq{}Hkv{}Nk{}D{}s{}".format(*s))
def test_graph_replay_matches_direct_call(shape):
    B, Hq, Hkv, Nk, D, nsplit = shape
    w = W.custom(B, Hq, Hkv, 1, Nk, D, False, seed_index=800 + Nk % 89, decode=True,
                 nsplit=nsplit)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    g = attn.DecodeGraph(q, k, v, nsplit)
    try:
        o_g, l_g = g.replay()
        o_d, l_d = direct(q, k, v, nsplit)
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_d) and torch.equal(l_g, l_d)
        check_oracle(o_g, l_g, q, k, v)
        # new contents at the same addresses: the next step's query, an
        # updated cache entry; the replay sees them
        w2 = W.custom(B, Hq, Hkv, 1, Nk, D, False, seed_index=850 + Nk % 89, decode=True,
                      nsplit=nsplit)
        q2, k2, _ = (t.cuda() for t in W.make_inputs(w2, "cpu"))
        q.copy_(q2)
        k[:, :, Nk // 2].copy_(k2[:, :, 0])
        o_g, l_g = g.replay()
        o_d, l_d = direct(q, k, v, nsplit)
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_d) and torch.equal(l_g, l_d)
        check_oracle(o_g, l_g, q, k, v)
    finally:
        g.close()
    assert attn.attn_get_device_error() == 0


def test_graph_many_replays_and_streams():
    w = W.custom(4, 32, 8, 1, 8192, 128, False, seed_index=860, decode=True, nsplit=16)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    g = attn.DecodeGraph(q, k, v, 16)
    ref_o, ref_l = direct(q, k, v, 16)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(100):
            g.replay(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(g.o, ref_o) and torch.equal(g.lse, ref_l)
    g.close()
    g.close()  # idempotent
    assert attn.attn_get_device_error() == 0


def test_graph_create_errors_launch_nothing():
    q = torch.zeros(1, 4, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 2, 64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.DecodeGraph(q, k, k, 65)  # nsplit > Nk
    assert e.value.status == -3
    with pytest.raises(attn.AttnError) as e:
        attn.attn_decode_graph_launch(0)
    assert e.value.status == -1
