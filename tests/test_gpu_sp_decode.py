"""Sequence-parallel decode building blocks on one GPU: the key axis is cut
into rank shards (uneven, one possibly empty), each shard is decoded into an
fp32 state by attn_decode_splitkv_states, and attn_combine_states recombines
the stacked states; the result must match the oracle over the whole cache.
Ranks are emulated one after another (no inter-rank waiting on one GPU)."""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_sm_gb300 import binding as attn
from attention_forward_sm_gb300 import sp_decode
from attention_forward_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    from attention_forward_sm_gb300 import _build
    _build.build()
    attn.load()
    assert torch.cuda.is_available(), "gpu tests need a CUDA device"


@pytest.mark.parametrize("world,B,Hq,Hkv,Nk,D", [(3, 2, 8, 2, 1000, 128), (4, 1, 4, 4, 5000, 64),
                                                (8, 8, 32, 8, 65536, 128), (5, 1, 4, 1, 3, 128)])
def test_sharded_states_recombine_to_full_decode(world, B, Hq, Hkv, Nk, D):
    w = W.custom(B, Hq, Hkv, 1, Nk, D, False, seed_index=900 + world, decode=True, nsplit=8)
    q, k, v = W.make_inputs(w, "cuda")
    states = []
    for r in range(world):
        s0, s1 = sp_decode.shard_range(Nk, world, r)
        ks, vs = k[:, :, s0:s1].contiguous(), v[:, :, s0:s1].contiguous()
        if s1 > s0:
            o_r, l_r = sp_decode._library_local_states(q, ks, vs, 8)
        else:
            o_r = torch.zeros(B * Hq, D, device="cuda")
            l_r = torch.full((B * Hq,), -math.inf, device="cuda")
        states.append(sp_decode.pack_state(o_r, l_r))
    part_o, part_lse = sp_decode.unpack_states(torch.stack(states))
    o, lse = sp_decode._library_combine(part_o, part_lse)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(q.cpu(), k.cpu(), v.cpu(), B, Hq, Hkv, Nk, D,
                                   scale=float(np.float32(1.0 / math.sqrt(D))))
    err = np.abs(o.float().cpu().numpy() - o_ref)
    assert not ((err > 2e-2) & (err > 2e-2 * np.abs(o_ref))).any(), err.max()
    assert err.mean() <= 2e-3
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3
    assert attn.attn_get_device_error() == 0


def test_states_entry_matches_plain_decode():
    w = W.custom(2, 8, 2, 1, 3000, 128, False, seed_index=950, decode=True, nsplit=16)
    q, k, v = W.make_inputs(w, "cuda")
    o_state = torch.empty(2, 8, 128, device="cuda")
    l_state = torch.empty(2, 8, device="cuda")
    attn.attn_decode_splitkv_states(q, k, v, o_state, l_state, 2, 8, 2, 3000, 128, 16)
    o = torch.empty_like(q)
    lse = torch.empty(2, 8, device="cuda")
    attn.attn_decode_splitkv(q, k, v, o, lse, 2, 8, 2, 3000, 128, 16)
    torch.cuda.synchronize()
    assert torch.equal(o_state.to(torch.bfloat16), o)
    assert torch.equal(l_state, lse)
