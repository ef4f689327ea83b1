"""attn_fwd_rows (query rows at a global offset) and the sequence-parallel
prefill on one GPU.

attn_fwd_rows with q_offset = 0 is attn_fwd bit for bit.  With an offset,
the rows of a block are compared with the oracle's rows of the whole
sequence (the oracle sees the full Q, so no offset logic is shared).  The
sequence-parallel prefill is emulated rank after rank (each rank's all-gather
replaced by the whole K and V; no inter-rank waiting on one GPU), and the
joined blocks must match the oracle over the whole sequence."""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_sm_gb300 import binding as attn
from attention_forward_sm_gb300 import sp_decode, sp_prefill
from attention_forward_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_ABS, TOL_REL, TOL_MEAN, TOL_LSE = 2e-2, 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    from attention_forward_sm_gb300 import _build
    _build.build()
    attn.load()
    assert torch.cuda.is_available(), "gpu tests need a CUDA device"


def check(o, lse, o_ref, lse_ref):
    o64 = o.float().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    err = np.abs(o64 - o_ref)
    assert not ((err > TOL_ABS) & (err > TOL_REL * np.abs(o_ref))).any(), err.max()
    assert err.mean() <= TOL_MEAN
    dl = np.abs(lse.float().cpu().numpy().astype(np.float64).reshape(lse_ref.shape) - lse_ref)
    assert dl.max() <= TOL_LSE, dl.max()


def block_rows(B, Hq, N, r0, r1, limit=None, seed=0):
    rows = np.array([(b * Hq + h) * N + i for b in range(B) for h in range(Hq)
                     for i in range(r0, r1)], dtype=np.int64)
    if limit is not None and rows.size > limit:
        sel = np.sort(np.random.default_rng(seed).choice(rows.size, limit, replace=False))
        return rows, sel
    return rows, None


def rows_call(q_blk, k, v, causal, q0, scale):
    B, Hq, n, D = q_blk.shape
    o = torch.empty_like(q_blk)
    lse = torch.empty((B, Hq, n), dtype=torch.float32, device=q_blk.device)
    attn.attn_fwd_rows(q_blk, k, v, o, lse, B, Hq, k.shape[1], n, k.shape[2], D, causal, q0,
                       scale)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_offset_zero_is_attn_fwd(causal):
    w = W.custom(1, 4, 2, 700, 700, 128, causal, seed_index=1200)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o1, l1 = rows_call(q, k, v, causal, 0, w.scale)
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    attn.attn_fwd(q, k, v, o2, l2, 1, 4, 2, 700, 700, 128, causal, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# B, Hq, Hkv, N, D, first row, rows
OFFSET_CASES = [
    (1, 2, 2, 600, 128, 128, 200),   # offset on a tile boundary
    (1, 4, 2, 1000, 64, 333, 300),   # ragged offset and block
    (2, 2, 1, 500, 128, 499, 1),     # the last row alone
    (1, 2, 2, 300, 128, 0, 300),     # the whole sequence
    (1, 2, 2, 257, 64, 100, 157),    # rows up to the end
    (1, 8, 2, 2048, 128, 1500, 548),
]


@pytest.mark.parametrize("case", OFFSET_CASES,
                         ids=lambda c: "B{}Hq{}Hkv{}N{}D{}r{}n{}".format(*c))
def test_rows_at_an_offset_match_the_whole_sequence(case):
    B, Hq, Hkv, N, D, r0, n = case
    w = W.custom(B, Hq, Hkv, N, N, D, True, seed_index=1210 + r0 % 97)
    q, k, v = W.make_inputs(w, "cpu")
    qb = q[:, :, r0:r0 + n].contiguous().cuda()
    o, lse = rows_call(qb, k.cuda(), v.cuda(), True, r0, w.scale)
    torch.cuda.synchronize()
    rows, _ = block_rows(B, Hq, N, r0, r0 + n)
    o_ref, lse_ref = oracle.attn_rows(q, k, v, B, Hq, Hkv, N, N, D, True,
                                      float(np.float32(w.scale)), rows=rows)
    check(o, lse, o_ref, lse_ref)


def test_offset_past_the_keys_sees_every_key():
    """Rows whose global index is >= Nk see all keys: the causal call equals
    the non-causal one there."""
    w = W.custom(1, 2, 2, 256, 300, 128, True, seed_index=1230)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o1, l1 = rows_call(q, k, v, True, 300, w.scale)
    o2, l2 = rows_call(q, k, v, False, 0, w.scale)
    torch.cuda.synchronize()
    torch.testing.assert_close(o1, o2, atol=0, rtol=0)
    torch.testing.assert_close(l1, l2, atol=0, rtol=0)


@pytest.mark.parametrize("world,B,Hq,Hkv,N,D,causal",
                         [(2, 1, 4, 2, 1000, 128, True), (3, 2, 4, 4, 777, 64, True),
                          (4, 1, 8, 2, 8192, 128, True), (3, 1, 4, 1, 500, 128, False),
                          (5, 1, 2, 2, 3, 128, True)])
def test_sp_prefill_emulated_ranks(world, B, Hq, Hkv, N, D, causal):
    w = W.custom(B, Hq, Hkv, N, N, D, causal, seed_index=1240 + world)
    q, k, v = W.make_inputs(w, "cpu")
    kd, vd = k.cuda(), v.cuda()
    limit = 4096 if N > 2000 else None
    for r in range(world):
        s0, s1 = sp_decode.shard_range(N, world, r)
        if s1 == s0:
            continue
        qb = q[:, :, s0:s1].contiguous().cuda()
        o, lse = sp_prefill._library_local_attn(qb, kd, vd, causal, s0, w.scale)
        torch.cuda.synchronize()
        rows, sel = block_rows(B, Hq, N, s0, s1, limit=limit, seed=r)
        o = o.reshape(-1, D)
        lse = lse.reshape(-1)
        if sel is not None:
            rows, o, lse = rows[sel], o[torch.from_numpy(sel).cuda()], lse[torch.from_numpy(sel).cuda()]
        o_ref, lse_ref = oracle.attn_rows(q, k, v, B, Hq, Hkv, N, N, D, causal,
                                          float(np.float32(w.scale)), rows=rows)
        check(o, lse, o_ref, lse_ref)


def test_negative_offset_is_rejected():
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 8, dtype=torch.float32, device="cuda")
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_rows(q, q, q, o, lse, 1, 1, 1, 8, 8, 64, True, -1, 0.125)
