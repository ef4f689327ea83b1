"""The per-stream scratch cache behind attn_decode_splitkv, on the GPU.

The cache changes where the partial states live, not what the kernels
compute, so every result is compared bit for bit with the no-allocation
variant (same kernels, fixed scratch) and with the oracle within the decode
tolerance: repeated calls on one stream, a call that needs a larger buffer,
more streams than the cache remembers (entries pass from stream to stream)
running at the same time, and a call captured into a CUDA graph (which takes
the stream-ordered allocation path)."""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_sm_gb300 import binding as attn
from attention_forward_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_ABS, TOL_REL, TOL_MEAN, TOL_LSE = 2e-2, 2e-2, 2e-3, 1e-3
CACHE_ENTRIES = 8  # streams remembered per device (decode_scratch.cu)


@pytest.fixture(scope="module", autouse=True)
def _library():
    from attention_forward_sm_gb300 import _build
    _build.build()
    attn.load()
    assert torch.cuda.is_available(), "gpu tests need a CUDA device"


def inputs(B, Hq, Hkv, Nk, D, nsplit, seed):
    w = W.custom(B, Hq, Hkv, 1, Nk, D, False, seed_index=seed, decode=True, nsplit=nsplit)
    return tuple(t.cuda() for t in W.make_inputs(w, "cpu"))


def decode(q, k, v, nsplit, stream=None, noalloc=False):
    B, Hq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    fn = attn.attn_decode_splitkv_noalloc if noalloc else attn.attn_decode_splitkv
    fn(q, k, v, o, lse, B, Hq, k.shape[1], k.shape[2], D, nsplit,
       stream.cuda_stream if stream is not None else None)
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


def test_repeated_calls_and_growth_on_one_stream():
    s = torch.cuda.Stream()
    small = inputs(1, 8, 2, 1000, 128, 4, 970)
    large = inputs(2, 16, 4, 3000, 128, 24, 971)  # 2*16*24*129*4 bytes > the small call's
    with torch.cuda.stream(s):
        outs = [decode(*small, 4, s), decode(*large, 24, s), decode(*small, 4, s),
                decode(*large, 24, s)]
    s.synchronize()
    ref_small = decode(*small, 4, noalloc=True)
    ref_large = decode(*large, 24, noalloc=True)
    torch.cuda.synchronize()
    for (o, l), (ro, rl) in zip(outs, [ref_small, ref_large, ref_small, ref_large]):
        assert torch.equal(o, ro) and torch.equal(l, rl)
    check_oracle(*outs[0], *small)
    check_oracle(*outs[1], *large)


def test_more_streams_than_cache_entries_concurrently():
    n = CACHE_ENTRIES + 3
    streams = [torch.cuda.Stream() for _ in range(n)]
    data = [inputs(1, 8, 2, 2048 + 64 * i, 64 if i % 2 else 128, 3 + i % 5, 972 + i)
            for i in range(n)]
    torch.cuda.synchronize()
    outs = []
    for rnd in range(2):  # the second round finds most entries taken over
        for i, (s, d) in enumerate(zip(streams, data)):
            with torch.cuda.stream(s):
                outs.append((i, decode(*d, 3 + i % 5, s)))
    torch.cuda.synchronize()
    for i, (o, l) in outs:
        ro, rl = decode(*data[i], 3 + i % 5, noalloc=True)
        torch.cuda.synchronize()
        assert torch.equal(o, ro) and torch.equal(l, rl), f"stream {i}"
    check_oracle(*outs[0][1], *data[0])
    check_oracle(*outs[1][1], *data[1])


def test_call_captured_in_a_cuda_graph():
    q, k, v = inputs(2, 8, 2, 1500, 128, 6, 990)
    o = torch.empty_like(q)
    lse = torch.empty((2, 8), dtype=torch.float32, device=q.device)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        # warm the cache on this stream first, then capture on it
        attn.attn_decode_splitkv(q, k, v, o, lse, 2, 8, 2, 1500, 128, 6, s.cuda_stream)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        attn.attn_decode_splitkv(q, k, v, o, lse, 2, 8, 2, 1500, 128, 6,
                                 torch.cuda.current_stream().cuda_stream)
    o.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    ro, rl = decode(q, k, v, 6, noalloc=True)
    torch.cuda.synchronize()
    assert torch.equal(o, ro) and torch.equal(lse, rl)
    check_oracle(o, lse, q, k, v)
    del g
