"""GPU parity: the CUDA library (called through its C ABI) against the CPU
fp64 oracle on the same seeded bf16 inputs.

Tolerance (per element of O): |dO| <= 2e-2 absolute OR <= 2e-2 relative to
|O_ref|; over the checked elements mean |dO| <= 2e-3; max |dLSE| <= 1e-3
(absolute, natural log).  Large workloads are checked on >= 4096 sampled
query rows (row 0 and the last row always included, plus the first and last
row of every 128-row tile of one head when causal).
"""
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


def check(o_gpu, lse_gpu, o_ref, lse_ref, label=""):
    o = o_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    lse = lse_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(lse_ref.shape)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), f"{label}: non-finite output"
    err = np.abs(o - o_ref)
    bad = (err > TOL_ABS) & (err > TOL_REL * np.abs(o_ref))
    assert not bad.any(), (f"{label}: {int(bad.sum())} elements out of tolerance, "
                           f"max |dO| = {err.max():.3e}")
    assert err.mean() <= TOL_MEAN, f"{label}: mean |dO| = {err.mean():.3e}"
    dl = np.abs(lse - lse_ref).max()
    assert dl <= TOL_LSE, f"{label}: max |dLSE| = {dl:.3e}"
    return err.max(), err.mean(), dl


def run_prefill(w, q, k, v, stream=None):
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=q.device)
    attn.attn_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, w.scale, stream)
    torch.cuda.synchronize()
    return o, lse


def oracle_prefill(w, q, k, v, rows=None, scale=None):
    s = float(np.float32(w.scale if scale is None else scale))
    return oracle.attn_rows(q.cpu(), k.cpu(), v.cpu(), w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D,
                            w.causal, s, rows)


# ----------------------------------------------------------------------------- prefill

PREFILL_SHAPES = [
    # B, Hq, Hkv, Nq, Nk, D, causal
    (1, 2, 2, 256, 256, 64, False),
    (2, 4, 4, 100, 100, 128, False),
    (1, 2, 2, 129, 300, 128, True),
    (1, 8, 2, 513, 513, 128, True),
    (2, 4, 1, 300, 77, 64, False),
    (1, 2, 2, 1, 1, 128, False),
    (1, 2, 2, 1000, 1, 64, True),
    (1, 2, 2, 700, 200, 128, True),
    (1, 4, 4, 1024, 1024, 128, False),
    (1, 2, 2, 2048, 2048, 64, True),
    (1, 1, 1, 600, 4096, 128, False),
    (1, 4, 2, 1280, 1280, 128, True),
]


@pytest.mark.parametrize("shape", PREFILL_SHAPES, ids=lambda s: "B{}Hq{}Hkv{}Nq{}Nk{}D{}{}".format(
    *s[:6], "c" if s[6] else ""))
def test_prefill_sweep(shape):
    B, Hq, Hkv, Nq, Nk, D, causal = shape
    w = W.custom(B, Hq, Hkv, Nq, Nk, D, causal, seed_index=hash(shape) % 1000)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o, lse = run_prefill(w, q, k, v)
    o_ref, lse_ref = oracle_prefill(w, q, k, v)
    check(o, lse, o_ref.reshape(B, Hq, Nq, D), lse_ref.reshape(B, Hq, Nq), str(shape))


def test_tiny_workload():
    w = W.WORKLOADS["tiny"]
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o, lse = run_prefill(w, q, k, v)
    o_ref, lse_ref = oracle_prefill(w, q, k, v)
    check(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape), "tiny")


@pytest.mark.parametrize("name", ["prefill", "causal", "long_gqa"])
def test_full_size_sampled(name):
    """The full-size workloads, same launch as the benchmark, >= 4096 sampled rows."""
    w = W.WORKLOADS[name]
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = run_prefill(w, q, k, v)
    rows = W.sample_rows(w, 4096)
    assert rows.numel() >= 4096
    o_ref, lse_ref = oracle_prefill(w, q, k, v, rows.numpy())
    o_s = o.reshape(-1, w.D)[rows.cuda()]
    l_s = lse.reshape(-1)[rows.cuda()]
    check(o_s, l_s, o_ref, lse_ref, name)
    if w.causal:
        # causal row 0 of every head attends to key 0 only: O = V[0] exactly (rounded to bf16)
        G = w.Hq // w.Hkv
        v0 = v[:, :, 0, :].repeat_interleave(G, dim=1)
        assert torch.equal(o[:, :, 0, :], v0)


def test_full_size_sampled_d64():
    """The D = 64 benchmark shape (B8 H32 N8192, non-causal; the path that
    issues half of the next Q K^T during the softmax pass), same launch as
    the benchmark, >= 4096 sampled rows."""
    w = W.custom(8, 32, 32, 8192, 8192, 64, False, seed_index=960)
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = run_prefill(w, q, k, v)
    assert attn.attn_get_device_error() == 0
    rows = W.sample_rows(w, 4096)
    assert rows.numel() >= 4096
    o_ref, lse_ref = oracle_prefill(w, q, k, v, rows.numpy())
    check(o.reshape(-1, w.D)[rows.cuda()], lse.reshape(-1)[rows.cuda()], o_ref, lse_ref, "d64")


def test_causal_unit_groups_with_a_partial_last_group():
    """Causal units run in groups of whole KV heads sized to L2 (K+V of
    16.8 MB per KV head at Nk = 32768 gives two KV heads per group); with
    three KV heads the last group holds one.  Every row of every head is
    computed: sampled rows of all six query heads against the oracle, and
    row 0 of each head is V[0] exactly."""
    w = W.custom(1, 6, 3, 32768, 32768, 128, True, seed_index=1200)
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = run_prefill(w, q, k, v)
    rows = W.sample_rows(w, 1024)
    o_ref, lse_ref = oracle_prefill(w, q, k, v, rows.numpy())
    check(o.reshape(-1, w.D)[rows.cuda()], lse.reshape(-1)[rows.cuda()], o_ref, lse_ref,
          "causal groups")
    heads = set((rows // w.Nq).tolist())
    assert heads == set(range(w.B * w.Hq))
    assert torch.equal(o[:, :, 0, :], v[:, :, 0, :].repeat_interleave(2, dim=1))


def test_more_than_2_31_elements():
    """Tensors of more than 2^31 elements (B2 H32 N266240 D128 causal: 4.4 GB each):
    every offset the kernel forms stays in range.  Sampled rows from both
    batch entries against the oracle, and causal row 0 of every head."""
    w = W.custom(2, 32, 32, 266240, 266240, 128, True, seed_index=1300)
    assert w.B * w.Hq * w.Nq * w.D > 2 ** 31
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = run_prefill(w, q, k, v)
    g = torch.Generator().manual_seed(11)
    total = w.B * w.Hq * w.Nq
    rows = torch.unique(torch.cat([torch.randint(0, total, (192,), generator=g),
                                   torch.tensor([total - 1, total // 2 - 1, total // 2])]))
    o_ref, lse_ref = oracle_prefill(w, q, k, v, rows.numpy())
    check(o.reshape(-1, w.D)[rows.cuda()], lse.reshape(-1)[rows.cuda()], o_ref, lse_ref,
          "2^31+ elements")
    assert torch.equal(o[:, :, 0, :], v[:, :, 0, :])
    del q, k, v, o, lse
    torch.cuda.empty_cache()


RANDOM_SHAPES = 24


@pytest.mark.parametrize("case", range(RANDOM_SHAPES))
def test_random_shapes(case):
    """Seeded random shapes over the supported space: B 1-3, KV heads 1-4,
    group size 1-4, Nq and Nk 1-1500, D 64 or 128, causal or not, scale in
    [0, 0.3]."""
    g = torch.Generator().manual_seed(4000 + case)
    ri = lambda lo, hi: int(torch.randint(lo, hi + 1, (1,), generator=g))
    Hkv = ri(1, 4)
    B, Hq, Nq, Nk = ri(1, 3), Hkv * ri(1, 4), ri(1, 1500), ri(1, 1500)
    D, causal = (64, 128)[ri(0, 1)], bool(ri(0, 1))
    scale = float(torch.rand(1, generator=g)) * 0.3
    w = W.custom(B, Hq, Hkv, Nq, Nk, D, causal, seed_index=4100 + case)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    attn.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, causal, scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_prefill(w, q, k, v, scale=scale)
    check(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape),
          f"B{B} Hq{Hq} Hkv{Hkv} Nq{Nq} Nk{Nk} D{D} causal{causal} scale{scale:.3f}")


def test_scale_zero_is_uniform():
    """scale = 0: every visible key has the same weight (oracle and closed form)."""
    w = W.custom(1, 2, 2, 300, 300, 128, True, seed_index=501)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 300), dtype=torch.float32, device="cuda")
    attn.attn_fwd(q, k, v, o, lse, 1, 2, 2, 300, 300, 128, True, 0.0)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_prefill(w, q, k, v, scale=0.0)
    check(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape), "scale0")
    np.testing.assert_allclose(lse.cpu().numpy()[0, 0], np.log(np.arange(1, 301)), atol=1e-4)


def test_deterministic_and_stream():
    w = W.custom(2, 8, 2, 777, 900, 128, True, seed_index=502)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o1, l1 = run_prefill(w, q, k, v)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2 = torch.empty_like(q)
        l2 = torch.empty_like(l1)
        attn.attn_fwd(q, k, v, o2, l2, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, True, w.scale, s)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_back_to_back_odd_shapes():
    """Many launches of odd shapes in a row; the last results still match and no
    kernel gave up a wait."""
    shapes = [(1, 2, 1, n, n + 37, 128 if n % 2 else 64, bool(n % 3)) for n in range(1, 400, 29)]
    data = []
    for sh in shapes:
        w = W.custom(*sh, seed_index=sh[3])
        q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
        data.append((w, q, k, v, torch.empty_like(q),
                     torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device="cuda")))
    for _ in range(20):
        for (w, q, k, v, o, lse) in data:
            attn.attn_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, w.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    for (w, q, k, v, o, lse) in data[::3]:
        o_ref, lse_ref = oracle_prefill(w, q, k, v)
        check(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape), w.label())


# ----------------------------------------------------------------------------- decode


def run_decode(w, q, k, v, nsplit):
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=q.device)
    attn.attn_decode_splitkv(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nk, w.D, nsplit)
    torch.cuda.synchronize()
    return o, lse


def oracle_decode(w, q, k, v):
    s = float(np.float32(1.0 / math.sqrt(w.D)))
    return oracle.decode(q.cpu(), k.cpu(), v.cpu(), w.B, w.Hq, w.Hkv, w.Nk, w.D, scale=s)


def test_decode_workload():
    w = W.WORKLOADS["decode"]
    q, k, v = W.make_inputs(w, "cuda")
    o, lse = run_decode(w, q, k, v, w.nsplit)
    o_ref, lse_ref = oracle_decode(w, q, k, v)
    check(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape), "decode")


DECODE_SHAPES = [
    # B, Hq, Hkv, Nk, D, nsplit
    (1, 4, 1, 1000, 128, 7),
    (2, 8, 2, 9, 64, 4),        # last chunk empty (chunk = 3 keys)
    (1, 3, 1, 513, 128, 1),     # G = 3, no split
    (1, 16, 2, 300, 128, 300),  # one key per chunk
    (2, 2, 2, 4096, 64, 32),    # MHA, D = 64
    (1, 32, 2, 2048, 128, 16),  # G = 16 (two head groups per KV head)
    (3, 12, 4, 777, 64, 5),
]


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=lambda s: "B{}Hq{}Hkv{}Nk{}D{}s{}".format(*s))
def test_decode_sweep(shape):
    B, Hq, Hkv, Nk, D, nsplit = shape
    w = W.custom(B, Hq, Hkv, 1, Nk, D, False, seed_index=600 + Nk % 97, decode=True,
                 nsplit=nsplit)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o, lse = run_decode(w, q, k, v, nsplit)
    o_ref, lse_ref = oracle_decode(w, q, k, v)
    check(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape), str(shape))


@pytest.mark.parametrize("case", range(16))
def test_decode_random_shapes(case):
    """Seeded random decode shapes: B 1-4, KV heads 1-8, group size 1-12 (odd
    ones included), Nk 1-20000, D 64 or 128, nsplit 1..min(Nk, 64)."""
    g = torch.Generator().manual_seed(5000 + case)
    ri = lambda lo, hi: int(torch.randint(lo, hi + 1, (1,), generator=g))
    B, Hkv, G = ri(1, 4), ri(1, 8), ri(1, 12)
    Nk, D = ri(1, 20000), (64, 128)[ri(0, 1)]
    nsplit = ri(1, min(Nk, 64))
    w = W.custom(B, Hkv * G, Hkv, 1, Nk, D, False, seed_index=5100 + case, decode=True,
                 nsplit=nsplit)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o, lse = run_decode(w, q, k, v, nsplit)
    o_ref, lse_ref = oracle_decode(w, q, k, v)
    check(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape),
          f"B{B} Hq{Hkv * G} Hkv{Hkv} Nk{Nk} D{D} nsplit{nsplit}")


def test_decode_split_invariance():
    """Different nsplit give the same result (LSE recombination), within tolerance."""
    w = W.custom(2, 8, 2, 1, 5000, 128, False, seed_index=700, decode=True, nsplit=1)
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o1, l1 = run_decode(w, q, k, v, 1)
    for ns in (2, 3, 32, 257):
        o2, l2 = run_decode(w, q, k, v, ns)
        assert (o1.float() - o2.float()).abs().max().item() < 2e-3
        assert (l1 - l2).abs().max().item() < 1e-4


# ----------------------------------------------------------------------------- boundary


def test_errors_are_returned_not_launched():
    q = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 2, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd(q.data_ptr() + 2, q, q, o, lse, 1, 2, 2, 128, 128, 64, False, 0.125)
    assert e.value.status == -2
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd(q, q, q, o, lse, 1, 2, 2, 128, 128, 96, False, 0.125)
    assert e.value.status == -3
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd(q, q, q, o, lse, 1, 2, 2, 128, 128, 64, False, -1.0)
    assert e.value.status == -3
    with pytest.raises(attn.AttnError) as e:
        attn.attn_decode_splitkv(q, q, q, o, lse, 1, 2, 2, 64, 64, 65)
    assert e.value.status == -3
    assert torch.count_nonzero(o).item() == 0
    assert attn.attn_get_device_error() == 0


# ----------------------------------------------------------------------------- correction path
#
# Inputs whose tile maxima climb, so the kernel's O rescale (the correction
# step: the running max moved by more than 2^8) runs on most (row, tile)
# pairs; tests/correction_cases.py builds them and replays the kernel's rule
# on the host to show that it does.  "exact": integer log2 scores, rises of
# exactly the threshold (no rescale), one over it and far over it, so every
# weight is a power of two and the output also meets a tight bound;
# "near": rises a quarter log2 unit under and over the threshold; "ramp":
# N(0,1) inputs plus a key ramp.

import correction_cases as CC  # noqa: E402

CORRECTION_SHAPES = [
    # B, Hq, Hkv, Nq, Nk, D, causal
    (2, 4, 2, 300, 2000, 128, False),
    (1, 4, 1, 1000, 1000, 128, True),
    (2, 4, 2, 300, 2000, 64, False),
    (1, 2, 2, 700, 1500, 64, True),
]


@pytest.mark.parametrize("construction", ["exact", "near", "ramp"])
@pytest.mark.parametrize("shape", CORRECTION_SHAPES, ids=lambda s: "B{}Hq{}Hkv{}Nq{}Nk{}D{}{}".format(
    *s[:6], "c" if s[6] else ""))
def test_correction_path(shape, construction):
    B, Hq, Hkv, Nq, Nk, D, causal = shape
    case = CC.make_case(construction, "bf16", shape)
    u = CC.log2_scores(case, B, Hq, Hkv, Nq, Nk, D)
    fires, active, top = CC.replay_rescale(u, Nq, Nk, causal, case["R"])
    frac = CC.fire_fraction(fires, active)
    assert frac >= 0.5, f"the inputs rescale only {frac:.2f} of (row, tile >= 1) pairs"
    w = W.custom(B, Hq, Hkv, Nq, Nk, D, causal)
    q, k, v = (case[x].cuda() for x in "qkv")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    attn.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, causal, case["scale"])
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    o_ref, lse_ref = oracle_prefill(w, q, k, v, scale=case["scale"])
    label = f"{construction} {shape} rescale on {frac:.2f}"
    check(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape), label)
    if construction == "exact":
        # every weight is a power of two (the largest 2^8): the only rounding
        # left is bf16 O (2^-9 relative) and fp32 accumulation
        assert top.max() == case["R"]
        og = o.float().cpu().numpy().astype(np.float64).reshape(-1, D)
        ref = o_ref.reshape(-1, D)
        bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * v.float().abs().max().item()
        bad = np.abs(og - ref) > bound
        assert not bad.any(), f"{label}: {int(bad.sum())} elements over the tight bound"


# ----------------------------------------------------------------------------- unit scheduling
#
# The prefill grid has one CTA per (batch*head, query-tile pair) unit, and
# running CTAs take over the ones not started yet (cluster launch control),
# so a CTA works through several units with its barriers and K/V ring
# carried over.  These check every output row when there are several times
# more units than SMs, and two launches running at once on two streams.


@pytest.mark.parametrize("shape", [(2, 16, 4, 1536, 1536, 128, True), (1, 64, 64, 2048, 2048, 64, False),
                                   (3, 32, 8, 640, 2000, 128, False)],
                         ids=lambda s: "B{}Hq{}Hkv{}Nq{}Nk{}D{}{}".format(*s[:6], "c" if s[6] else ""))
def test_many_units_every_row(shape):
    B, Hq, Hkv, Nq, Nk, D, causal = shape
    w = W.custom(B, Hq, Hkv, Nq, Nk, D, causal, seed_index=1400 + Nq % 97)
    units = B * Hq * ((Nq + 255) // 256)
    assert units > 152
    q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
    o, lse = run_prefill(w, q, k, v)
    assert attn.attn_get_device_error() == 0
    o_ref, lse_ref = oracle_prefill(w, q, k, v)
    check(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape), f"{units} units")


def test_two_streams_at_once():
    """Two different problems launched back to back on two streams, with no
    ordering between them, run concurrently; each grid's CTAs take over only
    its own units, so both results match the oracle."""
    w1 = W.custom(2, 16, 16, 2048, 2048, 128, False, seed_index=1500)
    w2 = W.custom(1, 16, 4, 3000, 3000, 64, True, seed_index=1501)
    data = []
    for w in (w1, w2):
        q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
        data.append((w, q, k, v, torch.empty_like(q),
                     torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device="cuda")))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        for s, (w, q, k, v, o, lse) in zip(streams, data):
            attn.attn_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, w.scale, s)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    for (w, q, k, v, o, lse) in data:
        o_ref, lse_ref = oracle_prefill(w, q, k, v)
        check(o, lse, o_ref.reshape(o.shape), lse_ref.reshape(lse.shape), w.label())


def test_random_sweep_many_units():
    """160 seeded random problems (D 64 or 128, causal or not, GQA groups 1-4,
    B 1-3, Nq 1-1800, Nk 1-2400, scales up to 0.6 so that rescales happen),
    every row against the oracle; with up to 3*12*8 units per launch, CTAs
    also take over several units in turn."""
    rng = np.random.default_rng(20261203)
    for ci in range(160):
        D = int(rng.choice([64, 128]))
        G, Hkv = int(rng.choice([1, 2, 4])), int(rng.integers(1, 4))
        B, Nq, Nk = int(rng.integers(1, 4)), int(rng.integers(1, 1800)), int(rng.integers(1, 2400))
        causal = bool(rng.integers(0, 2))
        scale = float(rng.choice([1.0 / math.sqrt(D), 0.3, 0.05, 0.6]))
        w = W.custom(B, Hkv * G, Hkv, Nq, Nk, D, causal, seed_index=7000 + ci)
        q, k, v = (t.cuda() for t in W.make_inputs(w, "cpu"))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device="cuda")
        attn.attn_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, scale)
        torch.cuda.synchronize()
        assert attn.attn_get_device_error() == 0
        o_ref, lse_ref = oracle_prefill(w, q, k, v, scale=scale)
        check(o, lse, o_ref, lse_ref, f"case {ci}: {w.label()} scale {scale:.3f}")
