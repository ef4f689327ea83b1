"""FP8 (E4M3) forward, attn_fwd_fp8, against the oracle on the GPU.

Tolerance, from the arithmetic of the FP8 path: the scores, the softmax
statistics and the normaliser are fp32 from exact E4M3 products, so LSE
keeps the bf16 bound (1e-3).  O differs from the exact result by the
rounding of each weight p to E4M3 before the P*V product: at most 2^-4 of p
for normal codes (3 mantissa bits, round to nearest), so at most
2^-4 * v_scale * sum_j w_j |V_jd| -- the oracle's output for |V| -- plus
the bf16 rounding of O (2^-8 relative) and an absolute 2^-7 * v_scale for
weights that round in the subnormal range (absolute error <= 2^-10 of the
2^6-scaled weight each, zero-mean).  For the mean: the roundings are
independent and zero-mean with E[delta^2] <= (2^-4)^2 / 3, so the expected
|dO| is at most 2^-4 / sqrt(3) * sqrt(sum_j w_j^2 V_jd^2), which is below
the per-element bound / sqrt(3); mean |dO| <= max(2e-3, mean(bound) / sqrt(3)).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_sm_gb300 import binding as attn
from attention_forward_sm_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SC = W.FP8_SCALES
TOL_LSE, TOL_MEAN = 1e-3, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    from attention_forward_sm_gb300 import _build
    _build.build()
    attn.load()
    assert torch.cuda.is_available(), "gpu tests need a CUDA device"


def run_fp8(w, q8, k8, vt8):
    o = torch.empty((w.B, w.Hq, w.Nq, w.D), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=q8.device)
    attn.attn_fwd_fp8(q8, k8, vt8, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, w.scale,
                      SC["q"], SC["k"], SC["v"])
    torch.cuda.synchronize()
    return o, lse


def check_fp8(w, o, lse, q8, k8, v8, rows=None, label="", scales=None, scale=None):
    sc = SC if scales is None else scales
    args = (w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, w.scale if scale is None else scale,
            sc["q"], sc["k"], sc["v"])
    q8c, k8c, v8c = q8.cpu(), k8.cpu(), v8.cpu()
    o_ref, lse_ref = oracle.attn_rows_fp8(q8c, k8c, v8c, *args, rows=rows)
    # sum_j w_j |V_jd| * v_scale: the oracle on |V| (sign bit cleared)
    v_abs = (v8c.view(torch.uint8) & 0x7F).view(torch.float8_e4m3fn)
    o_abs, _ = oracle.attn_rows_fp8(q8c, k8c, v_abs, *args, rows=rows)
    og = o.float().cpu().numpy().astype(np.float64).reshape(w.B * w.Hq * w.Nq, w.D)
    lg = lse.float().cpu().numpy().astype(np.float64).reshape(-1)
    if rows is not None:
        idx = np.asarray(rows, dtype=np.int64)
        og, lg = og[idx], lg[idx]
    assert np.isfinite(og).all() and np.isfinite(lg).all(), f"{label}: non-finite output"
    err = np.abs(og - o_ref)
    bound = 2.0 ** -4 * o_abs + 2.0 ** -8 * np.abs(o_ref) + 2.0 ** -7 * sc["v"]
    bad = err > bound
    assert not bad.any(), (f"{label}: {int(bad.sum())} elements out of tolerance, "
                           f"max |dO| = {err.max():.3e}, max |dO|/bound = {(err / bound).max():.3f}")
    tol_mean = max(TOL_MEAN, bound.mean() / math.sqrt(3.0))
    assert err.mean() <= tol_mean, f"{label}: mean |dO| = {err.mean():.3e} > {tol_mean:.3e}"
    dl = np.abs(lg - lse_ref).max()
    assert dl <= TOL_LSE, f"{label}: max |dLSE| = {dl:.3e}"
    return err.max(), err.mean(), (err / bound).max()


FP8_SHAPES = [
    # B, Hq, Hkv, Nq, Nk, causal
    (1, 2, 1, 256, 256, False),
    (1, 2, 2, 300, 272, True),      # ragged query tail; key tail inside a 128-key tile
    (2, 4, 2, 128, 1024, False),    # GQA
    (1, 1, 1, 1, 16, False),        # one row, the smallest key count
    (1, 2, 1, 513, 4096, True),
    (1, 3, 3, 640, 640, False),     # MHA, 3 heads, several tiles
]


@pytest.mark.parametrize("shape", FP8_SHAPES, ids=lambda s: "B{}Hq{}Hkv{}Nq{}Nk{}{}".format(
    *s[:5], "c" if s[5] else ""))
def test_fp8_sweep(shape):
    B, Hq, Hkv, Nq, Nk, causal = shape
    w = W.custom(B, Hq, Hkv, Nq, Nk, 128, causal, seed_index=1000 + Nq % 97 + Nk % 89)
    q8, k8, v8, vt8 = (t.cuda() for t in W.make_inputs_fp8(w, "cpu"))
    o, lse = run_fp8(w, q8, k8, vt8)
    check_fp8(w, o, lse, q8, k8, v8, label=str(shape))


@pytest.mark.parametrize("name", ["prefill", "causal"])
def test_fp8_full_size_sampled(name):
    """The benchmark's prefill shapes with FP8 inputs, 4096 sampled rows."""
    w = W.WORKLOADS[name]
    q8, k8, v8, vt8 = W.make_inputs_fp8(w, "cuda")
    o, lse = run_fp8(w, q8, k8, vt8)
    rows = W.sample_rows(w, 4096)
    check_fp8(w, o, lse, q8, k8, v8, rows=rows.numpy(), label=name)


def test_fp8_argument_errors():
    q = torch.zeros(1, 1, 128, 128, dtype=torch.float8_e4m3fn, device="cuda")
    o = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(attn.AttnError) as e:  # Nk not a multiple of 16
        attn.attn_fwd_fp8(q, q, q, o, lse, 1, 1, 1, 128, 120, 128, False, 0.1, 1, 1, 1)
    assert e.value.status == -3
    with pytest.raises(attn.AttnError) as e:  # D = 64
        attn.attn_fwd_fp8(q, q, q, o, lse, 1, 1, 1, 128, 128, 64, False, 0.1, 1, 1, 1)
    assert e.value.status == -3
    with pytest.raises(attn.AttnError) as e:  # negative dequantisation scale
        attn.attn_fwd_fp8(q, q, q, o, lse, 1, 1, 1, 128, 128, 128, False, 0.1, 1, -1, 1)
    assert e.value.status == -3
    assert torch.count_nonzero(o).item() == 0


# ----------------------------------------------------------------------------- correction path
#
# FP8 inputs that make the running max rise past its threshold (2 in log2
# units) on most (row, tile) pairs, built and replayed on the host by
# tests/correction_cases.py.  "exact": integer log2 scores with rises of
# exactly 2 (no rescale: the weight reaches the 2^8 ceiling), 3 and 20, so
# every weight is a power of two, exact in E4M3, and the output meets a
# bound 16 times tighter than the general FP8 one -- a weight that
# saturated at 448 (it would be 2^9 with the threshold one too high) fails
# it; "near": rises 1.75 and 2.25; "ramp": N(0,1) inputs plus a key ramp.

import correction_cases as CC  # noqa: E402

FP8_CORRECTION_SHAPES = [
    # B, Hq, Hkv, Nq, Nk, causal
    (2, 4, 2, 300, 2000, False),
    (1, 4, 1, 1008, 1008, True),   # FP8 keys: a multiple of 16
]


@pytest.mark.parametrize("construction", ["exact", "near", "ramp"])
@pytest.mark.parametrize("shape", FP8_CORRECTION_SHAPES, ids=lambda s: "B{}Hq{}Hkv{}Nq{}Nk{}{}".format(
    *s[:5], "c" if s[5] else ""))
def test_fp8_correction_path(shape, construction):
    B, Hq, Hkv, Nq, Nk, causal = shape
    D = 128
    full = (B, Hq, Hkv, Nq, Nk, D, causal)
    case = CC.make_case(construction, "fp8", full)
    u = CC.log2_scores(case, *full[:6])
    fires, active, top = CC.replay_rescale(u, Nq, Nk, causal, case["R"])
    frac = CC.fire_fraction(fires, active)
    assert frac >= 0.5, f"the inputs rescale only {frac:.2f} of (row, tile >= 1) pairs"
    sc = {"q": case["q_scale"], "k": case["k_scale"], "v": case["v_scale"]}
    w = W.custom(B, Hq, Hkv, Nq, Nk, D, causal)
    q8, k8, v8, vt8 = (case[x].cuda() for x in ("q8", "k8", "v8", "vt8"))
    o = torch.empty((B, Hq, Nq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    attn.attn_fwd_fp8(q8, k8, vt8, o, lse, B, Hq, Hkv, Nq, Nk, D, causal, case["scale"],
                      sc["q"], sc["k"], sc["v"])
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    label = f"{construction} {shape} rescale on {frac:.2f}"
    check_fp8(w, o, lse, q8, k8, v8, label=label, scales=sc, scale=case["scale"])
    if construction == "exact":
        assert top.max() == case["R"]   # some weight reaches 2^(2 + 6) = 2^8
        o_ref, _ = oracle.attn_rows_fp8(q8.cpu(), k8.cpu(), v8.cpu(), B, Hq, Hkv, Nq, Nk, D,
                                        causal, case["scale"], sc["q"], sc["k"], sc["v"])
        og = o.float().cpu().numpy().astype(np.float64).reshape(-1, D)
        bound = 2.0 ** -8 * np.abs(o_ref) + 2.0 ** -12 * sc["v"] * v8.float().abs().max().item()
        bad = np.abs(og - o_ref) > bound
        assert not bad.any(), f"{label}: {int(bad.sum())} elements over the tight bound"


def test_fp8_random_sweep():
    """80 seeded random FP8 problems (Nk a multiple of 16, causal or not, GQA
    groups 1-4, Nq 1-1800, scales up to 0.6), every row against the oracle
    with the derived FP8 bound."""
    rng = np.random.default_rng(20261204)
    for ci in range(80):
        G, Hkv = int(rng.choice([1, 2, 4])), int(rng.integers(1, 4))
        B, Nq = int(rng.integers(1, 4)), int(rng.integers(1, 1800))
        Nk = max(16, int(rng.integers(1, 2400)) // 16 * 16)
        causal = bool(rng.integers(0, 2))
        scale = float(rng.choice([1.0 / math.sqrt(128), 0.3, 0.05, 0.6]))
        w = W.custom(B, Hkv * G, Hkv, Nq, Nk, 128, causal, seed_index=8000 + ci)
        q8, k8, v8, vt8 = (t.cuda() for t in W.make_inputs_fp8(w, "cpu"))
        o = torch.empty((w.B, w.Hq, w.Nq, w.D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device="cuda")
        attn.attn_fwd_fp8(q8, k8, vt8, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, scale,
                          SC["q"], SC["k"], SC["v"])
        torch.cuda.synchronize()
        assert attn.attn_get_device_error() == 0
        check_fp8(w, o, lse, q8, k8, v8, label=f"case {ci}: {w.label()} scale {scale:.3f}",
                  scale=scale)
