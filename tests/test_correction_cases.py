"""CPU checks of the correction-path inputs (tests/correction_cases.py):
they make the kernel's rescale rule fire on most (row, tile) pairs, they sit
where they claim (at, just under and just over the threshold), the exact
construction has integer log2 scores and reaches the 2^8 weight ceiling, and
the tight output bound used with it on the GPU would catch an FP8 weight that
saturated at 448.  No GPU needed."""
import math

import numpy as np
import pytest
import torch

import oracle
import correction_cases as CC

SHAPES = [
    # B, Hq, Hkv, Nq, Nk, D, causal
    (2, 4, 2, 300, 2000, 128, False),
    (1, 4, 1, 1000, 1000, 128, True),
    (2, 4, 2, 300, 2000, 64, False),
]


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
@pytest.mark.parametrize("construction", ["exact", "near", "ramp"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "Nq{}Nk{}D{}{}".format(
    s[3], s[4], s[5], "c" if s[6] else ""))
def test_cases_fire_the_rescale(shape, construction, kind):
    B, Hq, Hkv, Nq, Nk, D, causal = shape
    if kind == "fp8" and D != 128:
        pytest.skip("the FP8 forward has D = 128 only")
    case = CC.make_case(construction, kind, shape)
    u = CC.log2_scores(case, B, Hq, Hkv, Nq, Nk, D)
    fires, active, top = CC.replay_rescale(u, Nq, Nk, causal, case["R"])
    frac = CC.fire_fraction(fires, active)
    assert frac >= 0.5, f"rescale fires on {frac:.2f} of (row, tile >= 1) pairs"
    R = case["R"]
    if construction == "exact":
        assert np.array_equal(u, np.rint(u)), "scores are not integers in log2 units"
        # the largest weight reaches 2^(R + bias) = 2^8 exactly, never more
        assert top.max() == R
        assert (top == R).sum() >= 0.25 * len(top)
    if construction == "near":
        # tile maxima rising by R - 1/4 (no rescale) and R + 1/4 (rescale)
        rows = u.shape[0]
        i = np.arange(rows) % Nq
        vis = np.minimum(i + 1, Nk) if causal else np.full(rows, Nk)
        m = np.full(rows, -np.inf)
        under = over = 0
        for t in range(math.ceil(Nk / CC.TILE)):
            lo, hi = t * CC.TILE, min(Nk, (t + 1) * CC.TILE)
            seg = u[:, lo:hi].copy()
            seg[np.arange(lo, hi)[None, :] >= vis[:, None]] = -np.inf
            mt = seg.max(axis=1)
            ok = np.isfinite(mt) & np.isfinite(m)
            rise = np.where(ok, mt - m, np.nan)
            under += int(np.sum(ok & (rise > R - 0.5) & (rise <= R)))
            over += int(np.sum(ok & (rise > R) & (rise < R + 0.5)))
            m = np.where(fires[:, t], mt, m)
        assert under > 0.1 * rows and over > 0.1 * rows, (under, over)


def test_scale_search_is_exact():
    for target in (1.0, 16.0, 64.0, 0.25):
        s = np.float32(CC.scale_for_log2_step(target))
        assert np.float32(s * CC.LOG2E_F32) == np.float32(target)


def _emulate_fp8(case, shape, rows, R_rule):
    """The FP8 kernel's arithmetic on the exact construction, in fp64 with
    E4M3 rounding of the weights: running max moved past R_rule, weights
    p = 2^(u - m + 6) rounded (saturating at 448) for P*V, the row sum from
    the unrounded weights.  Returns O for the listed flat rows."""
    B, Hq, Hkv, Nq, Nk, D, causal = shape
    u = CC.log2_scores(case, B, Hq, Hkv, Nq, Nk, D)[rows]
    G = Hq // Hkv
    v = case["v8"].double()
    out = np.zeros((len(rows), D))
    for n, r in enumerate(rows):
        b, h, i = r // (Hq * Nq), (r // Nq) % Hq, r % Nq
        vis = min(i + 1, Nk) if causal else Nk
        vr = v[b, h // G].numpy()
        m, l, acc = -np.inf, 0.0, np.zeros(D)
        for t in range(math.ceil(vis / CC.TILE)):
            lo, hi = t * CC.TILE, min(vis, (t + 1) * CC.TILE)
            mt = u[n, lo:hi].max()
            if m == -np.inf or mt > m + R_rule:
                alpha = 0.0 if m == -np.inf else 2.0 ** (m - mt)
                acc *= alpha
                l *= alpha
                m = mt
            p = 2.0 ** (u[n, lo:hi] - m + 6.0)
            p8 = torch.from_numpy(np.minimum(p, 448.0)).to(torch.float8_e4m3fn).double().numpy()
            acc += p8 @ vr[lo:hi]
            l += p.sum()
        out[n] = acc * case["v_scale"] / l
    return out


def test_tight_fp8_bound_sees_saturation():
    """The exact construction's tight bound (2^-8 |O| + 2^-12 v_scale max|V|)
    holds for the kernel's rule and fails when the threshold is one too high
    (weights 2^9 saturate at 448)."""
    shape = (1, 2, 1, 64, 1024, 128, False)
    B, Hq, Hkv, Nq, Nk, D, causal = shape
    case = CC.level_case(*shape, kind="fp8", seed=3)
    rows = np.arange(B * Hq * Nq)
    o_ref, _ = oracle.attn_rows_fp8(case["q8"], case["k8"], case["v8"], B, Hq, Hkv, Nq, Nk, D,
                                    causal, case["scale"], case["q_scale"], case["k_scale"],
                                    case["v_scale"], rows=rows)
    bound = 2.0 ** -8 * np.abs(o_ref) + 2.0 ** -12 * case["v_scale"] * \
        case["v8"].double().abs().max().item()
    good = _emulate_fp8(case, shape, rows, CC.THRESHOLD["fp8"])
    assert (np.abs(good - o_ref) <= bound).all()
    bad = _emulate_fp8(case, shape, rows, CC.THRESHOLD["fp8"] + 1)
    assert (np.abs(bad - o_ref) > bound).any()
