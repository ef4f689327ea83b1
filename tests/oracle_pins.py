"""Pins for the CPU oracle: facts fixed by the pages and by the mathematics,
none of which re-types the oracle's own formula.

Each ``pin_*`` function takes a loaded oracle library and raises
AssertionError when the oracle disagrees with the pinned fact.  They run
against the real oracle in ``test_oracle_pins.py`` and against deliberately
broken copies of it in ``test_oracle_mutants.py`` (every plausible mistake
must trip at least one pin).

Sources of the facts:
  * softmax weights are a probability distribution, so attention output is a
    convex combination of value rows (definition of softmax attention, which
    FlashAttention reproduces exactly -- "FlashAttention-3 vs Triton
    Kernels", introduction);
  * the online running-max/sum recurrence ("correction" role, PyTorch autoWS
    design note, "How the compiler does it") equals the two-pass result;
  * key shards recombined through their lse states equal the unsplit result,
    while summing raw partial outputs does not (smzdm digest, section 5, the
    "denominator pitfall");
  * grouped KV heads are plain MHA with each KV head repeated G times;
  * a hand-worked two-key example with rational answers (tests/golden).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bf16(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def rand_bf16(shape, seed, sigma=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * sigma).to(torch.bfloat16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _run(lib, q, k, v, causal, scale, **kw):
    B, Hq, Nq, D = q.shape
    _, Hkv, Nk, _ = k.shape
    return oracle.attn_rows(q, k, v, B, Hq, Hkv, Nq, Nk, D, causal, scale, lib=lib, **kw)


# --------------------------------------------------------------------------- closed forms


def pin_rows_are_distributions(lib):
    """V = identity (D = Nk) makes O the probability matrix itself: every row
    is non-negative and sums to 1."""
    for causal in (False, True):
        Nk = 24
        q = rand_bf16((1, 2, 24, Nk), 11)
        k = rand_bf16((1, 2, Nk, Nk), 12)
        v = bf16(torch.eye(Nk).expand(1, 2, Nk, Nk).contiguous())
        o, _ = _run(lib, q, k, v, causal, 0.7)
        assert (o >= 0).all()
        np.testing.assert_allclose(o.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        if causal:
            # row i puts zero weight on keys j > i
            P = o.reshape(2, 24, Nk)
            for i in range(24):
                assert np.all(P[:, i, i + 1:] == 0.0)
                assert np.all(P[:, i, : i + 1] > 0.0)


def pin_constant_values(lib):
    """All value rows equal to c -> O = c for any Q, K, causal or not."""
    c = bf16(torch.linspace(-3, 3, 16))
    for causal in (False, True):
        q = rand_bf16((2, 2, 20, 16), 21)
        k = rand_bf16((2, 2, 33, 16), 22)
        v = c.expand(2, 2, 33, 16).contiguous()
        o, _ = _run(lib, q, k, v, causal, 0.25)
        np.testing.assert_allclose(o, np.broadcast_to(f64(c), o.shape), rtol=0, atol=1e-13)


def pin_single_key(lib):
    """Nk = 1: O = V[0] and LSE = scale * <q, k0> (small integers, exact)."""
    q = bf16([[[[1, 2, -1, 3], [0, 1, 0, -2], [4, -3, 2, 1]]]])    # [1,1,3,4]
    k = bf16([[[[2, -1, 1, 1]]]])                                   # [1,1,1,4]
    v = bf16([[[[0.5, -7, 3, 2.25]]]])
    o, lse = _run(lib, q, k, v, False, 0.5)
    dots = np.array([1 * 2 + 2 * -1 + -1 * 1 + 3 * 1, 0 * 2 + 1 * -1 + 0 + -2 * 1,
                     4 * 2 + -3 * -1 + 2 * 1 + 1 * 1], dtype=np.float64)
    np.testing.assert_allclose(lse, 0.5 * dots, rtol=0, atol=1e-15)
    np.testing.assert_allclose(o, np.tile([0.5, -7, 3, 2.25], (3, 1)), rtol=0, atol=0)


def pin_causal_row0(lib):
    """Causal row 0 sees key 0 only: O[0] = V[0], LSE[0] = scale*<q0, k0>."""
    q = bf16(torch.randint(-3, 4, (1, 2, 9, 8)).float())
    k = bf16(torch.randint(-3, 4, (1, 2, 9, 8)).float())
    v = rand_bf16((1, 2, 9, 8), 31)
    o, lse = _run(lib, q, k, v, True, 0.125, rows=[0, 9])
    for r, h in ((0, 0), (1, 1)):
        dot = float((f64(q[0, h, 0]) * f64(k[0, h, 0])).sum())
        assert lse[r] == 0.125 * dot
        np.testing.assert_array_equal(o[r], f64(v[0, h, 0]))


def pin_uniform_attention(lib):
    """Q = 0 makes every visible key equally likely: O = mean of the visible
    value rows, LSE = ln(#visible).  Causal row i: prefix mean, ln(i+1);
    with Nq > Nk the visible set saturates at Nk keys."""
    Nq, Nk = 12, 10
    q = bf16(torch.zeros(1, 1, Nq, 8))
    k = rand_bf16((1, 1, Nk, 8), 41)
    v = rand_bf16((1, 1, Nk, 8), 42)
    V = f64(v[0, 0])
    o, lse = _run(lib, q, k, v, False, 1.0)
    np.testing.assert_allclose(o, np.broadcast_to(V.mean(0), o.shape), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(Nk), rtol=0, atol=1e-14)
    o, lse = _run(lib, q, k, v, True, 1.0)
    for i in range(Nq):
        n = min(i + 1, Nk)
        np.testing.assert_allclose(o[i], V[:n].mean(0), rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[i], math.log(n), rtol=0, atol=1e-14)
    # scale = 0 reduces to the same case for any Q
    q2 = rand_bf16((1, 1, Nq, 8), 43)
    o, lse = _run(lib, q2, k, v, False, 0.0)
    np.testing.assert_allclose(o, np.broadcast_to(V.mean(0), o.shape), rtol=0, atol=1e-14)


def pin_two_keys_closed_form(lib):
    """Two keys with scores a, b: weights are the logistic sigma(a-b) and
    sigma(b-a), LSE = max + log1p(exp(-|a-b|)).  Gaps up to 200 check that
    the max is subtracted (no overflow) with the right sign."""
    for gap in (0.0, 1.0, 5.0, 50.0, 200.0):
        # q = [1, 0], k0 = [gap, 0], k1 = [0, 0] -> a = gap*scale, b = 0
        q = bf16([[[[1.0, 0.0]]]])
        k = bf16([[[[gap, 0.0], [0.0, 0.0]]]])
        v = bf16([[[[2.0, -1.0], [-4.0, 8.0]]]])
        a, b = float(bf16(gap)), 0.0
        o, lse = _run(lib, q, k, v, False, 1.0)
        w0 = 1.0 / (1.0 + math.exp(-(a - b)))
        w1 = 1.0 / (1.0 + math.exp(-(b - a)))
        np.testing.assert_allclose(o[0], [w0 * 2 + w1 * -4, w0 * -1 + w1 * 8], rtol=1e-14,
                                   atol=1e-14)
        np.testing.assert_allclose(lse[0], max(a, b) + math.log1p(math.exp(-abs(a - b))),
                                   rtol=1e-15, atol=1e-15)


def pin_golden_hand_worked(lib):
    """The hand-worked example in tests/golden/hand_worked.json (rational
    answers derived on paper, see the file)."""
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = bf16(c["q"]).reshape(1, 1, -1, c["D"])
        k = bf16(c["k"]).reshape(1, 1, -1, c["D"])
        v = bf16(c["v"]).reshape(1, 1, -1, c["D"])
        scale = eval(c["scale"], {"math": math})  # noqa: S307 (fixture expression)
        o, lse = _run(lib, q, k, v, c["causal"], scale)
        np.testing.assert_allclose(o, np.array(c["O"], dtype=np.float64), rtol=1e-14, atol=1e-14)
        want = [eval(x, {"math": math}) for x in c["LSE"]]  # noqa: S307
        np.testing.assert_allclose(lse, want, rtol=1e-14, atol=1e-14)


# --------------------------------------------------------------------------- invariants


def pin_key_permutation(lib):
    """Non-causal: permuting K and V rows together changes nothing."""
    q = rand_bf16((1, 2, 7, 16), 51)
    k = rand_bf16((1, 2, 29, 16), 52)
    v = rand_bf16((1, 2, 29, 16), 53)
    perm = torch.randperm(29, generator=torch.Generator().manual_seed(54))
    o1, l1 = _run(lib, q, k, v, False, 0.3)
    o2, l2 = _run(lib, q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), False, 0.3)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def pin_value_linearity(lib):
    """O is linear in V and LSE does not depend on V: O(aV1 + V2) =
    a O(V1) + O(V2) (a = 2, exact in bf16 scaling)."""
    q = rand_bf16((1, 1, 5, 8), 55)
    k = rand_bf16((1, 1, 13, 8), 56)
    v1 = rand_bf16((1, 1, 13, 8), 57)
    v2 = rand_bf16((1, 1, 13, 8), 58)
    vs = (2 * v1.float() + v2.float()).to(torch.bfloat16)
    ok = (vs.float() == 2 * v1.float() + v2.float()).all()
    for causal in (False, True):
        oa, la = _run(lib, q, k, v1, causal, 0.4)
        ob, lb = _run(lib, q, k, v2, causal, 0.4)
        os_, ls = _run(lib, q, k, vs, causal, 0.4)
        np.testing.assert_allclose(la, lb, rtol=0, atol=0)
        np.testing.assert_allclose(la, ls, rtol=0, atol=0)
        if ok:
            np.testing.assert_allclose(os_, 2 * oa + ob, rtol=0, atol=1e-12)


def pin_shift_invariance(lib):
    """Adding the same vector to every key row shifts each row's scores by a
    constant: O is unchanged and LSE moves by exactly scale*<q, delta>.
    (Non-causal; delta and q are small integers so the shift is exact.)"""
    q = bf16(torch.randint(-2, 3, (1, 1, 6, 8)).float())
    k = bf16(torch.randint(-3, 4, (1, 1, 11, 8)).float())
    delta = torch.randint(-2, 3, (8,)).float()
    k2 = bf16(k.float() + delta)
    v = rand_bf16((1, 1, 11, 8), 59)
    o1, l1 = _run(lib, q, k, v, False, 0.25)
    o2, l2 = _run(lib, q, k2, v, False, 0.25)
    shift = 0.25 * (f64(q[0, 0]) @ delta.double().numpy())
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2 - l1, shift, rtol=0, atol=1e-12)


def pin_online_equals_two_pass(lib):
    """Running max/sum with rescale over blocks of 1, 7, 64, 128 keys equals
    the two-pass definition (algebraic identity) to 1e-12."""
    q = rand_bf16((1, 2, 40, 32), 61)
    k = rand_bf16((1, 2, 300, 32), 62, sigma=2.0)
    v = rand_bf16((1, 2, 300, 32), 63)
    for causal in (False, True):
        o0, l0 = _run(lib, q, k, v, causal, 0.5)
        for block in (1, 7, 64, 128):
            o1, l1 = _run(lib, q, k, v, causal, 0.5, mode="online", block=block)
            np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
            np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)


def pin_split_equals_unsplit(lib):
    """Key chunks recombined through their lse states give the unsplit result
    for nsplit = 1, 2, 3, 32, Nk (ragged and empty chunks included)."""
    Nk = 96
    q = rand_bf16((2, 2, 50, 16), 71)
    k = rand_bf16((2, 2, Nk, 16), 72)
    v = rand_bf16((2, 2, Nk, 16), 73)
    for causal in (False, True):
        o0, l0 = _run(lib, q, k, v, causal, 0.35)
        for ns in (1, 2, 3, 32, 7, Nk):
            o1, l1 = _run(lib, q, k, v, causal, 0.35, mode="split", nsplit=ns)
            np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
            np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)


def pin_naive_partial_sum_is_wrong(lib):
    """The denominator pitfall: summing (or averaging) the raw per-chunk
    outputs does NOT reproduce attention, while the lse combine does."""
    B, H, Nq, Nk, D = 1, 1, 4, 64, 8
    q = rand_bf16((B, H, Nq, D), 81, sigma=2.0)
    k = rand_bf16((B, H, Nk, D), 82, sigma=2.0)
    v = rand_bf16((B, H, Nk, D), 83)
    o0, l0 = _run(lib, q, k, v, False, 0.5)
    po, pl = oracle.partials(q, k, v, B, H, H, Nq, Nk, D, False, 0.5, 4, lib=lib)
    naive_sum = po.sum(axis=1)
    naive_mean = po.mean(axis=1)
    assert np.abs(naive_sum - o0).max() > 1e-2
    assert np.abs(naive_mean - o0).max() > 1e-2
    oc, lc = oracle.combine(po, pl, lib=lib)
    np.testing.assert_allclose(oc, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lc, l0, rtol=0, atol=1e-12)
    # each partial is itself the attention of its chunk alone
    for c in range(4):
        oc1, lc1 = _run(lib, q, k[:, :, c * 16:(c + 1) * 16].contiguous(),
                        v[:, :, c * 16:(c + 1) * 16].contiguous(), False, 0.5)
        np.testing.assert_allclose(po[:, c], oc1, rtol=0, atol=1e-13)
        np.testing.assert_allclose(pl[:, c], lc1, rtol=0, atol=1e-13)


def pin_gqa_is_repeated_mha(lib):
    """Hq = 4*Hkv with kv head floor(h/4) equals MHA on K, V with each head
    repeated 4 times along the head axis."""
    q = rand_bf16((2, 8, 9, 16), 91)
    k = rand_bf16((2, 2, 17, 16), 92)
    v = rand_bf16((2, 2, 17, 16), 93)
    kr = k.repeat_interleave(4, dim=1).contiguous()
    vr = v.repeat_interleave(4, dim=1).contiguous()
    for causal in (False, True):
        o1, l1 = _run(lib, q, k, v, causal, 0.25)
        o2, l2 = _run(lib, q, kr, vr, causal, 0.25)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def pin_row_subset_consistency(lib):
    """Asking for a subset of rows (any order) returns exactly those rows of
    the full result."""
    q = rand_bf16((2, 3, 10, 8), 95)
    k = rand_bf16((2, 3, 12, 8), 96)
    v = rand_bf16((2, 3, 12, 8), 97)
    o, l = _run(lib, q, k, v, True, 0.3)
    rows = [59, 0, 17, 3, 42]
    o2, l2 = _run(lib, q, k, v, True, 0.3, rows=rows)
    np.testing.assert_array_equal(o2, o[rows])
    np.testing.assert_array_equal(l2, l[rows])


# --------------------------------------------------------------------------- independent implementations


def pin_textbook_torch_float64(lib):
    """torch float64 softmax(scale*QK^T + mask) @ V and logsumexp on tiny
    shapes (GQA via repeat_interleave), causal and not, Nq != Nk."""
    for (B, Hq, Hkv, Nq, Nk, D, seed) in ((1, 2, 2, 16, 16, 8, 1), (2, 4, 2, 13, 21, 16, 2),
                                          (1, 4, 1, 33, 20, 8, 3)):
        q = rand_bf16((B, Hq, Nq, D), 100 + seed)
        k = rand_bf16((B, Hkv, Nk, D), 200 + seed)
        v = rand_bf16((B, Hkv, Nk, D), 300 + seed)
        G = Hq // Hkv
        Q = q.double()
        K = k.double().repeat_interleave(G, dim=1)
        V = v.double().repeat_interleave(G, dim=1)
        for causal in (False, True):
            S = torch.matmul(Q, K.transpose(-1, -2)) * 0.3
            if causal:
                mask = torch.ones(Nq, Nk, dtype=torch.bool).triu(1)
                S = S.masked_fill(mask, float("-inf"))
            ref_o = torch.matmul(torch.softmax(S, dim=-1), V).reshape(-1, D).numpy()
            ref_l = torch.logsumexp(S, dim=-1).reshape(-1).numpy()
            o, l = _run(lib, q, k, v, causal, 0.3)
            np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(l, ref_l, rtol=1e-13, atol=1e-13)


def pin_brute_force_fsum(lib):
    """Pure-Python third implementation with an explicit score matrix and
    math.fsum (correctly rounded sums), B=1, H<=2, N<=16, D<=8."""
    for (Hq, Hkv, Nq, Nk, D, causal, seed) in ((2, 1, 5, 16, 8, False, 4), (2, 2, 16, 11, 4, True, 5),
                                              (1, 1, 3, 3, 2, True, 6)):
        q = rand_bf16((1, Hq, Nq, D), 400 + seed)
        k = rand_bf16((1, Hkv, Nk, D), 500 + seed)
        v = rand_bf16((1, Hkv, Nk, D), 600 + seed)
        scale = 0.45
        Q, K, V = q.double().tolist(), k.double().tolist(), v.double().tolist()
        G = Hq // Hkv
        want_o, want_l = [], []
        for h in range(Hq):
            g = h // G
            for i in range(Nq):
                keys = [j for j in range(Nk) if (not causal or j <= i)]
                s = [scale * math.fsum(Q[0][h][i][d] * K[0][g][j][d] for d in range(D))
                     for j in keys]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                z = math.fsum(e)
                want_l.append(m + math.log(z))
                want_o.append([math.fsum(e[t] / z * V[0][g][j][d] for t, j in enumerate(keys))
                               for d in range(D)])
        o, l = _run(lib, q, k, v, causal, scale)
        np.testing.assert_allclose(o, np.array(want_o), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(l, np.array(want_l), rtol=1e-14, atol=1e-14)


def pin_decode_matches_prefill_last_row(lib):
    """Decode (one query, all keys) equals the non-causal prefill of a
    single-row query tensor, and the last row of a causal prefill whose
    query count equals the key count."""
    B, Hq, Hkv, Nk, D = 2, 4, 2, 37, 16
    qd = rand_bf16((B, Hq, D), 701)
    k = rand_bf16((B, Hkv, Nk, D), 702)
    v = rand_bf16((B, Hkv, Nk, D), 703)
    od, ld = oracle.decode(qd, k, v, B, Hq, Hkv, Nk, D, scale=0.25, lib=lib)
    # embed the decode query as the last row of a causal Nq = Nk prefill
    qp = torch.zeros(B, Hq, Nk, D, dtype=torch.bfloat16)
    qp[:, :, -1] = qd
    rows = [(b * Hq + h) * Nk + Nk - 1 for b in range(B) for h in range(Hq)]
    op, lp = oracle.attn_rows(qp, k, v, B, Hq, Hkv, Nk, Nk, D, True, 0.25, rows, lib=lib)
    np.testing.assert_array_equal(od, op)
    np.testing.assert_array_equal(ld, lp)


# --------------------------------------------------------------------------- FP8 inputs


# Code -> value facts of the E4M3 format (OCP 8-bit floating point): zero,
# the smallest subnormal 2^-9, the largest subnormal 7 * 2^-9, the smallest
# normal 2^-6, one, 1 + 1/8, two, the largest finite value 448, and the
# sign bit.
E4M3_FACTS = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
              0x39: 1.125, 0x40: 2.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9)}


def pin_e4m3_format_facts(lib):
    """Values the format fixes, and NaN codes rejected."""
    codes = torch.tensor(sorted(E4M3_FACTS), dtype=torch.uint8)
    got = oracle.e4m3_to_bf16(codes, lib=lib).double().tolist()
    assert got == [E4M3_FACTS[c] for c in sorted(E4M3_FACTS)], got
    for nan_code in (0x7F, 0xFF):
        try:
            oracle.e4m3_to_bf16(torch.tensor([nan_code], dtype=torch.uint8), lib=lib)
        except ValueError:
            continue
        raise AssertionError(f"NaN code {nan_code:#x} accepted")


def pin_e4m3_matches_torch_and_is_monotone(lib):
    """All 254 finite codes equal torch's own float8_e4m3fn decoding (an
    independent library routine); positive codes increase strictly and the
    sign bit negates."""
    codes = torch.tensor([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=torch.uint8)
    got = oracle.e4m3_to_bf16(codes, lib=lib).double()
    ref = codes.view(torch.float8_e4m3fn).double()
    assert torch.equal(got, ref)
    pos = got[:127]
    assert bool((pos[1:] > pos[:-1]).all())
    assert torch.equal(got[127:], -pos)


def rand_e4m3(shape, seed, sigma=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * sigma).clamp(-448, 448).to(torch.float8_e4m3fn)


def pin_fp8_brute_force_with_scales(lib):
    """FP8 attention with dequantisation scales against a pure-Python fp64
    computation on torch-decoded codes (q_scale*Q, k_scale*K, v_scale*V)."""
    Hq, Hkv, Nq, Nk, D = 2, 1, 6, 9, 8
    q8, k8, v8 = (rand_e4m3((1, h, n, D), 900 + i)
                  for i, (h, n) in enumerate(((Hq, Nq), (Hkv, Nk), (Hkv, Nk))))
    scale, qs, ks, vs = 0.3, 1.5, 0.75, 2.5
    Q = (q8.double() * qs).tolist()
    K = (k8.double() * ks).tolist()
    V = (v8.double() * vs).tolist()
    for causal in (False, True):
        want_o, want_l = [], []
        for h in range(Hq):
            for i in range(Nq):
                keys = [j for j in range(Nk) if (not causal or j <= i)]
                s_ = [scale * math.fsum(Q[0][h][i][d] * K[0][0][j][d] for d in range(D))
                      for j in keys]
                m = max(s_)
                e = [math.exp(x - m) for x in s_]
                z = math.fsum(e)
                want_l.append(m + math.log(z))
                want_o.append([math.fsum(e[t] / z * V[0][0][j][d] for t, j in enumerate(keys))
                               for d in range(D)])
        o, l = oracle.attn_rows_fp8(q8, k8, v8, 1, Hq, Hkv, Nq, Nk, D, causal, scale, qs, ks, vs,
                                    lib=lib)
        np.testing.assert_allclose(o, np.array(want_o), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l, np.array(want_l), rtol=1e-13, atol=1e-13)


ALL_PINS = [
    pin_rows_are_distributions, pin_constant_values, pin_single_key, pin_causal_row0,
    pin_uniform_attention, pin_two_keys_closed_form, pin_golden_hand_worked, pin_key_permutation,
    pin_value_linearity, pin_shift_invariance, pin_online_equals_two_pass,
    pin_split_equals_unsplit, pin_naive_partial_sum_is_wrong, pin_gqa_is_repeated_mha,
    pin_row_subset_consistency, pin_textbook_torch_float64, pin_brute_force_fsum,
    pin_decode_matches_prefill_last_row, pin_e4m3_format_facts,
    pin_e4m3_matches_torch_and_is_monotone, pin_fp8_brute_force_with_scales,
]
