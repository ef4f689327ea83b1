"""Inputs that drive the online-softmax correction (the O rescale) on purpose,
and a replay of the kernel's rescale rule to show that they do.

The correction step rescales the accumulated output when a row's running max
changes ("Warp Specialization in Triton: Design and Roadmap", *How the
compiler does it*, the correction partition).  The forward kernel keeps a
stale running max m (log2 units) and moves it -- rescaling O and the row sum
by 2^(m_old - m_new) -- only when a key tile's row max m_tile rises past it by
more than a threshold R: R = 8 for bf16 inputs, R = 2 for FP8, where the
weights p = 2^(u - m + 6) must stay <= 2^8 < 448 (the largest E4M3 value).
Seeded random inputs at the usual scale almost never trigger it after the
first tile, so these cases build scores whose tile maxima climb.

Two constructions:

* ``level_case``: every key j carries an integer level L_j (in units of
  ``quantum`` log2), written in binary into ten spread-out head dimensions
  of K (0/1 digits); every query row i has weight c_i in {1, 2} on those
  dimensions (times the digit's power of two).  With the score scale chosen
  so that scale * log2(e) rounds in fp32 to an exact power of two, every
  score in log2 units is u_ij = c_i * L_j * quantum, exactly, in fp32 as in
  fp64.  Tile t of each KV head has a peak level P_t (four keys), keys one
  and two quanta below it, and the rest 30 log2 units below.  The peaks
  climb so that, for rows with c = 1, the rise over the stale max cycles
  through the three values of ``rises``; a rise moves the max only when it
  exceeds R, and the last tile takes the last entry.  Rows with c = 2 rise
  twice as far.  With ``quantum`` = 1 and rises (R + 18, R, R + 1) -- far
  over the threshold, exactly at it (no rescale), one over it -- every
  weight p is an exact power of two (so P in bf16, and in E4M3 too, is
  exact), the largest reaches 2^(R + bias) = 2^8 exactly, and weights of old
  tiles drop out of E4M3's range in one step rather than being rounded on
  the way: an output check much tighter than the usual tolerance can then
  see a weight that saturated at 448 (a threshold one too high, or a larger
  P bias, gives 2^9 on the tiles that rise by R + 1, the last one among
  them).  With ``quantum`` = 1/4 and rises (R - 1/4, R + 1/4, R + 1/4) the
  rises sit a quarter log2 unit under and over the threshold.
* ``ramp_case``: N(0,1) inputs plus a ramp along one head dimension: query
  rows get a weight in [2, 4] there and the keys of tile t the value
  t * step, so tile maxima climb by well over R on most rows, with random
  noise on top.

``replay_rescale`` applies the kernel's rule (fp32 scale, strict ">", the
first visible tile always sets m) to the scores computed from the actual
bf16 / E4M3 inputs, and reports per (row, tile) whether the rescale fires.
"""
from __future__ import annotations

import math

import numpy as np
import torch

TILE = 128                      # keys per K/V tile of the forward kernel
LOG2E_F32 = np.float32(1.4426950408889634)
THRESHOLD = {"bf16": 8.0, "fp8": 2.0}
P_BIAS = {"bf16": 0.0, "fp8": 6.0}
FP8_SCALES = {"q": 0.5, "k": 2.0, "v": 0.75}   # q*k = 1 exactly
_N_DIGITS = 10
_DIGIT_SHIFT = 6          # q digit weight c * 2^(b - 6)


def scale_for_log2_step(target: float) -> float:
    """An fp32 score scale s with fl32(s * fl32(log2 e)) == target exactly
    (the product the library forms on the host)."""
    s0 = np.float32(target / 1.4426950408889634)
    for k in range(-64, 65):
        s = np.float32(s0 + np.float32(k) * np.spacing(s0))
        if np.float32(s * LOG2E_F32) == np.float32(target):
            return float(s)
    raise AssertionError("no fp32 scale gives an exact log2 step")


def _climb(n_tiles: int, rises, R: float) -> list[float]:
    """Peak level per tile (log2 units for c = 1 rows): the rise over the
    stale max cycles through ``rises``, aligned so that the last tile takes
    the last entry; the max moves past R only."""
    P, m = [0.0], 0.0
    for t in range(1, n_tiles):
        rise = rises[(t - n_tiles) % len(rises)]
        P.append(m + rise)
        if rise > R:
            m = m + rise
    return P


def level_case(B, Hq, Hkv, Nq, Nk, D, causal, *, kind="bf16", quantum=1.0, rises=None,
               seed=0):
    """Inputs of the level construction (module docstring).  Returns a dict
    with q, k, v (bf16) or q8, k8, v8, vt8 (E4M3), the score scale and, for
    FP8, the dequantisation scales.  ``rises`` defaults to (R + 18, R, R + 1)."""
    R = THRESHOLD[kind]
    rises = (R + 18, R, R + 1) if rises is None else rises
    assert D in (64, 128)
    dims = [(D // _N_DIGITS) * b + 3 for b in range(_N_DIGITS)]  # spread over the head dims
    n_tiles = math.ceil(Nk / TILE)
    rng = np.random.default_rng(seed)
    P = _climb(n_tiles, rises, R)
    base = 32.0
    # levels in quanta, per (b, kv head, key)
    L = np.zeros((B, Hkv, Nk), dtype=np.int64)
    for bh in range(B * Hkv):
        b, h = divmod(bh, Hkv)
        for t in range(n_tiles):
            lo, hi = t * TILE, min(Nk, (t + 1) * TILE)
            n = hi - lo
            off = np.full(n, -30.0)
            idx = rng.permutation(n)
            off[idx[:min(4, n)]] = 0.0
            off[idx[4:12]] = -quantum
            off[idx[12:28]] = -2 * quantum
            L[b, h, lo:hi] = np.rint((base + P[t] + off) / quantum).astype(np.int64)
    assert L.min() >= 0 and L.max() < (1 << _N_DIGITS), "levels exceed the binary digits"
    c = rng.integers(1, 3, size=(B, Hq, Nq)).astype(np.float64)
    q = np.zeros((B, Hq, Nq, D))
    k = np.zeros((B, Hkv, Nk, D))
    for b_i, d in enumerate(dims):
        q[..., d] = c * 2.0 ** (b_i - _DIGIT_SHIFT)
        k[..., d] = (L >> b_i) & 1
    # u = scale_log2 * <q, k> = c * L * 2^-shift * scale_log2 = c * L * quantum
    scale_log2 = quantum * 2.0 ** _DIGIT_SHIFT
    out = {"kind": kind, "R": R, "scale_log2": scale_log2}
    g = torch.Generator().manual_seed(seed + 17)
    vv = torch.randn((B, Hkv, Nk, D), generator=g)
    if kind == "bf16":
        out["scale"] = scale_for_log2_step(scale_log2)
        out["q"] = torch.from_numpy(q).to(torch.bfloat16)
        out["k"] = torch.from_numpy(k).to(torch.bfloat16)
        out["v"] = vv.to(torch.bfloat16)
        assert torch.equal(out["q"].double(), torch.from_numpy(q))
    else:
        # the kernel's score scale is scale * q_scale * k_scale * log2 e; with
        # q_scale * k_scale = 1 exactly it is the bf16 one
        out["scale"] = scale_for_log2_step(scale_log2)
        out["q_scale"], out["k_scale"], out["v_scale"] = (FP8_SCALES[x] for x in "qkv")
        # real operand = scale * code: codes carry q / q_scale and k / k_scale
        q8 = torch.from_numpy(q / FP8_SCALES["q"]).to(torch.float8_e4m3fn)
        k8 = torch.from_numpy(k / FP8_SCALES["k"]).to(torch.float8_e4m3fn)
        assert torch.equal(q8.double() * FP8_SCALES["q"], torch.from_numpy(q))
        assert torch.equal(k8.double() * FP8_SCALES["k"], torch.from_numpy(k))
        v8 = vv.clamp(-448, 448).to(torch.float8_e4m3fn)
        out.update(q8=q8, k8=k8, v8=v8, vt8=v8.transpose(2, 3).contiguous())
    return out


def ramp_case(B, Hq, Hkv, Nq, Nk, D, causal, *, kind="bf16", seed=0):
    """Inputs of the ramp construction (module docstring)."""
    R = THRESHOLD[kind]
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Hq, Nq, D), generator=g)
    k = torch.randn((B, Hkv, Nk, D), generator=g)
    v = torch.randn((B, Hkv, Nk, D), generator=g)
    q[..., 0] = 2.0 + 2.0 * torch.rand((B, Hq, Nq), generator=g)
    scale = 1.0 / math.sqrt(D)
    # rise per tile for the smallest weight 2: 1.5 R (plus noise)
    step = 1.5 * R / (2.0 * scale * 1.4426950408889634)
    if kind == "fp8":
        step /= FP8_SCALES["q"] * FP8_SCALES["k"]
    tiles = torch.arange(Nk) // TILE
    k[..., 0] = (tiles.to(torch.float32) * step).expand(B, Hkv, Nk)
    out = {"kind": kind, "R": R, "scale": scale}
    if kind == "bf16":
        out.update(q=q.to(torch.bfloat16), k=k.to(torch.bfloat16), v=v.to(torch.bfloat16))
        out["scale_log2"] = float(np.float32(np.float32(scale) * LOG2E_F32))
    else:
        out["q_scale"], out["k_scale"], out["v_scale"] = (FP8_SCALES[x] for x in "qkv")
        q8 = (q / FP8_SCALES["q"]).clamp(-448, 448).to(torch.float8_e4m3fn)
        k8 = (k / FP8_SCALES["k"]).clamp(-448, 448).to(torch.float8_e4m3fn)
        v8 = v.clamp(-448, 448).to(torch.float8_e4m3fn)
        out.update(q8=q8, k8=k8, v8=v8, vt8=v8.transpose(2, 3).contiguous())
        s = np.float32(np.float32(np.float32(scale) * np.float32(FP8_SCALES["q"])) *
                       np.float32(FP8_SCALES["k"]))
        out["scale_log2"] = float(np.float32(s * LOG2E_F32))
    return out


def make_case(construction, kind, shape, seed=1):
    """One of the three constructions for ``shape`` = (B, Hq, Hkv, Nq, Nk, D,
    causal): "exact" (levels, rises R + 18, R, R + 1), "near" (quarter-unit
    levels, rises R - 1/4, R + 1/4, R + 1/4) or "ramp"."""
    if construction == "exact":
        return level_case(*shape, kind=kind, seed=seed)
    if construction == "near":
        R = THRESHOLD[kind]
        return level_case(*shape, kind=kind, quantum=0.25, rises=(R - 0.25, R + 0.25, R + 0.25),
                          seed=seed)
    if construction == "ramp":
        return ramp_case(*shape, kind=kind, seed=seed)
    raise ValueError(construction)


def log2_scores(case, B, Hq, Hkv, Nq, Nk, D):
    """u [B*Hq*Nq, Nk] fp64: the scores in log2 units as the kernel forms
    them (fp32 scale_log2 times the exact dot products of the inputs)."""
    if case["kind"] == "bf16":
        q, k = case["q"].double(), case["k"].double()
    else:
        q, k = case["q8"].double(), case["k8"].double()
    G = Hq // Hkv
    kk = k.repeat_interleave(G, dim=1)                   # [B, Hq, Nk, D]
    s = torch.matmul(q, kk.transpose(2, 3))              # [B, Hq, Nq, Nk]
    return (s * case["scale_log2"]).reshape(B * Hq * Nq, Nk).numpy()


def replay_rescale(u, Nq, Nk, causal, R):
    """The kernel's rescale rule per (row, key tile).  Returns (fires,
    active, top): fires[r, t] when tile t moves row r's running max,
    active[r, t] when the row sees a key of tile t, and top[r] the largest
    u - m over the row's visible keys after each tile's decision (the
    exponent of the row's largest weight, before the P bias)."""
    rows = u.shape[0]
    n_tiles = math.ceil(Nk / TILE)
    i = np.arange(rows) % Nq
    vis = np.minimum(i + 1, Nk) if causal else np.full(rows, Nk)
    fires = np.zeros((rows, n_tiles), dtype=bool)
    active = np.zeros((rows, n_tiles), dtype=bool)
    m = np.full(rows, -np.inf)
    top = np.full(rows, -np.inf)
    for t in range(n_tiles):
        lo, hi = t * TILE, min(Nk, (t + 1) * TILE)
        seg = u[:, lo:hi].copy()
        seg[np.arange(lo, hi)[None, :] >= vis[:, None]] = -np.inf
        mt = seg.max(axis=1)
        act = np.isfinite(mt)
        with np.errstate(invalid="ignore"):
            fire = act & (~np.isfinite(m) | (mt > m + R))
        m = np.where(fire, mt, m)
        top = np.maximum(top, np.where(act, mt - m, -np.inf))
        fires[:, t] = fire
        active[:, t] = act
    return fires, active, top


def fire_fraction(fires, active):
    """Share of (row, tile >= 1) pairs with a visible key where the rescale fires."""
    f, a = fires[:, 1:], active[:, 1:]
    return float(f[a].mean()) if a.any() else 0.0
