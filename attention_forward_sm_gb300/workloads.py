"""Seeded synthetic workloads for the attention forward and split-KV decode calls.

This module only draws random inputs and names the standard shapes; it holds
none of the attention arithmetic.  Tests feed the same tensors to the CUDA
library and to the CPU oracle, and the benchmark uses the same shapes.

Recipe: one ``torch.Generator`` per workload seeded with ``20260000 + index``;
Q, K and V are drawn in that order as ``randn * sigma`` in fp32 and rounded to
bf16 (round-to-nearest-even, torch's conversion).  The pages measure on
synthetic random tensors of shape (batch, heads, seq, head_dim)
("FlashAttention-3 vs Triton Kernels", the benchmark listing and the
"Empirical Production Benchmarks" sweep), so no dataset stands behind them.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int          # 1-based position in the standard list; seed = 20260000 + index
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    D: int
    causal: bool
    sigma: float = 1.0
    decode: bool = False
    nsplit: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def seed(self) -> int:
        return 20260000 + self.index

    def flops(self) -> float:
        """4*B*Hq*Nq*Nk*D (QK^T and PV, 2 flops per MAC), halved when causal."""
        f = 4.0 * self.B * self.Hq * self.Nq * self.Nk * self.D
        return f / 2.0 if self.causal else f

    def decode_bytes(self) -> int:
        """Algorithmic bytes of one decode call: the K and V caches once, q in,
        o out (bf16) and lse out (fp32).  Split-state scratch is excluded."""
        kv = 2 * self.B * self.Hkv * self.Nk * self.D * 2
        qo = 2 * self.B * self.Hq * self.D * 2
        return kv + qo + self.B * self.Hq * 4

    def prefill_bytes(self) -> int:
        """Compulsory bytes of one prefill call: Q, K, V read, O written (bf16),
        LSE written (fp32)."""
        q = self.B * self.Hq * self.Nq * self.D * 2
        kv = 2 * self.B * self.Hkv * self.Nk * self.D * 2
        return 2 * q + kv + self.B * self.Hq * self.Nq * 4

    def label(self) -> str:
        if self.decode:
            return (f"decode B{self.B} Hq{self.Hq} Hkv{self.Hkv} Nk{self.Nk} D{self.D} "
                    f"nsplit{self.nsplit}")
        return (f"{'causal' if self.causal else 'non-causal'} B{self.B} Hq{self.Hq} Hkv{self.Hkv} "
                f"Nq{self.Nq} Nk{self.Nk} D{self.D}")


WORKLOADS = {
    "tiny": Workload("tiny", 1, B=1, Hq=2, Hkv=2, Nq=256, Nk=256, D=64, causal=False),
    "prefill": Workload("prefill", 2, B=8, Hq=32, Hkv=32, Nq=8192, Nk=8192, D=128, causal=False),
    "causal": Workload("causal", 3, B=4, Hq=16, Hkv=16, Nq=16384, Nk=16384, D=128, causal=True),
    "long_gqa": Workload("long_gqa", 4, B=1, Hq=32, Hkv=8, Nq=131072, Nk=131072, D=128,
                         causal=True, sigma=0.5),
    "decode": Workload("decode", 5, B=8, Hq=32, Hkv=8, Nq=1, Nk=65536, D=128, causal=False,
                       decode=True, nsplit=32),
}


def custom(B, Hq, Hkv, Nq, Nk, D, causal=False, sigma=1.0, seed_index=100, decode=False,
           nsplit=0) -> Workload:
    """A workload of any shape (used by the parity sweeps)."""
    return Workload("custom", seed_index, B=B, Hq=Hq, Hkv=Hkv, Nq=Nq, Nk=Nk, D=D, causal=causal,
                    sigma=sigma, decode=decode, nsplit=nsplit)


def _draw(gen, shape, sigma, device):
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(torch.bfloat16)


def make_inputs(w: Workload, device="cpu"):
    """(q, k, v) bf16 tensors for workload ``w`` drawn on ``device``.

    Prefill: q [B,Hq,Nq,D], k/v [B,Hkv,Nk,D].  Decode: q [B,Hq,D] and the
    contiguous caches [B,Hkv,Nk,D].  The generator lives on ``device`` so a
    multi-GB workload never passes through host memory; the same seed on the
    same device type gives the same bits."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    qshape = (w.B, w.Hq, w.D) if w.decode else (w.B, w.Hq, w.Nq, w.D)
    kvshape = (w.B, w.Hkv, w.Nk, w.D)
    q = _draw(gen, qshape, w.sigma, device)
    k = _draw(gen, kvshape, w.sigma, device)
    v = _draw(gen, kvshape, w.sigma, device)
    return q, k, v


# Per-tensor dequantisation scales of the FP8 inputs (arbitrary, not 1, so
# that a dropped or swapped scale shows).
FP8_SCALES = {"q": 0.5, "k": 1.25, "v": 0.75}


def make_inputs_fp8(w: Workload, device="cpu"):
    """(q8, k8, v8, vt8) E4M3 code tensors (torch.float8_e4m3fn) for a prefill
    workload ``w``: ``randn * sigma`` in fp32, clamped to the largest finite
    E4M3 value 448, rounded to E4M3 by torch's conversion; Q, K, V drawn in
    that order from the workload's seed + 50000.  vt8 = V transposed to
    [B, Hkv, D, Nk] (keys fastest), the layout attn_fwd_fp8 reads; v8 is
    [B, Hkv, Nk, D]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed + 50000)

    def draw(shape):
        x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
        if w.sigma != 1.0:
            x.mul_(w.sigma)
        return x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)

    q8 = draw((w.B, w.Hq, w.Nq, w.D))
    k8 = draw((w.B, w.Hkv, w.Nk, w.D))
    v8 = draw((w.B, w.Hkv, w.Nk, w.D))
    vt8 = v8.transpose(2, 3).contiguous()
    return q8, k8, v8, vt8


def sample_rows(w: Workload, n: int, seed: int = 7) -> torch.Tensor:
    """Flat query-row indices ``(b*Hq + h)*Nq + i`` to check on a large
    workload: ``n`` uniform draws from a fixed seed, plus row 0 and row
    Nq-1 of the first and last head, plus (causal) the first and last row of
    every 128-row tile of one head.  Sorted, unique, int64."""
    g = torch.Generator().manual_seed(seed)
    total = w.B * w.Hq * w.Nq
    picks = torch.randint(0, total, (n,), generator=g, dtype=torch.int64)
    extra = [0, w.Nq - 1, total - w.Nq, total - 1]
    if w.causal:
        bh = (w.B * w.Hq) // 2
        for t0 in range(0, w.Nq, 128):
            extra += [bh * w.Nq + t0, bh * w.Nq + min(t0 + 127, w.Nq - 1)]
    rows = torch.cat([picks, torch.tensor(extra, dtype=torch.int64)])
    return torch.unique(rows)
