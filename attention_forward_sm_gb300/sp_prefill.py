"""Sequence-parallel prefill across ranks (SP AllGather attention).

The sequence is cut into contiguous rank blocks (``sp_decode.shard_range``:
the first N % world ranks get one position more).  Rank r holds its block of
the queries and of the keys and values; it all-gathers the key and value
blocks of every rank, so it has the whole K and V, and attends its own query
rows to them.  With the causal mask a row's visibility depends on its global
position, so the local call is ``attn_fwd_rows`` with the block's first row
as ``q_offset``; every rank computes its rows' final O and LSE, and no
further exchange is needed (smzdm digest, section 5, on Triton-distributed's
SP AllGather attention).  The exchanged volume per rank is its K and V
block, 2 * B * Hkv * N_r * D bf16 values.

The gather is ``torch.distributed.all_gather`` on blocks padded to the
largest block (ranks' blocks differ by at most one position); the padding is
cut off before the blocks are joined.  ``local_attn`` may be passed
explicitly (the multi-rank CPU tests pass the oracle's); by default it is
the library call, with no fallback.
"""
from __future__ import annotations

import torch

from .sp_decode import shard_range


def _library_local_attn(q_block, k_full, v_full, causal, q_offset, scale):
    from . import binding as attn
    B, Hq, n, D = q_block.shape
    Hkv, Nk = k_full.shape[1], k_full.shape[2]
    o = torch.empty_like(q_block)
    lse = torch.empty((B, Hq, n), dtype=torch.float32, device=q_block.device)
    attn.attn_fwd_rows(q_block, k_full, v_full, o, lse, B, Hq, Hkv, n, Nk, D, causal, q_offset,
                       scale)
    return o, lse


def gather_blocks(block: torch.Tensor, N: int, group=None) -> torch.Tensor:
    """All-gather every rank's block [B, H, N_r, D] of a length-N sequence
    into the whole [B, H, N, D] (blocks as ``shard_range`` cuts them)."""
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    if world == 1:
        return block.contiguous()
    rank = dist.get_rank(group)
    width = shard_range(N, world, 0)[1]  # the largest block
    s0, s1 = shard_range(N, world, rank)
    if block.shape[2] != s1 - s0:
        raise ValueError("block length does not match this rank's shard")
    B, H, _, D = block.shape
    padded = block.new_zeros((B, H, width, D))
    padded[:, :, : s1 - s0] = block
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded, group=group)
    pieces = []
    for r in range(world):
        a, b = shard_range(N, world, r)
        pieces.append(parts[r][:, :, : b - a])
    return torch.cat(pieces, dim=2).contiguous()


def sp_prefill(q_block, k_block, v_block, N: int, causal: bool, scale: float, group=None, *,
               local_attn=None):
    """Attention of this rank's query rows to the whole sequence.

    q_block [B, Hq, N_r, D] and k_block / v_block [B, Hkv, N_r, D] are the
    rank's blocks of a length-N sequence (``shard_range(N, world, rank)``).
    Returns O [B, Hq, N_r, D] and LSE [B, Hq, N_r] of those rows, equal to the
    rows of single-GPU attention over the whole sequence."""
    import torch.distributed as dist
    local_attn = local_attn or _library_local_attn
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if world > 1 else 0
    s0, _ = shard_range(N, world, rank)
    k_full = gather_blocks(k_block, N, group)
    v_full = gather_blocks(v_block, N, group)
    if q_block.shape[2] == 0:  # a rank with no rows only lends its (empty) keys
        B, Hq, _, D = q_block.shape
        return (q_block.new_empty((B, Hq, 0, D)),
                torch.empty((B, Hq, 0), dtype=torch.float32, device=q_block.device))
    return local_attn(q_block, k_full, v_full, causal, s0, scale)
