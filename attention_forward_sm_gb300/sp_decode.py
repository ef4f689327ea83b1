"""Sequence-parallel split-KV decode across ranks (SP FlashDecode).

Each rank holds a contiguous shard of every (batch, kv head) K/V cache along
the key axis.  It decodes its shard into one state per (batch, q head): the
shard's softmax-normalised output and its log-sum-exp, D + 1 numbers.  The
ranks all-gather those states and recombine them through their lse weights
(L = ln sum_r exp(lse_r), O = sum_r exp(lse_r - L) O_r).  Adding the raw
per-shard outputs would be wrong, because every shard's softmax has its own
denominator; carrying lse_r fixes that, and the exchanged volume,
B * Hq * (D + 1) floats per rank, does not grow with the cache length (smzdm
digest, section 5, on Triton-distributed's SP FlashDecode).

The local decode and the combine run in the CUDA library
(``attn_decode_splitkv_states``, ``attn_combine_states``); the exchange is a
``torch.distributed`` all-gather.  ``local_states`` / ``combine`` may be
passed explicitly (the multi-rank CPU tests pass the oracle's); by default
they are the library calls, with no fallback.
"""
from __future__ import annotations

import math

import torch


def shard_range(Nk: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous key range [start, end) of `rank`: the first Nk % world ranks
    get one key more than the others."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world size")
    base, rem = divmod(Nk, world)
    start = rank * base + min(rank, rem)
    return start, start + base + (1 if rank < rem else 0)


def pack_state(o_state: torch.Tensor, lse: torch.Tensor) -> torch.Tensor:
    """[rows, D] fp32 output and [rows] fp32 lse -> one [rows, D + 1] buffer."""
    rows = lse.numel()
    return torch.cat([o_state.reshape(rows, -1).float(), lse.reshape(rows, 1).float()], dim=1)


def unpack_states(gathered: torch.Tensor):
    """[world, rows, D + 1] -> part_o [rows, world, D], part_lse [rows, world]
    (contiguous, the layout attn_combine_states reads)."""
    part_o = gathered[:, :, :-1].permute(1, 0, 2).contiguous()
    part_lse = gathered[:, :, -1].permute(1, 0).contiguous()
    return part_o, part_lse


def _library_local_states(q, k_shard, v_shard, nsplit):
    from . import binding as attn
    B, Hq, D = q.shape
    Hkv, nk = k_shard.shape[1], k_shard.shape[2]
    o_state = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    attn.attn_decode_splitkv_states(q, k_shard, v_shard, o_state, lse, B, Hq, Hkv, nk, D,
                                    max(1, min(nsplit, nk)))
    return o_state.reshape(B * Hq, D), lse.reshape(B * Hq)


def _library_combine(part_o, part_lse):
    from . import binding as attn
    rows, nparts, D = part_o.shape
    o = torch.empty((rows, D), dtype=torch.bfloat16, device=part_o.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=part_o.device)
    attn.attn_combine_states(part_o, part_lse, o, lse, rows, nparts, D)
    return o, lse


def sp_flash_decode(q, k_shard, v_shard, nsplit: int, group=None, *, local_states=None,
                    combine=None):
    """Decode q [B, Hq, D] against the full cache whose key shard this rank
    holds (k_shard / v_shard [B, Hkv, Nk_r, D], Nk_r may be 0).  Returns
    O [B*Hq, D] and LSE [B*Hq] of attention over all ranks' keys; every rank
    gets the same result."""
    import torch.distributed as dist
    local_states = local_states or _library_local_states
    combine = combine or _library_combine
    B, Hq, D = q.shape
    rows = B * Hq
    if k_shard.shape[2] > 0:
        o_state, lse = local_states(q, k_shard, v_shard, nsplit)
    else:  # an empty shard contributes nothing: weight exp(-inf) = 0
        o_state = torch.zeros((rows, D), dtype=torch.float32, device=q.device)
        lse = torch.full((rows,), -math.inf, dtype=torch.float32, device=q.device)
    state = pack_state(o_state, lse)
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    if world == 1:
        gathered = state.unsqueeze(0)
    else:
        parts = [torch.empty_like(state) for _ in range(world)]
        dist.all_gather(parts, state, group=group)
        gathered = torch.stack(parts)
    part_o, part_lse = unpack_states(gathered)
    return combine(part_o, part_lse)
