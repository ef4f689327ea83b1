"""Multi-rank host logic on CPU ranks (gloo, world size 2 and 3): the
benchmark's max-over-ranks timing reduction and the sequence-parallel decode
(key shards, [D+1] state exchange, LSE recombination)."""
import socket

import pytest
import torch
import torch.multiprocessing as mp

import multirank_workers as W
from attention_forward_sm_gb300 import sp_decode


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("Nk,world", [(10, 3), (7, 7), (5, 8), (65536, 8), (1, 2), (100, 1)])
def test_shard_range_partitions_the_keys(Nk, world):
    spans = [sp_decode.shard_range(Nk, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == Nk
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in spans]
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0


def test_pack_unpack_roundtrip():
    o = torch.randn(6, 16)
    lse = torch.randn(6)
    gathered = torch.stack([sp_decode.pack_state(o + r, lse - r) for r in range(3)])
    part_o, part_lse = sp_decode.unpack_states(gathered)
    assert part_o.shape == (6, 3, 16) and part_lse.shape == (6, 3)
    for r in range(3):
        assert torch.equal(part_o[:, r], o + r) and torch.equal(part_lse[:, r], lse - r)


def test_bench_max_over_ranks_gloo():
    mp.spawn(W.max_over_ranks_worker, args=(2, _free_port()), nprocs=2, join=True)


@pytest.mark.parametrize("world,Nk", [(2, 300), (3, 1000), (3, 2)])
def test_sp_flash_decode_gloo(world, Nk):
    mp.spawn(W.sp_decode_worker, args=(world, _free_port(), 2, 8, 2, Nk, 16, 5 + world),
             nprocs=world, join=True)


@pytest.mark.parametrize("world,N,causal", [(2, 300, True), (3, 200, True), (3, 130, False),
                                            (4, 3, True)])
def test_sp_prefill_gloo(world, N, causal):
    """Sequence-parallel prefill on gloo ranks: K/V blocks all-gathered (ranks'
    blocks differ in length; N = 3 on 4 ranks leaves one rank empty), each
    rank's rows attended with their global offset, equal to the oracle over
    the whole sequence."""
    mp.spawn(W.sp_prefill_worker, args=(world, _free_port(), 1, 4, 2, N, 16, causal, 40 + world),
             nprocs=world, join=True)


@pytest.mark.parametrize("world,fail_rank,stall_s", [(2, 1, 0.0), (3, 0, 0.0), (3, 2, 0.0),
                                                     (2, 0, 12.0)])
def test_sp_decode_rank_failure_is_detected(world, fail_rank, stall_s):
    """A rank raises before the state exchange and exits -- at once, or after
    stalling past the process group's 5 s timeout without joining the
    all-gather; every other rank gets an error out of the all-gather
    instead of hanging (a dead peer within ~20 ms, a stalled one at the
    timeout), and no rank reports a result."""
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=W.sp_decode_failure_worker,
                         args=(r, world, port, fail_rank, results, stall_s))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=60)
    alive = [p for p in procs if p.is_alive()]
    for p in alive:
        p.kill()
    assert not alive, "a rank hung after a peer failed"
    got = {}
    while len(got) < world:
        r, what, dt = results.get(timeout=10)
        got[r] = (what, dt)
    assert got[fail_rank][0] == "RuntimeError"
    for r in range(world):
        assert got[r][0] != "completed", got
        assert got[r][1] < 30.0, got
        if r != fail_rank and stall_s > 0:
            assert got[r][1] < stall_s, got  # released by the timeout, not by the exit
    assert procs[fail_rank].exitcode == 3
