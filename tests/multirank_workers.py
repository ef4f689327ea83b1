"""Worker functions for the multi-rank CPU tests (run in spawned processes,
one per rank, over the gloo backend on 127.0.0.1)."""
import math
import os

import numpy as np
import torch
import torch.distributed as dist


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def max_over_ranks_worker(rank, world, port):
    _init(rank, world, port)
    import bench
    got = bench.max_over_ranks(float(10 * rank + 3), world)
    assert got == float(10 * (world - 1) + 3), got
    dist.destroy_process_group()


def sp_decode_worker(rank, world, port, B, Hq, Hkv, Nk, D, seed):
    """Each rank decodes its key shard with the oracle, the states are
    all-gathered over gloo and recombined (oracle combine); every rank checks
    the result against the oracle over the whole cache."""
    _init(rank, world, port)
    import oracle
    from attention_forward_sm_gb300 import sp_decode
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Nk, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Nk, D, generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    s0, s1 = sp_decode.shard_range(Nk, world, rank)
    ks, vs = k[:, :, s0:s1].contiguous(), v[:, :, s0:s1].contiguous()

    def local_states(q_, k_, v_, nsplit):
        o, l = oracle.attn_rows(q_, k_, v_, B, Hq, Hkv, 1, k_.shape[2], D, False, scale)
        return torch.from_numpy(o).float(), torch.from_numpy(l).float()

    def combine(part_o, part_lse):
        o, l = oracle.combine(part_o.double().numpy(), part_lse.double().numpy())
        return o, l

    o, lse = sp_decode.sp_flash_decode(q, ks, vs, 8, local_states=local_states, combine=combine)
    o_ref, lse_ref = oracle.decode(q, k, v, B, Hq, Hkv, Nk, D, scale=scale)
    assert np.abs(o - o_ref).max() < 1e-5, np.abs(o - o_ref).max()
    assert np.abs(lse - lse_ref).max() < 1e-5
    # the naive sum of the per-rank outputs is not attention (denominator pitfall)
    dist.destroy_process_group()


def sp_decode_failure_worker(rank, world, port, fail_rank, results, stall_s=0.0):
    """The sequence-parallel decode with one rank that fails before the state
    exchange -- at once, or after stalling `stall_s` seconds without joining
    the collective: the others must leave the all-gather with an error within
    the process group's short timeout (reported through `results`), not
    hang."""
    import datetime
    import time
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=5))
    import oracle
    from attention_forward_sm_gb300 import sp_decode
    B, Hq, Hkv, Nk, D = 1, 4, 2, 64, 16
    g = torch.Generator().manual_seed(7)
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Nk, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Nk, D, generator=g).to(torch.bfloat16)
    s0, s1 = sp_decode.shard_range(Nk, world, rank)
    ks, vs = k[:, :, s0:s1].contiguous(), v[:, :, s0:s1].contiguous()
    scale = 1.0 / math.sqrt(D)

    def local_states(q_, k_, v_, nsplit):
        if rank == fail_rank:
            time.sleep(stall_s)
            raise RuntimeError("injected failure on the host before the exchange")
        o, l = oracle.attn_rows(q_, k_, v_, B, Hq, Hkv, 1, k_.shape[2], D, False, scale)
        return torch.from_numpy(o).float(), torch.from_numpy(l).float()

    def combine(part_o, part_lse):
        return oracle.combine(part_o.double().numpy(), part_lse.double().numpy())

    t0 = time.monotonic()
    code = 0
    try:
        sp_decode.sp_flash_decode(q, ks, vs, 4, local_states=local_states, combine=combine)
        results.put((rank, "completed", time.monotonic() - t0))
    except Exception as e:  # noqa: BLE001 - any error is the detection we want
        results.put((rank, type(e).__name__, time.monotonic() - t0))
        if rank == fail_rank:
            code = 3  # the failing rank dies without a clean shutdown
    # flush the report before the hard exit (the queue's writer is a thread)
    results.close()
    results.join_thread()
    os._exit(code)


def sp_prefill_worker(rank, world, port, B, Hq, Hkv, N, D, causal, seed):
    """Each rank holds its block of Q, K and V, all-gathers K and V over gloo
    and attends its rows with the global row offset (oracle as the local
    attention); every rank checks its rows against the oracle over the whole
    sequence."""
    _init(rank, world, port)
    import oracle
    from attention_forward_sm_gb300 import sp_decode, sp_prefill
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, N, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, N, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, N, D, generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    s0, s1 = sp_decode.shard_range(N, world, rank)
    qb, kb, vb = (t[:, :, s0:s1].contiguous() for t in (q, k, v))

    def local_attn(q_blk, k_full, v_full, causal_, q0, scale_):
        # the oracle has no row offset: put the block behind q0 zero rows
        n = q_blk.shape[2]
        qpad = torch.cat([torch.zeros(B, Hq, q0, D, dtype=q_blk.dtype), q_blk], dim=2)
        rows = [(b * Hq + h) * (q0 + n) + q0 + i for b in range(B) for h in range(Hq)
                for i in range(n)]
        o, l = oracle.attn_rows(qpad, k_full, v_full, B, Hq, Hkv, q0 + n, N, D, causal_,
                                scale_, rows=rows)
        return torch.from_numpy(o).reshape(B, Hq, n, D), torch.from_numpy(l).reshape(B, Hq, n)

    o, lse = sp_prefill.sp_prefill(qb, kb, vb, N, causal, scale, local_attn=local_attn)
    assert o.shape == (B, Hq, s1 - s0, D)
    rows = [(b * Hq + h) * N + i for b in range(B) for h in range(Hq) for i in range(s0, s1)]
    if rows:
        o_ref, lse_ref = oracle.attn_rows(q, k, v, B, Hq, Hkv, N, N, D, causal, scale, rows=rows)
        assert np.abs(o.reshape(-1, D).numpy() - o_ref).max() < 1e-12
        assert np.abs(lse.reshape(-1).numpy() - lse_ref).max() < 1e-12
    dist.destroy_process_group()
