"""The multi-GPU plumbing of bench.py on the CPU: two gloo ranks (replicas,
no data-path collective) agree on the slowest rank's time, each computes the
same seeded workload independently, and the reference arm runs on rank 0
only."""
import os
import socket
import time
import types

import numpy as np
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from draft_token_markov_gb300 import workloads as W
        env = bench._dist()
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank)
        # replicas: every rank runs its own copy of the same seeded call
        w = W.TINY
        head, embed = W.make_weights(w)
        inp = W.make_call(w)
        toks, cache = oracle.chain(oracle.bf16_bits(inp["base"]), oracle.bf16_bits(head),
                                   oracle.bf16_bits(embed), inp["anchor"].numpy(),
                                   inp["temperature"].numpy(), inp["seeds"].numpy(),
                                   inp["row_state_idx"].numpy(), w.mode, nthreads=1)
        digest = int(np.bitwise_xor.reduce(cache.astype(np.uint64).ravel() * 2654435761 % (1 << 32)))
        got = [None] * world
        dist.all_gather_object(got, (toks.tolist(), digest))
        # the reference arm: ranks other than 0 return at once, printing nothing
        t0 = time.perf_counter()
        if rank != 0:
            bench.run_reference(types.SimpleNamespace(steps=1, warmup=0))
        ref_s = time.perf_counter() - t0
        dist.barrier()
        q.put((rank, env, slowest, got, ref_s))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    for _ in procs:
        rank, env, slowest, got, ref_s = q.get(timeout=240)
        results[rank] = (env, slowest, got, ref_s)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (env, slowest, got, ref_s) in results.items():
        assert env == (2, rank, rank)
        assert slowest == 15.0
        assert got[0] == got[1]
        if rank != 0:
            assert ref_s < 1.0


def _shard_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from draft_token_markov_gb300 import api
        V = 129280
        off, width = api.shard_range(rank, world, V)
        ok = api.agree_on_shards(None, V, off, width)
        # a rank that holds another rank's shard: every rank learns it
        bad = api.agree_on_shards(None, V, off if rank == 0 else off - 16, width)
        q.put((rank, off, width, ok, bad))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_vocab_shards():
    # the host side of the vocabulary-sharded chain on a future multi-GPU
    # box: each rank's shard is rows [k V / world, (k + 1) V / world) of the
    # head, and the ranks check together that each holds its own
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r[1], r[2]) for r in res] == [(0, 64640), (64640, 64640)]
    assert all(r[3] for r in res) and not any(r[4] for r in res)
