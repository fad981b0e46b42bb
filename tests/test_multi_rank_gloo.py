"""Multi-rank host logic on CPU (gloo, world size 2).

The path shards by sequence with no data-path collective: each rank runs its own sequences with
replicated tables and weights, and only the step time is reduced (max over ranks). These tests run
that host logic, in two processes, without a GPU:
  * bench.reduce_max returns the max over ranks;
  * bench.shard_seed gives each rank its own shard of sequences;
  * running the forward (the oracle stands in for the device path here) on per-rank shards gives
    exactly the result of one process running every sequence: nothing crosses ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import synth
        from oracle import engram as E

        # 1. timing reduction
        mx = bench.reduce_max(10.0 + 5.0 * rank)
        # 2. each rank's shard: its own sequences
        geom = synth.TINY
        model = synth.make_model(geom, synth.BASE_SEED)
        batch = synth.make_batch(geom, 2, 24, bench.shard_seed(synth.BASE_SEED + 100, rank))
        t = model.tables
        st = E.NgramHashState(t.token_map, t.pad_id, t.multipliers, t.primes, t.offsets,
                              geom.n_heads, geom.max_ngram_size, 2)
        r = E.forward(st, model.table, model.scales, model.wkv, model.q, model.k, batch.x,
                      batch.tokens, None, model.eps)
        # gather every rank's tokens and outputs on rank 0 (test plumbing only)
        toks = [torch.zeros(2, 24, dtype=torch.int64) for _ in range(world)]
        outs = [torch.zeros(r["out"].shape, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(toks, torch.from_numpy(batch.tokens.astype(np.int64)))
        dist.all_gather(outs, torch.from_numpy(r["out"].astype(np.int32)))
        if rank == 0:
            q.put(("ok", mx, [x.numpy() for x in toks], [o.numpy() for o in outs]))
    except Exception as e:  # report to the parent instead of hanging it
        q.put(("error", repr(e), None, None))
        raise
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_sequences_and_reduce_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        status, mx, toks, outs = q.get(timeout=240)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert status == "ok", mx
    assert mx == 15.0                                   # max over ranks
    assert not np.array_equal(toks[0], toks[1])         # disjoint shards of sequences
    # one process, every sequence at once: identical to the per-rank results
    import synth
    from oracle import engram as E
    geom = synth.TINY
    model = synth.make_model(geom, synth.BASE_SEED)
    t = model.tables
    xs = [synth.make_batch(geom, 2, 24, synth.BASE_SEED + 100 + 1000 * r).x for r in range(2)]
    st = E.NgramHashState(t.token_map, t.pad_id, t.multipliers, t.primes, t.offsets,
                          geom.n_heads, geom.max_ngram_size, 4)
    r = E.forward(st, model.table, model.scales, model.wkv, model.q, model.k,
                  np.concatenate(xs), np.concatenate(toks).astype(np.int32), None, model.eps)
    np.testing.assert_array_equal(r["out"].astype(np.int32), np.concatenate(outs))
    assert all(p.exitcode == 0 for p in procs)
