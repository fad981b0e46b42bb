"""Row-sharded table, host side (CPU; gloo, world size 2): which rank holds which rows, and the
exchange that completes a sharded gather.

Each rank holds the rows deepseek_v4_engram_gb300.table_shard_range gives it and writes, for a
gather of ids, its own rows and bf16 -0.0 for the others (the contract of
engram_embed_rows_shard, restated here on the CPU from the oracle's gather). One all-reduce
(exchange_rows) must then give every rank the unsharded gather bit for bit, signed zeros included.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from deepseek_v4_engram_gb300.shard import exchange_rows, row_owner, table_shard_range

NEG_ZERO = np.uint16(0x8000)


@pytest.mark.parametrize("n,W", [(10, 3), (12587554, 2), (12587554, 8), (5, 8), (1, 1), (7, 7)])
def test_shard_ranges_tile_the_table_and_agree_with_row_owner(n, W):
    ranges = [table_shard_range(n, W, r) for r in range(W)]
    assert ranges[0][0] == 0
    for (b0, c0), (b1, _) in zip(ranges, ranges[1:]):
        assert b0 + c0 == b1                                   # contiguous, in rank order
    assert sum(c for _, c in ranges) == n
    assert max(c for _, c in ranges) - min(c for _, c in ranges) <= 1
    # row_owner inverts the split: every boundary row and a sample of the rest
    ids = np.unique(np.concatenate([[b for b, c in ranges if c], [b + c - 1 for b, c in ranges if c],
                                    np.random.default_rng(n).integers(0, n, 1000)]))
    want = np.array([next(r for r, (b, c) in enumerate(ranges) if b <= i < b + c) for i in ids])
    np.testing.assert_array_equal(row_owner(ids, n, W), want)


def test_shard_range_rejects_bad_arguments():
    for args in [(10, 0, 0), (10, 2, 2), (10, 2, -1), (-1, 2, 0)]:
        with pytest.raises(ValueError):
            table_shard_range(*args)
    with pytest.raises(ValueError):
        row_owner([10], 10, 2)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _partial_rows(table, scales, ids, rank, world):
    """This rank's share of a gather, as engram_embed_rows_shard writes it."""
    from oracle import engram as E
    rows = E.embed_rows(table, scales, ids)
    own = row_owner(ids, table.shape[0], world) == rank
    return np.where(own[:, None], rows, NEG_ZERO).astype(np.uint16)


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import synth
        model = synth.make_model(synth.TINY, synth.BASE_SEED + 31)
        n = model.table.shape[0]
        rng = np.random.default_rng(77)          # the same ids on every rank (replicated hash)
        bounds = [table_shard_range(n, world, r)[0] for r in range(1, world)]
        ids = np.concatenate([rng.integers(0, n, 500), bounds, [b - 1 for b in bounds], [0, n - 1]])
        part = _partial_rows(model.table, model.scales, ids.astype(np.int32), rank, world)
        out = torch.from_numpy(part.view(np.int16).copy()).view(torch.bfloat16)
        exchange_rows(out)
        q.put((rank, "ok", ids, out.view(torch.int16).numpy().view(np.uint16)))
    except Exception as e:  # report to the parent instead of hanging it
        q.put((rank, "error", repr(e), None))
        raise
    finally:
        dist.destroy_process_group()


def test_two_ranks_exchange_gives_the_unsharded_gather():
    import synth
    from oracle import engram as E
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        got = dict((r, (s, i, o)) for r, s, i, o in (q.get(timeout=240) for _ in range(world)))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(got[r][0] == "ok" for r in range(world)), got
    model = synth.make_model(synth.TINY, synth.BASE_SEED + 31)
    ids = got[0][1]
    want = E.embed_rows(model.table, model.scales, ids.astype(np.int32))
    for r in range(world):
        np.testing.assert_array_equal(got[r][2], want)
    assert (want == NEG_ZERO).any()          # -0 rows elements survive the exchange
    assert all(p.exitcode == 0 for p in procs)
