"""GPU: stage 2 over a row-sharded table (engram_embed_rows_shard), one GPU standing in for every
rank in turn. Each rank's output holds its own rows as engram_embed_rows writes them and bf16 -0.0
elsewhere; the bf16 sum of all ranks' outputs is the unsharded gather bit for bit."""
import numpy as np
import pytest
import torch

import deepseek_v4_engram_gb300 as eg
import synth
from deepseek_v4_engram_gb300 import _lib
from deepseek_v4_engram_gb300.shard import row_owner, table_shard_range
from oracle import engram as E
from tests.helpers import dev, empty_bf16, host

pytestmark = pytest.mark.gpu

NEG_ZERO = 0x8000


@pytest.fixture(scope="module")
def table():
    rng = np.random.default_rng(synth.BASE_SEED + 41)
    n, hd = 100003, 64
    codes = synth.make_fp8_rows(n, hd, rng)
    scales = synth.make_scales(n, hd, rng, "pow2")
    desc = eg.make_desc(256, 4, 8, 4, hd, n, 1e-6)
    return desc, codes, scales, dev(codes), dev(scales)


def shard_ids(n, W, rng, count=20000):
    cuts = [table_shard_range(n, W, r)[0] for r in range(1, W)]
    return np.concatenate([rng.integers(0, n, count), cuts, [c - 1 for c in cuts], [0, n - 1]]
                          ).astype(np.int32)


@pytest.mark.parametrize("W", [2, 3, 8])
def test_shards_sum_to_the_unsharded_gather(table, W):
    desc, codes, scales, tab, sc = table
    n, hd = codes.shape
    ids = shard_ids(n, W, np.random.default_rng(W))
    want = E.embed_rows(codes, scales, ids)
    assert (want == NEG_ZERO).any()              # e4m3 -0 codes are in the sample
    ids_d = dev(ids)
    owner = row_owner(ids, n, W)
    total = None
    for r in range(W):
        b, c = table_shard_range(n, W, r)
        out = empty_bf16(len(ids), hd)
        eg.engram_embed_rows_shard(desc, tab[b:b + c], sc[b:b + c], b, ids_d, out)
        assert eg.engram_check_errors() == 0
        got = host(out)
        own = owner == r
        np.testing.assert_array_equal(got[own], want[own])
        assert (got[~own] == NEG_ZERO).all()
        bf = out.view(torch.bfloat16)
        total = bf.clone() if total is None else total + bf      # bf16 adds, rank order
    np.testing.assert_array_equal(host(total.view(torch.int16)), want)
    # and against the library's own unsharded gather
    full = empty_bf16(len(ids), hd)
    eg.engram_embed_rows(desc, tab, sc, ids_d, full)
    np.testing.assert_array_equal(host(full), want)


def test_rank_without_rows_and_out_of_range_ids(table):
    desc, codes, scales, tab, sc = table
    n, hd = codes.shape
    ids = np.array([0, 5, n - 1, n, -3], dtype=np.int32)
    out = empty_bf16(len(ids), hd)
    eg.engram_embed_rows_shard(desc, None, None, n, dev(ids), out)     # no rows: an empty shard
    assert eg.engram_check_errors() & 4                                 # ids n and -3
    o = host(out)
    assert (o[:3] == NEG_ZERO).all() and (o[3:] == 0).all()
    out = empty_bf16(len(ids), hd)
    eg.engram_embed_rows_shard(desc, tab[:10], sc[:10], 0, dev(ids), out)
    assert eg.engram_check_errors() & 4
    o = host(out)
    np.testing.assert_array_equal(o[:2], E.embed_rows(codes, scales, ids[:2]))
    assert (o[2] == NEG_ZERO).all() and (o[3:] == 0).all()


def test_shard_outside_the_table_is_rejected(table):
    desc, codes, scales, tab, sc = table
    n, hd = codes.shape
    ids = dev(np.zeros(4, dtype=np.int32))
    out = empty_bf16(4, hd)
    for begin, rows in [(-1, 10), (n - 5, 10)]:
        with pytest.raises(eg.EngramError) as e:
            eg.engram_embed_rows_shard(desc, tab[:rows], sc[:rows], begin, ids, out)
        assert e.value.code == _lib.ENGRAM_EINVAL


def test_embed_rows_sharded_on_one_rank_is_the_gather(table):
    # world size 1 (no process group): the whole table is this rank's shard, no exchange
    desc, codes, scales, tab, sc = table
    ids = shard_ids(codes.shape[0], 1, np.random.default_rng(5), 3000)
    out = empty_bf16(len(ids), codes.shape[1])
    eg.embed_rows_sharded(desc, tab, sc, 0, dev(ids), out)
    assert eg.engram_check_errors() == 0
    np.testing.assert_array_equal(host(out), E.embed_rows(codes, scales, ids))
