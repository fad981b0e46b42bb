"""GPU parity of engram_hash_rows_layers: stages 1 + 2 for several Engram layers in one launch.

Each layer's hash ids and rows must equal, bit for bit, the oracle's push_layers (one shared
look-back cache, each layer's own constants) followed by its embed_rows on that layer's table;
the cache and its lengths must equal a single engram_hash call's.
"""
import numpy as np
import pytest
import torch

import deepseek_v4_engram_gb300 as eg
import synth
from oracle import engram as E
from tests.helpers import dev, empty_bf16, host

pytestmark = pytest.mark.gpu

FULLISH = synth.Geometry(dim=5120, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=64,
                         vocab=129280, n_compressed=100000, prime_floor=1 << 14)


class Layers:
    """A model's shared token map plus n_layers layers' constants and tables, host and device."""

    def __init__(self, geom, n_layers, seed, pad_id=0):
        self.geom = geom
        self.tables = synth.make_tables(geom, np.random.default_rng(seed), pad_id=pad_id)
        self.layers = synth.make_layer_hashes(geom, n_layers, seed + 1)
        t = self.tables
        self.desc = eg.make_desc(geom.dim, geom.hc_mult, geom.n_heads, geom.max_ngram_size,
                                 geom.head_dim, t.num_embeddings)
        self.dtables = eg.DeviceTables(dev(t.token_map), t.pad_id, dev(t.multipliers),
                                       dev(t.primes), dev(t.offsets))
        self.dev = [dict(multipliers=dev(lh.multipliers), primes=dev(lh.primes),
                         offsets=dev(lh.offsets), table=dev(lh.table), scales=dev(lh.scales))
                    for lh in self.layers]

    def run(self, tokens, cache, length, with_ids=True, table_rows=None):
        """One engram_hash_rows_layers call; returns per-layer (ids, rows) on the host."""
        B, T = tokens.shape
        S, hd = self.geom.n_hash_cols, self.geom.head_dim
        recs = []
        for i, d in enumerate(self.dev):
            table, scales = d["table"], d["scales"]
            if table_rows is not None and table_rows[i] is not None:
                table, scales = table[:table_rows[i]], scales[:table_rows[i]]
            recs.append(eg.DeviceLayerHash(
                d["multipliers"], d["primes"], d["offsets"], table, scales,
                empty_bf16(B * T, S * hd),
                torch.full((B * T, S), -7, dtype=torch.int32, device="cuda") if with_ids else None))
        eg.engram_hash_rows_layers(self.desc, self.dtables, recs, dev(tokens), cache, length)
        return [(None if r.hash_ids is None else host(r.hash_ids), host(r.rows)) for r in recs]

    def oracle_state(self, B):
        t = self.tables
        return E.NgramHashState(t.token_map, t.pad_id, t.multipliers, t.primes, t.offsets,
                                self.geom.n_heads, self.geom.max_ngram_size, B)

    def consts(self):
        return [(lh.multipliers, lh.primes, lh.offsets) for lh in self.layers]


def new_cache(B, cap):
    return (torch.zeros((B, cap), dtype=torch.int32, device="cuda"),
            torch.zeros(B, dtype=torch.int32, device="cuda"))


def check_layers(L, got, ref_ids, B, T):
    S, hd = L.geom.n_hash_cols, L.geom.head_dim
    for i, ((ids, rows), lh) in enumerate(zip(got, L.layers)):
        if ids is not None:
            np.testing.assert_array_equal(ids.reshape(B, T, S), ref_ids[i], err_msg=f"layer {i}")
        ref_rows = E.embed_rows(lh.table, lh.scales, ref_ids[i])          # [B, T, S, hd]
        np.testing.assert_array_equal(rows.reshape(B, T, S, hd), ref_rows,
                                      err_msg=f"layer {i} rows")


@pytest.mark.parametrize("n_layers,B,T", [(1, 3, 37), (2, 3, 37), (3, 2, 129), (16, 2, 21)])
def test_layers_match_oracle_tiny(n_layers, B, T):
    # 16 layers: 384 (layer, slot) items per position, more than a block's threads
    L = Layers(synth.TINY, n_layers, synth.BASE_SEED + 300 + n_layers, pad_id=11)
    rng = np.random.default_rng(n_layers * 100 + T)
    tokens = rng.integers(0, L.geom.vocab, (B, T + 2), dtype=np.int32)
    cache, length = new_cache(B, T + 2)
    st = L.oracle_state(B)
    # a prefill of T positions, then two single-token decode steps looking back into it
    for a, b in ((0, T), (T, T + 1), (T + 1, T + 2)):
        got = L.run(tokens[:, a:b], cache, length)
        assert eg.engram_check_errors() == 0
        check_layers(L, got, st.push_layers(tokens[:, a:b], L.consts()), B, b - a)
        np.testing.assert_array_equal(host(length), [b] * B)
    np.testing.assert_array_equal(host(cache), L.tables.token_map[tokens])


def test_layers_full_width_and_optional_ids():
    L = Layers(FULLISH, 4, synth.BASE_SEED + 400)
    B, T = 2, 301   # ragged over the block's positions (2 per block at 4 x 24 items)
    tokens = np.random.default_rng(401).integers(0, L.geom.vocab, (B, T + 1), dtype=np.int32)
    cache, length = new_cache(B, T + 1)
    st = L.oracle_state(B)
    got = L.run(tokens[:, :T], cache, length, with_ids=False)
    assert eg.engram_check_errors() == 0
    check_layers(L, got, st.push_layers(tokens[:, :T], L.consts()), B, T)
    got = L.run(tokens[:, T:], cache, length)
    assert eg.engram_check_errors() == 0
    check_layers(L, got, st.push_layers(tokens[:, T:], L.consts()), B, 1)


def test_layers_agree_with_single_layer_calls():
    # each layer's ids equal engram_hash run with that layer's constants on its own cache copy
    L = Layers(synth.TINY, 3, synth.BASE_SEED + 500)
    B, T = 4, 50
    tokens = dev(np.random.default_rng(501).integers(0, L.geom.vocab, (B, T), dtype=np.int32))
    cache, length = new_cache(B, T)
    got = L.run(host(tokens), cache, length)
    for i, d in enumerate(L.dev):
        tab = eg.DeviceTables(L.dtables.token_map, L.tables.pad_id, d["multipliers"],
                              d["primes"], d["offsets"])
        c2, l2 = new_cache(B, T)
        ids = torch.empty((B, T, L.geom.n_hash_cols), dtype=torch.int32, device="cuda")
        eg.engram_hash(L.desc, tab, tokens, c2, l2, ids)
        np.testing.assert_array_equal(host(ids).reshape(B * T, -1), got[i][0])
        np.testing.assert_array_equal(host(c2), host(cache))
    assert eg.engram_check_errors() == 0


def test_layer_out_of_range_rows_flag_and_zero():
    # layer 1 gets a table cut below its largest ids: those rows are zero and the error bit is
    # set; layer 0 is untouched
    L = Layers(synth.TINY, 2, synth.BASE_SEED + 600)
    B, T = 1, 64
    tokens = np.random.default_rng(601).integers(0, L.geom.vocab, (B, T), dtype=np.int32)
    cache, length = new_cache(B, T)
    cut = int(L.layers[1].offsets[12])   # ids of slots 12.. are out of range
    got = L.run(tokens, cache, length, table_rows=[None, cut])
    assert eg.engram_check_errors() & 4
    ref = L.oracle_state(B).push_layers(tokens, L.consts())
    S, hd = L.geom.n_hash_cols, L.geom.head_dim
    np.testing.assert_array_equal(got[0][1].reshape(B, T, S, hd),
                                  E.embed_rows(L.layers[0].table, L.layers[0].scales, ref[0]))
    rows1 = got[1][1].reshape(B, T, S, hd)
    assert (rows1[:, :, 12:] == 0).all()
    np.testing.assert_array_equal(rows1[:, :, :12], E.embed_rows(
        L.layers[1].table, L.layers[1].scales, ref[1][:, :, :12]))


def test_layers_empty_is_noop():
    L = Layers(synth.TINY, 2, synth.BASE_SEED + 700)
    cache, length = new_cache(2, 4)
    got = L.run(np.zeros((2, 0), dtype=np.int32), cache, length)
    assert eg.engram_check_errors() == 0
    assert all(r.size == 0 for _, r in got)
    np.testing.assert_array_equal(host(length), [0, 0])
