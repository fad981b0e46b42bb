"""GPU parity of the decode path (up to 64 tokens per call) against the oracle.

At these sizes engram_forward hashes and gathers in one kernel, streams the weight over every SM
in a second (64-row units, a fixed share per SM) and gates in a third. The cases cover what
decode adds to the prefill tests: windows that reach into caches of different lengths per
sequence (0, 1, 2 and more than max_ngram - 1 entries, so the pad, the cache and this call's
tokens all feed windows), several tokens of one sequence in one call, token counts that are not
multiples of 32 (zero rows in the MMA's N), a non-zero pad id, given hash ids, the cache append,
masks, and the device error bits.
"""
import numpy as np
import pytest
import torch

import deepseek_v4_engram_gb300 as eg
import synth
from oracle import engram as E
from tests.helpers import (assert_gate_close, assert_kv_close, assert_out_close, dev, empty_bf16,
                           host)

pytestmark = pytest.mark.gpu

WIDE = synth.Geometry(dim=5120, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=64,
                      vocab=129280, n_compressed=100000, prime_floor=1 << 14)


@pytest.fixture(scope="module")
def wide():
    from tests.gpu_fixtures import DeviceModel
    return DeviceModel(synth.make_model(WIDE, synth.BASE_SEED + 31, scale_mode="pow2", pad_id=7))


def prefilled(dm, lens, cap, seed):
    """Device cache and oracle state holding the same compressed ids: sequence b has lens[b]."""
    t, g = dm.model.tables, dm.geom
    B = len(lens)
    st = E.NgramHashState(t.token_map, t.pad_id, t.multipliers, t.primes, t.offsets, g.n_heads,
                          g.max_ngram_size, B)
    rng = np.random.default_rng(seed)
    cache = np.zeros((B, cap), dtype=np.int32)
    for b, n in enumerate(lens):
        c = np.asarray(t.token_map)[rng.integers(0, g.vocab, n)]
        cache[b, :n] = c
        st.cache[b] = c.astype(np.int64)
    return st, dev(cache), dev(np.asarray(lens, dtype=np.int32))


def run_step(dm, batch, cache, length, mask=None):
    B, T = batch.tokens.shape
    g = dm.geom
    out = empty_bf16(B, T, g.hc_mult, g.dim)
    ids = torch.full((B, T, g.n_hash_cols), -1, dtype=torch.int32, device="cuda")
    gate = torch.full((B, T, g.hc_mult), float("nan"), device="cuda")
    kv = empty_bf16(B, T, g.N)
    eg.engram_forward(dm.desc, dm.tables, dm.weights, dev(batch.x), dev(batch.tokens), cache,
                      length, None if mask is None else dev(mask), out, dm.workspace(B * T),
                      hash_ids_out=ids, gate_out=gate, kv_out=kv)
    return dict(out=host(out), ids=host(ids), gate=host(gate), kv=host(kv))


def check_stagewise(dm, batch, r, ref_ids, mask=None):
    m, g = dm.model, dm.geom
    B, T = batch.tokens.shape
    M = B * T
    np.testing.assert_array_equal(r["ids"], ref_ids)
    rows = E.embed_rows(m.table, m.scales, ref_ids).reshape(M, -1)
    kv = r["kv"].reshape(M, -1)
    assert_kv_close(kv, E.linear_bf16(rows, m.wkv), rows, m.wkv)
    x = batch.x.reshape(M, g.hc_mult, g.dim)
    mk = None if mask is None else mask.reshape(M)
    o2, g2 = E.gate_and_add(x, kv, m.q, m.k, mk, m.eps)
    assert_gate_close(r["gate"].reshape(M, -1), g2)
    assert_out_close(r["out"].reshape(M, g.hc_mult, g.dim), o2, kv[:, g.hc_mult * g.dim:])
    if mk is not None:
        np.testing.assert_array_equal(r["out"].reshape(M, g.hc_mult, g.dim)[~mk], x[~mk])
        assert (r["gate"].reshape(M, -1)[~mk] == 0).all()


@pytest.mark.parametrize("lens,T", [
    ([0], 1), ([5], 1), ([0, 1, 2, 3, 9], 3), ([2, 40], 32), ([1] * 31, 1), ([3] * 32, 1),
    ([0] * 33, 1), ([17], 64), ([11] * 64, 1), ([0, 2], 8)])
def test_decode_step_matches_oracle(wide, lens, T):
    B = len(lens)
    cap = max(lens) + T + 3
    st, cache, length = prefilled(wide, lens, cap, 1000 + B * 7 + T)
    batch = synth.make_batch(wide.geom, B, T, synth.BASE_SEED + 1100 + B + T,
                             x_dist="student_t3")
    mask = None
    if B * T > 4:
        mask = np.random.default_rng(B + T).random((B, T)) > 0.2
    r = run_step(wide, batch, cache, length, mask)
    assert eg.engram_check_errors() == 0
    ref_ids = st.push(batch.tokens)
    check_stagewise(wide, batch, r, ref_ids, mask)
    # the cache grew by this call's compressed ids, and every length by T
    np.testing.assert_array_equal(host(length), np.asarray(lens) + T)
    got = host(cache)
    for b in range(B):
        np.testing.assert_array_equal(got[b, :lens[b] + T], st.cache[b])


@pytest.mark.parametrize("B,T", [(1, 1), (7, 3), (64, 1)])
def test_decode_step_from_given_ids_is_bit_identical(wide, B, T):
    # engram_forward_ids runs the same kernel with the ids given instead of hashed
    st, cache, length = prefilled(wide, [4] * B, 4 + T, 77 + B)
    batch = synth.make_batch(wide.geom, B, T, synth.BASE_SEED + 1200 + B)
    r = run_step(wide, batch, cache, length)
    g, M = wide.geom, B * T
    out = empty_bf16(M, g.hc_mult, g.dim)
    gate = torch.full((M, g.hc_mult), float("nan"), device="cuda")
    kv = empty_bf16(M, g.N)
    eg.engram_forward_ids(wide.desc, wide.weights, dev(batch.x.reshape(M, g.hc_mult, g.dim)),
                          dev(r["ids"].reshape(M, -1)), None, out, wide.workspace(M),
                          gate_out=gate, kv_out=kv)
    assert eg.engram_check_errors() == 0
    np.testing.assert_array_equal(host(out), r["out"].reshape(M, g.hc_mult, g.dim))
    np.testing.assert_array_equal(host(gate), r["gate"].reshape(M, -1))
    np.testing.assert_array_equal(host(kv), r["kv"].reshape(M, -1))
    check_stagewise(wide, batch, r, st.push(batch.tokens))


def test_decode_step_consecutive_steps_equal_one_prefill(wide):
    # eight decode steps of 16 sequences, each reading the cache the previous one appended to
    B, T = 16, 8
    batch = synth.make_batch(wide.geom, B, T, synth.BASE_SEED + 1300)
    st, cache, length = prefilled(wide, [0] * B, T, 5)
    ids = []
    for t in range(T):
        step = synth.Batch(batch.tokens[:, t:t + 1], batch.x[:, t:t + 1], None)
        r = run_step(wide, step, cache, length)
        check_stagewise(wide, step, r, st.push(step.tokens))
        ids.append(r["ids"])
    assert eg.engram_check_errors() == 0
    whole = E.NgramHashState(wide.model.tables.token_map, wide.model.tables.pad_id,
                             wide.model.tables.multipliers, wide.model.tables.primes,
                             wide.model.tables.offsets, wide.geom.n_heads,
                             wide.geom.max_ngram_size, B)
    np.testing.assert_array_equal(np.concatenate(ids, 1), whole.push(batch.tokens))


def test_decode_step_error_bits(wide):
    g = wide.geom
    # a token outside the vocabulary is flagged
    st, cache, length = prefilled(wide, [3, 3], 8, 9)
    batch = synth.make_batch(g, 2, 1, synth.BASE_SEED + 1400)
    bad = synth.Batch(batch.tokens.copy(), batch.x, None)
    bad.tokens[1, 0] = g.vocab
    run_step(wide, bad, cache, length)
    assert eg.engram_check_errors() & 1
    # a full cache is flagged (capacity 3, length 3)
    st, cache, length = prefilled(wide, [3], 3, 10)
    run_step(wide, synth.make_batch(g, 1, 1, synth.BASE_SEED + 1401), cache, length)
    assert eg.engram_check_errors() & 2
