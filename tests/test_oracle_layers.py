"""Pins for the oracle's hash over several Engram layers (NgramHashState.push_layers).

Each Engram layer takes its own entry of the hash layout (Engram listing, __init__:
layer_hash_index, and an embedding of that entry's num_embeddings rows), so each layer hashes the
same windows with its own multipliers, primes and offsets; the compressed ids depend only on the
tokens, so one look-back cache serves all layers. These tests pin that structure: a closed form per
layer under bit-packing multipliers (a layer given another layer's constants, or a window taken
from the wrong cache position, fails it), equality with one independent single-layer state per
layer across prefill and decode calls, and a cache that grows once per call.
"""
import numpy as np

import synth
from oracle.engram import NgramHashState

H, NMAX = 8, 4
S = (NMAX - 1) * H


def offsets_of(primes):
    o = np.zeros(S, dtype=np.int64)
    o[1:] = np.cumsum(np.asarray(primes, dtype=np.int64)[:-1])
    return o


def test_bit_packing_closed_form_per_layer():
    # Layer l uses multipliers 2^(12k + l): look-back k lands in bits [12k + l, 12k + l + 12), so
    # its window is packed and shifted by l; its moduli (> 2^50) leave the packed value untouched.
    rng = np.random.default_rng(21)
    V = 4096
    token_map = rng.permutation(V).astype(np.int64)
    pad = 0x5A5
    layers = []
    for layer in range(3):
        mults = np.array([1 << (12 * k + layer) for k in range(NMAX)], dtype=np.uint64)
        primes = np.array([(1 << 50) + 977 * s + 131 * layer + 1 for s in range(S)],
                          dtype=np.uint64)
        layers.append((mults, primes, offsets_of(primes)))
    st = NgramHashState(token_map, pad, layers[0][0], layers[0][1], layers[0][2], H, NMAX, 1)
    tokens = rng.integers(0, V, size=(1, 29))
    out = st.push_layers(tokens, layers)
    assert len(out) == 3
    c = token_map[tokens[0]]
    for layer, (_, _, offsets) in enumerate(layers):
        for p in range(29):
            for n in range(2, NMAX + 1):
                packed = sum((int(c[p - k]) if p - k >= 0 else pad) << (12 * k + layer)
                             for k in range(n))
                for head in range(H):
                    s = (n - 2) * H + head
                    assert out[layer][0, p, s] == packed + int(offsets[s])


def test_layers_equal_independent_states_across_calls():
    geom = synth.TINY
    model = synth.make_model(geom, 31)
    t = model.tables
    layers = synth.make_layer_hashes(geom, 4, 32, with_tables=False)
    consts = [(lh.multipliers, lh.primes, lh.offsets) for lh in layers]
    B = 3
    tokens = np.random.default_rng(33).integers(0, geom.vocab, size=(B, 30))
    shared = NgramHashState(t.token_map, 7, t.multipliers, t.primes, t.offsets, H, NMAX, B)
    own = [NgramHashState(t.token_map, 7, m, p, o, H, NMAX, B) for (m, p, o) in consts]
    # a prefill of 26 positions, then four single-token decode steps
    for a, b in ((0, 26), (26, 27), (27, 28), (28, 29), (29, 30)):
        got = shared.push_layers(tokens[:, a:b], consts)
        for layer in range(4):
            np.testing.assert_array_equal(got[layer], own[layer].push(tokens[:, a:b]))
        for bb in range(B):
            assert len(shared.cache[bb]) == b   # appended once per call, not once per layer
            np.testing.assert_array_equal(shared.cache[bb], own[0].cache[bb])


def test_one_layer_is_push_and_layers_differ():
    geom = synth.TINY
    t = synth.make_model(geom, 41).tables
    layers = synth.make_layer_hashes(geom, 2, 42, with_tables=False)
    tokens = np.random.default_rng(43).integers(0, geom.vocab, size=(2, 17))
    a = NgramHashState(t.token_map, 0, t.multipliers, t.primes, t.offsets, H, NMAX, 2)
    b = NgramHashState(t.token_map, 0, t.multipliers, t.primes, t.offsets, H, NMAX, 2)
    np.testing.assert_array_equal(
        a.push_layers(tokens, [(t.multipliers, t.primes, t.offsets)])[0], b.push(tokens))
    c = NgramHashState(t.token_map, 0, t.multipliers, t.primes, t.offsets, H, NMAX, 2)
    ids = c.push_layers(tokens, [(lh.multipliers, lh.primes, lh.offsets) for lh in layers])
    # each layer's ids fall in its own slot ranges, and the layers' tables have different sizes
    for lh, got in zip(layers, ids):
        assert (got >= lh.offsets[None, None]).all()
        assert (got < (lh.offsets + lh.primes.astype(np.int64))[None, None]).all()
    assert layers[0].num_embeddings != layers[1].num_embeddings
    assert not np.array_equal(ids[0], ids[1])
