"""Pins for the oracle's n-gram hash (Module engram, stage 1 / NgramHashState).

No real hash tables or captures exist, so the hash is pinned to its stated structure: closed
forms under special multipliers, the unsigned 64-bit wrap, the pad window, the look-back cache
across calls, and which slots depend on which look-backs.
"""
import numpy as np
import pytest

import synth
from oracle.engram import NgramHashState

H, NMAX = 8, 4
S = (NMAX - 1) * H


def state(token_map, mults, primes, pad=0, batch=1):
    primes = np.asarray(primes, dtype=np.uint64)
    offsets = np.zeros(S, dtype=np.int64)
    offsets[1:] = np.cumsum(primes[:-1].astype(np.int64))
    return NgramHashState(token_map, pad, np.asarray(mults, dtype=np.uint64), primes, offsets,
                          H, NMAX, batch), offsets


def test_bit_packing_closed_form():
    # Multipliers 2^(12k) with ids < 2^12 put look-back k in bits [12k, 12k+12), so the XOR-roll is
    # the packed window sum_k c_{p-k} 2^(12k); moduli above 2^48 leave it untouched. This pins the
    # window order, the look-back/multiplier pairing, the pad, slot order and the offsets at once.
    rng = np.random.default_rng(0)
    V = 4096
    token_map = rng.permutation(V).astype(np.int64)
    pad = 0xABC
    mults = [1 << (12 * k) for k in range(NMAX)]
    primes = [(1 << 48) + 1000 * s + 7 for s in range(S)]
    st, offsets = state(token_map, mults, primes, pad=pad)
    tokens = rng.integers(0, V, size=(1, 37))
    ids = st.push(tokens)[0]
    c = token_map[tokens[0]]
    for p in range(37):
        for n in range(2, NMAX + 1):
            packed = sum((int(c[p - k]) if p - k >= 0 else pad) << (12 * k) for k in range(n))
            for head in range(H):
                s = (n - 2) * H + head
                assert ids[p, s] == packed + offsets[s]


def test_single_lookback_is_textbook_mod():
    # m_0 = 1 and m_k = 0 (k >= 1): every slot is c_p mod P_s + O_s.
    rng = np.random.default_rng(1)
    token_map = rng.integers(0, 1 << 20, size=500)
    primes = synth.consecutive_primes(1009, S)
    st, offsets = state(token_map, [1, 0, 0, 0], primes, pad=5)
    tokens = rng.integers(0, 500, size=(1, 50))
    ids = st.push(tokens)[0]
    c = token_map[tokens[0]]
    for s in range(S):
        np.testing.assert_array_equal(ids[:, s], c % primes[s] + offsets[s])


def test_multiply_wraps_modulo_2_64():
    # m_0 = 2^63 + 1, c = 3: 3 * m_0 = 2^64 + 2^63 + 3 -> 2^63 + 3 after the 64-bit wrap.
    P = 1000003
    st, offsets = state(np.array([3]), [(1 << 63) + 1, 0, 0, 0], [P] * S)
    ids = st.push(np.zeros((1, 1), dtype=np.int64))[0, 0]
    np.testing.assert_array_equal(ids - offsets, [((1 << 63) + 3) % P] * S)


def test_pad_only_before_sequence_start_and_prefix_invariance():
    # A prefix of tokens whose compressed id IS the pad id must not change the ids of later
    # positions that can see it (n-gram windows only see pads or pad-valued ids either way).
    rng = np.random.default_rng(2)
    V, pad = 300, 17
    token_map = rng.integers(0, 200, size=V)
    token_map[0] = pad
    mults = rng.integers(0, 2 ** 63, size=NMAX).astype(np.uint64) * 2 + 1
    primes = synth.consecutive_primes(1009, S)
    tokens = rng.integers(1, V, size=(1, 20))
    a, _ = state(token_map, mults, primes, pad=pad)
    b, _ = state(token_map, mults, primes, pad=pad)
    ids_a = a.push(tokens)[0]
    ids_b = b.push(np.concatenate([np.zeros((1, NMAX - 1), dtype=np.int64), tokens], 1))[0]
    np.testing.assert_array_equal(ids_a, ids_b[NMAX - 1:])


def test_ids_in_slot_range():
    model = synth.make_model(synth.TINY, 11)
    t = model.tables
    st = NgramHashState(t.token_map, t.pad_id, t.multipliers, t.primes, t.offsets, H, NMAX, 2)
    ids = st.push(np.random.default_rng(3).integers(0, synth.TINY.vocab, size=(2, 300)))
    lo = t.offsets[None, None, :]
    hi = lo + t.primes.astype(np.int64)[None, None, :]
    assert ((ids >= lo) & (ids < hi)).all()


def test_cache_carries_lookback_across_calls():
    # prefill(T) == prefill(T - j) followed by j single-token decode steps, bit for bit.
    model = synth.make_model(synth.TINY, 12)
    t = model.tables
    tokens = np.random.default_rng(4).integers(0, synth.TINY.vocab, size=(3, 40))
    whole = NgramHashState(t.token_map, 9, t.multipliers, t.primes, t.offsets, H, NMAX, 3)
    ref = whole.push(tokens)
    for split in (0, 1, 2, 3, 39):
        st = NgramHashState(t.token_map, 9, t.multipliers, t.primes, t.offsets, H, NMAX, 3)
        parts = [st.push(tokens[:, :split])]
        for j in range(split, 40):
            parts.append(st.push(tokens[:, j:j + 1]))
        np.testing.assert_array_equal(np.concatenate(parts, 1), ref)


def test_sequences_are_independent():
    model = synth.make_model(synth.TINY, 13)
    t = model.tables
    tokens = np.random.default_rng(5).integers(0, synth.TINY.vocab, size=(4, 25))
    both = NgramHashState(t.token_map, 0, t.multipliers, t.primes, t.offsets, H, NMAX, 4)
    ids = both.push(tokens)
    for b in range(4):
        one = NgramHashState(t.token_map, 0, t.multipliers, t.primes, t.offsets, H, NMAX, 1)
        np.testing.assert_array_equal(one.push(tokens[b:b + 1])[0], ids[b])


def test_slot_dependence_on_lookbacks():
    # 2-gram slots (0..7) see c_p, c_{p-1}; 3-gram slots (8..15) add c_{p-2}; 4-gram slots add c_{p-3}.
    model = synth.make_model(synth.TINY, 14)
    t = model.tables
    base = np.array([[5, 6, 7, 8, 9]])

    def ids(tok):
        st = NgramHashState(t.token_map, 0, t.multipliers, t.primes, t.offsets, H, NMAX, 1)
        return st.push(tok)[0, -1]

    def with_token(i, v):
        b = base.copy()
        b[0, i] = v
        return b

    # pick replacements whose compressed id differs from the original
    tm = t.token_map
    alt = lambda i: next(v for v in range(1000) if tm[v] != tm[base[0, i]])
    r0 = ids(base)
    r_p3 = ids(with_token(1, alt(1)))   # changes c_{p-3}
    r_p2 = ids(with_token(2, alt(2)))   # changes c_{p-2}
    r_p1 = ids(with_token(3, alt(3)))   # changes c_{p-1}
    np.testing.assert_array_equal(r_p3[:16], r0[:16])
    assert (r_p3[16:] != r0[16:]).sum() >= 6
    np.testing.assert_array_equal(r_p2[:8], r0[:8])
    assert (r_p2[8:] != r0[8:]).sum() >= 12
    assert (r_p1 != r0).sum() >= 18


def test_brute_force_every_window_of_a_tiny_vocabulary():
    # Every window over 5 compressed ids, at every distance from the sequence start (so with 0
    # to 3 pad look-backs), against the formula evaluated in Python integers: for n = 2..4,
    # mix_n = XOR over k < n of (c_{p-k} * m_k mod 2^64), id = mix_n mod P_s + O_s. Generic odd
    # 64-bit multipliers exercise the wrap and the unsigned modulo on every slot.
    import itertools
    rng = np.random.default_rng(6)
    V, pad = 5, 3
    token_map = np.array([4, 0, 2, 1, 3], dtype=np.int64)   # a permutation: tokens != ids
    mults = [int(v) * 2 + 1 for v in rng.integers(0, 2 ** 63, size=NMAX, dtype=np.int64)]
    primes = synth.consecutive_primes(1009, S)
    offsets = [0] + list(np.cumsum([int(p) for p in primes[:-1]]))
    checked = 0
    for length in range(1, NMAX + 1):          # the last position p = length - 1
        for toks in itertools.product(range(V), repeat=length):
            st, _ = state(token_map, np.array(mults, dtype=np.uint64), primes, pad=pad)
            got = st.push(np.array([toks], dtype=np.int64))[0, -1]
            c = [int(token_map[t]) for t in toks]
            p = length - 1
            for n in range(2, NMAX + 1):
                mix = 0
                for k in range(n):
                    ck = c[p - k] if p - k >= 0 else pad
                    mix ^= (ck * mults[k]) % (1 << 64)
                for head in range(H):
                    s = (n - 2) * H + head
                    assert int(got[s]) == mix % int(primes[s]) + int(offsets[s]), (toks, s)
            checked += 1
    assert checked == sum(V ** L for L in range(1, NMAX + 1))
