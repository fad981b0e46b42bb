"""GPU parity of each stage entry point against the oracle (hash, rows, wkv, gate and add)."""
import numpy as np
import pytest
import torch

import deepseek_v4_engram_gb300 as eg
import synth
from oracle import engram as E
from oracle.numerics import bf16_to_f64
from tests.helpers import (assert_gate_close, assert_kv_close, assert_out_close, dev, empty_bf16,
                           host)

pytestmark = pytest.mark.gpu

FULLISH = synth.Geometry(dim=5120, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=64,
                         vocab=129280, n_compressed=100000, prime_floor=1 << 14)


@pytest.fixture(scope="module")
def tiny():
    from tests.gpu_fixtures import DeviceModel
    return DeviceModel(synth.make_model(synth.TINY, synth.BASE_SEED))


@pytest.fixture(scope="module")
def wide():
    # full-width geometry with a smaller table (primes from 2^14): same kernels, faster setup
    from tests.gpu_fixtures import DeviceModel
    return DeviceModel(synth.make_model(FULLISH, synth.BASE_SEED + 7, scale_mode="pow2"))


def oracle_state(dm, B, pad=None):
    t = dm.model.tables
    return E.NgramHashState(t.token_map, t.pad_id if pad is None else pad, t.multipliers,
                            t.primes, t.offsets, dm.geom.n_heads, dm.geom.max_ngram_size, B)


# ------------------------------------------------------------------------------------- hash


@pytest.mark.parametrize("B,T", [(1, 1), (1, 16), (3, 17), (2, 129), (5, 300)])
def test_hash_matches_oracle(tiny, B, T):
    tokens = np.random.default_rng(B * 1000 + T).integers(0, tiny.geom.vocab, (B, T), dtype=np.int32)
    cache, length = tiny.new_cache(B, T + 8)
    ids = torch.full((B, T, 24), -1, dtype=torch.int32, device="cuda")
    eg.engram_hash(tiny.desc, tiny.tables, dev(tokens), cache, length, ids)
    assert eg.engram_check_errors() == 0
    ref = oracle_state(tiny, B).push(tokens)
    np.testing.assert_array_equal(host(ids), ref)
    np.testing.assert_array_equal(host(length), [T] * B)
    np.testing.assert_array_equal(host(cache)[:, :T], tiny.model.tables.token_map[tokens])


def test_hash_lookback_spans_calls(wide):
    # prefill 2048 positions, then single-token decode steps that must look back into it
    B, P, steps = 8, 2048, 5
    rng = np.random.default_rng(21)
    tokens = rng.integers(0, wide.geom.vocab, (B, P + steps), dtype=np.int32)
    cache, length = wide.new_cache(B, P + steps)
    ids = torch.empty((B, P, 24), dtype=torch.int32, device="cuda")
    eg.engram_hash(wide.desc, wide.tables, dev(tokens[:, :P]), cache, length, ids)
    st = oracle_state(wide, B)
    np.testing.assert_array_equal(host(ids), st.push(tokens[:, :P]))
    for j in range(steps):
        step_ids = torch.empty((B, 1, 24), dtype=torch.int32, device="cuda")
        eg.engram_hash(wide.desc, wide.tables, dev(tokens[:, P + j:P + j + 1]), cache, length,
                       step_ids)
        np.testing.assert_array_equal(host(step_ids), st.push(tokens[:, P + j:P + j + 1]))
    assert eg.engram_check_errors() == 0
    np.testing.assert_array_equal(host(length), [P + steps] * B)


def test_hash_nonzero_pad_and_ragged_prefix_lengths(tiny):
    # sequences enter with different cache lengths (0, 1, 2, 5); pad id 9
    B = 4
    pre = [0, 1, 2, 5]
    rng = np.random.default_rng(22)
    tables = eg.DeviceTables(tiny.tables.token_map, 9, tiny.tables.multipliers,
                             tiny.tables.primes, tiny.tables.offsets)
    st = oracle_state(tiny, B, pad=9)
    cache, length = tiny.new_cache(B, 64)
    # fill prefixes one sequence at a time through the oracle and mirror them into the cache
    for b, n in enumerate(pre):
        toks = rng.integers(0, tiny.geom.vocab, (1, n), dtype=np.int32)
        one = E.NgramHashState(st.token_map, 9, st.multipliers, st.primes, st.offsets, 8, 4, 1)
        one.push(toks)
        st.cache[b] = one.cache[0]
        cache[b, :n] = torch.from_numpy(one.cache[0].astype(np.int32))
    length.copy_(torch.tensor(pre, dtype=torch.int32))
    tokens = rng.integers(0, tiny.geom.vocab, (B, 7), dtype=np.int32)
    ids = torch.empty((B, 7, 24), dtype=torch.int32, device="cuda")
    eg.engram_hash(tiny.desc, tables, dev(tokens), cache, length, ids)
    np.testing.assert_array_equal(host(ids), st.push(tokens))


def test_hash_device_errors(tiny):
    cache, length = tiny.new_cache(1, 4)
    ids = torch.empty((1, 6, 24), dtype=torch.int32, device="cuda")
    tokens = np.array([[1, 2, 3, 4, 5, 6]], dtype=np.int32)
    eg.engram_hash(tiny.desc, tiny.tables, dev(tokens), cache, length, ids)
    assert eg.engram_check_errors() & 2          # cache full
    assert eg.engram_check_errors() == 0         # cleared by the read
    cache, length = tiny.new_cache(1, 16)
    bad = np.array([[1, 5000, 3]], dtype=np.int32)
    ids = torch.empty((1, 3, 24), dtype=torch.int32, device="cuda")
    eg.engram_hash(tiny.desc, tiny.tables, dev(bad), cache, length, ids)
    assert eg.engram_check_errors() & 1          # token outside the vocabulary


def test_hash_empty_is_noop(tiny):
    cache, length = tiny.new_cache(2, 8)
    ids = torch.empty((2, 0, 24), dtype=torch.int32, device="cuda")
    eg.engram_hash(tiny.desc, tiny.tables, torch.empty((2, 0), dtype=torch.int32, device="cuda"),
                   cache, length, ids)
    assert eg.engram_check_errors() == 0
    np.testing.assert_array_equal(host(length), [0, 0])


# ------------------------------------------------------------------------------- table rows


@pytest.mark.parametrize("n", [1, 17, 129, 4096 * 24])
def test_rows_bit_exact(wide, n):
    rng = np.random.default_rng(n)
    ids = rng.integers(0, wide.model.tables.num_embeddings, n, dtype=np.int32)
    out = empty_bf16(n, 64)
    eg.engram_embed_rows(wide.desc, wide.weights.table, wide.weights.scales, dev(ids), out)
    assert eg.engram_check_errors() == 0
    np.testing.assert_array_equal(host(out), E.embed_rows(wide.model.table, wide.model.scales, ids))


def test_rows_every_code_and_scale():
    # all 256 e4m3 codes against scales 2^-4..2^4 (NaN codes compared as NaN)
    codes = np.tile(np.arange(256, dtype=np.uint8), (9, 1)).reshape(9 * 8, 32)
    codes = np.concatenate([codes, codes], 1)                      # head_dim 64
    scales = np.repeat((127 + np.arange(-4, 5)).astype(np.uint8), 8)[:, None].repeat(2, 1)
    desc = eg.make_desc(256, 4, 8, 4, 64, codes.shape[0], 1e-6)
    ids = np.arange(codes.shape[0], dtype=np.int32)
    out = empty_bf16(len(ids), 64)
    eg.engram_embed_rows(desc, dev(codes), dev(scales), dev(ids), out)
    got = bf16_to_f64(host(out))
    ref = bf16_to_f64(E.embed_rows(codes, scales, ids))
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_rows_out_of_range_id_flags_and_zeroes(tiny):
    ids = np.array([0, tiny.model.tables.num_embeddings, -1, 5], dtype=np.int32)
    out = empty_bf16(4, 32)
    eg.engram_embed_rows(tiny.desc, tiny.weights.table, tiny.weights.scales, dev(ids), out)
    assert eg.engram_check_errors() & 4
    o = host(out)
    assert (o[1] == 0).all() and (o[2] == 0).all()
    np.testing.assert_array_equal(o[[0, 3]], E.embed_rows(tiny.model.table, tiny.model.scales,
                                                          ids[[0, 3]]))


# -------------------------------------------------------------------------------- projection


@pytest.mark.parametrize("M", [1, 16, 17, 129, 300])
def test_wkv_tiny_within_one_ulp(tiny, M):
    rng = np.random.default_rng(M)
    a = synth.f32_to_bf16_bits(rng.standard_normal((M, 768)).astype(np.float32))
    kv = empty_bf16(M, 1280)
    eg.engram_wkv(dev(a), tiny.weights.wkv, kv)
    torch.cuda.synchronize()
    assert_kv_close(host(kv), E.linear_bf16(a, tiny.model.wkv), a, tiny.model.wkv)


@pytest.mark.parametrize("M", [1, 33, 64, 200, 513])
def test_wkv_full_width_within_one_ulp(wide, M):
    rng = np.random.default_rng(M + 1)
    ids = rng.integers(0, wide.model.tables.num_embeddings, (M, 24))
    a = E.embed_rows(wide.model.table, wide.model.scales, ids).reshape(M, -1)
    kv = empty_bf16(M, 25600)
    eg.engram_wkv(dev(a), wide.weights.wkv, kv)
    torch.cuda.synchronize()
    assert_kv_close(host(kv), E.linear_bf16(a, wide.model.wkv), a, wide.model.wkv)


# ---------------------------------------------------------------------------- gate and add


@pytest.mark.parametrize("M,masked", [(1, False), (37, True), (300, True)])
def test_gate_and_add_matches_oracle(wide, M, masked):
    rng = np.random.default_rng(M + 3)
    g = wide.geom
    x = synth.make_x((M, g.hc_mult, g.dim), rng, "student_t3")
    kv = synth.f32_to_bf16_bits(rng.standard_normal((M, g.N)).astype(np.float32))
    mask = (rng.random(M) > 0.3) if masked else None
    out = empty_bf16(M, g.hc_mult, g.dim)
    gate = torch.full((M, g.hc_mult), float("nan"), device="cuda")
    eg.engram_gate_and_add(wide.desc, dev(x), dev(kv), wide.weights.q_weight,
                           wide.weights.k_weight, None if mask is None else dev(mask), out, gate)
    torch.cuda.synchronize()
    ref_out, ref_gate = E.gate_and_add(x, kv, wide.model.q, wide.model.k, mask, wide.model.eps)
    assert_gate_close(host(gate), ref_gate)
    assert_out_close(host(out), ref_out, kv[:, g.hc_mult * g.dim:])
    if mask is not None:
        np.testing.assert_array_equal(host(out)[~mask], x[~mask])


def test_gate_zero_key_and_tiny(tiny):
    M, g = 16, tiny.geom
    rng = np.random.default_rng(5)
    x = synth.make_x((M, g.hc_mult, g.dim), rng)
    kv = synth.f32_to_bf16_bits(rng.standard_normal((M, g.N)).astype(np.float32))
    kv[:4, : g.hc_mult * g.dim] = 0                        # key = 0 -> gate = sigmoid(1e-3)
    out = empty_bf16(M, g.hc_mult, g.dim)
    gate = torch.empty((M, g.hc_mult), device="cuda")
    eg.engram_gate_and_add(tiny.desc, dev(x), dev(kv), tiny.weights.q_weight,
                           tiny.weights.k_weight, None, out, gate)
    torch.cuda.synchronize()
    ref_out, ref_gate = E.gate_and_add(x, kv, tiny.model.q, tiny.model.k, None, tiny.model.eps)
    np.testing.assert_allclose(host(gate)[:4], 1 / (1 + np.exp(-1e-3)), atol=1e-6)
    assert_gate_close(host(gate), ref_gate)
    assert_out_close(host(out), ref_out, kv[:, g.hc_mult * g.dim:])


@pytest.mark.parametrize("nbytes", [16, 48 * 1024 + 16, 78643200])
def test_stream_probe_reads_without_error(nbytes):
    # the measurement call: every share of the buffer read, every wait completed in time
    buf = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda").fill_(7)
    for method in (0, 1, 2):
        eg.api.engram_probe_stream_read(buf, method)
    torch.cuda.synchronize()
    assert eg.engram_check_errors() == 0
