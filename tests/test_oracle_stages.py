"""Pins for the oracle's table rows, wkv projection, gate-and-add and whole forward."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import engram as E
from oracle.numerics import bf16_to_f64, bf16_ulp, e4m3_to_f64, f64_to_bf16


def bits(a):
    return f64_to_bf16(np.asarray(a, dtype=np.float64))


def sigmoid(z):
    return 1.0 / (1.0 + math.exp(-z))


# ------------------------------------------------------------------------------ table rows


def test_embed_rows_gathers_the_right_rows_unit_scale():
    rng = np.random.default_rng(0)
    table = rng.integers(0, 256, size=(1000, 64)).astype(np.uint8)
    table[(table & 0x7F) == 0x7F] = 0x11                     # no NaN codes
    scales = np.full((1000, 2), 127, dtype=np.uint8)
    ids = rng.integers(0, 1000, size=(7, 24))
    out = bf16_to_f64(E.embed_rows(table, scales, ids))
    np.testing.assert_array_equal(out, e4m3_to_f64(table[ids]))


def test_embed_rows_scale_applies_to_its_block_only():
    table = np.full((4, 64), 0x38, dtype=np.uint8)          # 1.0 everywhere
    scales = np.array([[127, 127], [130, 127], [127, 123], [131, 131]], dtype=np.uint8)
    out = bf16_to_f64(E.embed_rows(table, scales, np.arange(4)))
    want = np.ones((4, 64))
    want[1, :32] = 8.0
    want[2, 32:] = 1 / 16
    want[3, :] = 16.0
    np.testing.assert_array_equal(out, want)


# ------------------------------------------------------------------------------ projection


def test_linear_matches_torch_bf16_within_one_ulp():
    rng = np.random.default_rng(1)
    a = synth.f32_to_bf16_bits(rng.standard_normal((33, 768)).astype(np.float32))
    w = synth.make_wkv(synth.TINY, rng)
    ours = bf16_to_f64(E.linear_bf16(a, w))
    at = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    wt = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16)
    ref = torch.nn.functional.linear(at, wt).to(torch.float64).numpy()
    assert (np.abs(ours - ref) <= bf16_ulp(ref)).all()
    assert (ours == ref).mean() > 0.99


def test_linear_one_hot_rows_pick_weight_columns():
    rng = np.random.default_rng(2)
    w = synth.f32_to_bf16_bits(rng.standard_normal((50, 40)).astype(np.float32))
    a = bits(np.eye(40))
    np.testing.assert_array_equal(E.linear_bf16(a, w), w.T)


def test_linear_rounds_the_exact_sum_once():
    # 1 + 2^-8 + 2^-30: exact sum is just above a bf16 tie, so it rounds up to 1 + 2^-7
    a = bits([[1.0, 1.0, 1.0]])
    w = bits([[1.0, 2.0 ** -8, 2.0 ** -30]])
    assert E.linear_bf16(a, w)[0, 0] == 0x3F81
    # integer-valued operands: small integer dot products are exact
    rng = np.random.default_rng(3)
    ai = rng.integers(-8, 9, size=(5, 16)).astype(np.float64)
    wi = rng.integers(-8, 9, size=(6, 16)).astype(np.float64)
    np.testing.assert_array_equal(bf16_to_f64(E.linear_bf16(bits(ai), bits(wi))), ai @ wi.T)


# ------------------------------------------------------------------------- gate and add


def gate_inputs(M=3, hc=4, dim=256, seed=4):
    rng = np.random.default_rng(seed)
    x = bits(rng.standard_normal((M, hc, dim)))
    kv = bits(rng.standard_normal((M, dim * (hc + 1))))
    q = bits(1 + rng.uniform(-0.05, 0.05, (hc, dim)))
    k = bits(1 + rng.uniform(-0.05, 0.05, (hc, dim)))
    return x, kv, q, k


def test_gate_zero_key_is_sigmoid_of_clamp():
    # key = 0 -> dot = +0 -> gate = sigmoid(+sqrt(1e-6)) = sigmoid(1e-3) (the pages' fixed fact)
    x, kv, q, k = gate_inputs()
    kv = kv.copy()
    kv[:, : 4 * 256] = 0
    _, g = E.gate_and_add(x, kv, q, k, None, 1e-6)
    np.testing.assert_allclose(g, sigmoid(1e-3), rtol=0, atol=1e-15)
    # all-(-0) terms still give +0: negative h with w > 0 and key = +0
    x2 = bits(-np.abs(bf16_to_f64(x)))
    _, g2 = E.gate_and_add(x2, kv, q, k, None, 1e-6)
    np.testing.assert_allclose(g2, sigmoid(1e-3), rtol=0, atol=1e-15)


def test_gate_closed_form_h_equals_key(page_facts):
    # w = 1 and key = h: a = S / (S/dim + eps) / sqrt(dim), S = sum h^2 -> ~ sqrt(dim)
    for dim in (256, page_facts["dim"]):
        rng = np.random.default_rng(5)
        hc = 4
        h = bits(rng.standard_normal((2, hc, dim)))
        hv = bf16_to_f64(h)
        kv = np.concatenate([h.reshape(2, hc * dim), bits(np.zeros((2, dim)))], 1)
        one = bits(np.ones((hc, dim)))
        eps = 1e-6
        _, g = E.gate_and_add(h, kv, one, one, None, eps)
        S = (hv * hv).sum(-1)
        a = S / (S / dim + eps) / math.sqrt(dim)
        want = 1 / (1 + np.exp(-np.sqrt(a)))
        np.testing.assert_allclose(g, want, rtol=0, atol=1e-14)
        # and with eps -> 0 it is sigmoid(dim^(1/4)): 0.98201 at 256, 0.99979 at 5120
        _, g0 = E.gate_and_add(h, kv, one, one, None, 0.0)
        np.testing.assert_allclose(g0, sigmoid(dim ** 0.25), rtol=0, atol=1e-12)
        # h = -key flips the sign of a: gate -> 1 - gate
        _, gn = E.gate_and_add(bits(-hv), kv, one, one, None, 0.0)
        np.testing.assert_allclose(gn, 1 - sigmoid(dim ** 0.25), rtol=0, atol=1e-12)


def test_gate_normalised_per_stream_not_jointly():
    # scaling one stream (by a power of two, exact in bf16) leaves every gate unchanged when eps = 0;
    # a joint normalisation over the streams would move the other streams' gates.
    x, kv, q, k = gate_inputs()
    _, g = E.gate_and_add(x, kv, q, k, None, 0.0)
    xs = bf16_to_f64(x)
    xs[:, 1] *= 64.0
    _, gs = E.gate_and_add(bits(xs), kv, q, k, None, 0.0)
    np.testing.assert_allclose(gs, g, rtol=0, atol=1e-13)
    # and the key norm is per stream too: scaling stream 2's key
    kvs = bf16_to_f64(kv)
    kvs[:, 2 * 256: 3 * 256] *= 1 / 32
    _, gk = E.gate_and_add(x, bits(kvs), q, k, None, 0.0)
    np.testing.assert_allclose(gk, g, rtol=0, atol=1e-13)


def test_gate_weight_is_q_times_k():
    # swapping q and k changes nothing; q = 2, k = 1/2 equals q = k = 1
    x, kv, q, k = gate_inputs()
    _, g = E.gate_and_add(x, kv, q, k, None, 1e-6)
    _, g2 = E.gate_and_add(x, kv, k, q, None, 1e-6)
    np.testing.assert_array_equal(g, g2)
    one = bits(np.ones((4, 256)))
    _, ga = E.gate_and_add(x, kv, bits(np.full((4, 256), 2.0)), bits(np.full((4, 256), 0.5)),
                           None, 1e-6)
    _, gb = E.gate_and_add(x, kv, one, one, None, 1e-6)
    np.testing.assert_array_equal(ga, gb)


def test_gate_range_and_mask_passthrough():
    x, kv, q, k = gate_inputs(M=6)
    mask = np.array([True, False, True, False, False, True])
    out, g = E.gate_and_add(x, kv, q, k, mask, 1e-6)
    assert ((g[mask] > 0) & (g[mask] < 1)).all()
    assert (g[~mask] == 0).all()
    np.testing.assert_array_equal(out[~mask], x[~mask])        # bit for bit
    # value = 0 also leaves x untouched
    kv0 = kv.copy()
    kv0[:, 4 * 256:] = 0
    out0, _ = E.gate_and_add(x, kv0, q, k, None, 1e-6)
    np.testing.assert_array_equal(out0, x)


def test_gate_output_adds_gate_times_shared_value():
    # key = 0 fixes the gate at sigmoid(1e-3); then out = bf16(h + g * value) for every stream
    x, kv, q, k = gate_inputs(M=2)
    kv = kv.copy()
    kv[:, : 4 * 256] = 0
    out, g = E.gate_and_add(x, kv, q, k, None, 1e-6)
    v = bf16_to_f64(kv[:, 4 * 256:])
    want = bits(bf16_to_f64(x) + sigmoid(1e-3) * v[:, None, :])
    np.testing.assert_array_equal(out, want)


def test_qk_parameter_count(page_facts):
    geom = synth.FULL
    q, k = synth.make_qk(geom, np.random.default_rng(0))
    assert q.size == page_facts["q_params"] and k.size == page_facts["k_params"]
    assert q.size + k.size == page_facts["qk_params_per_block"]
    assert geom.n_hash_cols == page_facts["n_hash_cols"]
    assert E.GATE_CLAMP == page_facts["gate_clamp"]


# ------------------------------------------------------------------------------- forward


def test_forward_tiny_composes_the_stages():
    geom = synth.TINY
    model = synth.make_model(geom, synth.BASE_SEED)
    batch = synth.make_batch(geom, 2, 16, synth.BASE_SEED + 100)
    t = model.tables
    st = E.NgramHashState(t.token_map, t.pad_id, t.multipliers, t.primes, t.offsets,
                          geom.n_heads, geom.max_ngram_size, 2)
    r = E.forward(st, model.table, model.scales, model.wkv, model.q, model.k, batch.x,
                  batch.tokens, batch.mask, model.eps)
    assert r["out"].shape == (2, 16, 4, 256) and r["hash_ids"].shape == (2, 16, 24)
    assert r["kv"].shape == (2, 16, 1280) and r["rows"].shape == (2, 16, 24, 32)
    assert ((r["gate"] > 0) & (r["gate"] < 1)).all()
    # the output differs from x (value is added) but by no more than |value|
    d = np.abs(bf16_to_f64(r["out"]) - bf16_to_f64(batch.x))
    v = np.abs(bf16_to_f64(r["kv"][..., 4 * 256:]))[:, :, None, :]
    assert (d <= v + bf16_ulp(bf16_to_f64(r["out"]))).all()
