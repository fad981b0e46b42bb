"""Parity at the full workload sizes, in the launch configuration the benchmark times.

Full geometry (dim 5120, hc 4, 24 rows x head_dim 64) with the full ~805 MB fp8 table:
  * prefill B1 T4096: the benchmark's step (engram_hash -> engram_embed_rows -> engram_wkv_gate)
    and engram_forward, every token compared with the oracle;
  * decode B64 after a 2048-token prefill per sequence: hash ids must reach into the cache;
  * masked batched prefill B8 T8192 (pow2 scales, Student-t x, ~10% masked spans): a sample of
    tokens compared with the oracle, and every masked token checked bit for bit;
  * sweep end points T = 1 and T = 65536 (sampled).
Runs of 640 tokens and more take the fused kernel; their sampled tokens are re-run alone through
engram_wkv_gate, which must reproduce them bit for bit and also returns the kv it used.
"""
import numpy as np
import pytest
import torch

import deepseek_v4_engram_gb300 as eg
import synth
from oracle import engram as E
from tests.helpers import assert_gate_close, assert_kv_close, assert_out_close, dev, host

pytestmark = pytest.mark.gpu

G = synth.FULL


@pytest.fixture(scope="module")
def full():
    from tests.gpu_fixtures import DeviceModel
    return DeviceModel(synth.make_model(G, synth.BASE_SEED + 1))


def oracle_state(m, B):
    t = m.tables
    return E.NgramHashState(t.token_map, t.pad_id, t.multipliers, t.primes, t.offsets, G.n_heads,
                            G.max_ngram_size, B)


def oracle_tokens(m, ids, x, mask, idx):
    """Oracle rows -> kv -> gate/out for the flat token indices idx (ids: [M, 24], x: [M,hc,dim])."""
    rows = E.embed_rows(m.table, m.scales, ids[idx]).reshape(len(idx), -1)
    kv = E.linear_bf16(rows, m.wkv)
    out, gate = E.gate_and_add(x[idx], kv, m.q, m.k, None if mask is None else mask[idx], m.eps)
    return rows, kv, out, gate


def check_tokens(dm, ids, x, mask, idx, out_gpu, gate_gpu):
    """Sampled parity for tokens idx of a large run.

    The projection of a token does not depend on the other tokens of its tile, so running the
    fused kernel on just these tokens (with the oracle's rows, which the GPU reproduces bit for
    bit) must reproduce the large run's outputs exactly, and it also returns the kv it used. The
    stage tolerances are then applied against the oracle given that kv, and the kv against the
    exact projection.
    """
    m = dm.model
    n = len(idx)
    rows = E.embed_rows(m.table, m.scales, ids[idx]).reshape(n, -1)
    xs = np.ascontiguousarray(x[idx])
    ms = None if mask is None else np.ascontiguousarray(mask[idx])
    out = torch.full((n, 4, 5120), 0x7FC1, dtype=torch.int16, device="cuda")
    gate = torch.full((n, 4), float("nan"), device="cuda")
    kv = torch.full((n, G.N), 0x7FC1, dtype=torch.int16, device="cuda")
    eg.engram_wkv_gate(dm.desc, dev(rows), dm.weights.wkv, dev(xs), dm.weights.q_weight,
                       dm.weights.k_weight, None if ms is None else dev(ms), out, gate, kv)
    assert eg.engram_check_errors() == 0
    np.testing.assert_array_equal(host(out), out_gpu[idx])
    np.testing.assert_array_equal(host(gate), gate_gpu[idx])
    kv_h = host(kv)
    assert_kv_close(kv_h, E.linear_bf16(rows, m.wkv), rows, m.wkv)
    o2, g2 = E.gate_and_add(xs, kv_h, m.q, m.k, ms, m.eps)
    assert_gate_close(gate_gpu[idx], g2)
    assert_out_close(out_gpu[idx], o2, kv_h[:, G.hc_mult * G.dim:])


def check_with_kv(m, ids, x, mask, out_gpu, gate_gpu, kv_gpu):
    """Stage-wise parity of every token of a run that also returned its kv."""
    rows = E.embed_rows(m.table, m.scales, ids).reshape(len(ids), -1)
    assert_kv_close(kv_gpu, E.linear_bf16(rows, m.wkv), rows, m.wkv)
    o2, g2 = E.gate_and_add(x, kv_gpu, m.q, m.k, mask, m.eps)
    assert_gate_close(gate_gpu, g2)
    assert_out_close(out_gpu, o2, kv_gpu[:, G.hc_mult * G.dim:])


def test_prefill_b1_t4096_bench_configuration(full):
    m = full.model
    B, T = 1, 4096
    M = B * T
    batch = synth.make_batch(G, B, T, synth.BASE_SEED + 101)
    x, tok = dev(batch.x), dev(batch.tokens)
    cache, length = full.new_cache(B, T)
    ids = torch.empty((B, T, 24), dtype=torch.int32, device="cuda")
    rows = torch.empty((M * 24, 64), dtype=torch.int16, device="cuda")
    out = torch.full_like(x, 0x7FC1)
    gate = torch.full((M, 4), float("nan"), device="cuda")
    kv = torch.full((M, G.N), 0x7FC1, dtype=torch.int16, device="cuda")
    eg.engram_hash(full.desc, full.tables, tok, cache, length, ids)
    eg.engram_embed_rows(full.desc, full.weights.table, full.weights.scales, ids.view(-1), rows)
    eg.engram_wkv_gate(full.desc, rows.view(M, -1), full.weights.wkv, x.view(M, 4, 5120),
                       full.weights.q_weight, full.weights.k_weight, None,
                       out.view(M, 4, 5120), gate, kv)
    assert eg.engram_check_errors() == 0
    st = oracle_state(m, B)
    ref_ids = st.push(batch.tokens)
    np.testing.assert_array_equal(host(ids), ref_ids)
    ids_f = ref_ids.reshape(M, 24)
    sample = np.random.default_rng(0).choice(M, 64, replace=False)
    np.testing.assert_array_equal(host(rows).reshape(M, 24, 64)[sample],
                                  E.embed_rows(m.table, m.scales, ids_f[sample]))
    # every token: projection, gate and output against the oracle
    ref_rows = E.embed_rows(m.table, m.scales, ids_f).reshape(M, -1)
    ref_kv = E.linear_bf16(ref_rows, m.wkv)
    kv_h = host(kv)
    assert_kv_close(kv_h, ref_kv, ref_rows, m.wkv)
    xf = batch.x.reshape(M, 4, 5120)
    o2, g2 = E.gate_and_add(xf, kv_h, m.q, m.k, None, m.eps)
    assert_gate_close(host(gate), g2)
    assert_out_close(host(out).reshape(M, 4, 5120), o2, kv_h[:, 4 * 5120:])
    # and the public forward (which takes the fused path at this size) gives the same result
    cache2, length2 = full.new_cache(B, T)
    out2 = torch.full_like(x, 0x7FC1)
    ws = full.workspace(M)
    eg.engram_forward(full.desc, full.tables, full.weights, x, tok, cache2, length2, None, out2, ws)
    assert eg.engram_check_errors() == 0
    np.testing.assert_array_equal(host(out2), host(out))


def test_decode_b64_after_2048_prefill(full):
    m = full.model
    B, P = 64, 2048
    rng = np.random.default_rng(synth.BASE_SEED + 102)
    pre = rng.integers(0, G.vocab, (B, P), dtype=np.int32)
    cache, length = full.new_cache(B, P + 4)
    ids_pre = torch.empty((B, P, 24), dtype=torch.int32, device="cuda")
    eg.engram_hash(full.desc, full.tables, dev(pre), cache, length, ids_pre)
    st = oracle_state(m, B)
    np.testing.assert_array_equal(host(ids_pre), st.push(pre))
    for step in range(2):
        batch = synth.make_batch(G, B, 1, synth.BASE_SEED + 700 + step)
        out = torch.full((B, 1, 4, 5120), 0x7FC1, dtype=torch.int16, device="cuda")
        gate = torch.full((B, 1, 4), float("nan"), device="cuda")
        ids = torch.empty((B, 1, 24), dtype=torch.int32, device="cuda")
        kv = torch.full((B, G.N), 0x7FC1, dtype=torch.int16, device="cuda")
        eg.engram_forward(full.desc, full.tables, full.weights, dev(batch.x), dev(batch.tokens),
                          cache, length, None, out, full.workspace(B), hash_ids_out=ids,
                          gate_out=gate, kv_out=kv)
        assert eg.engram_check_errors() == 0
        ref_ids = st.push(batch.tokens)
        np.testing.assert_array_equal(host(ids), ref_ids)     # look-back reaches the prefill
        check_with_kv(m, ref_ids.reshape(B, 24), batch.x.reshape(B, 4, 5120), None,
                      host(out).reshape(B, 4, 5120), host(gate).reshape(B, 4), host(kv))
    np.testing.assert_array_equal(host(length), [P + 2] * B)


def whole_tiles(M, tile=256):
    """Every token of three 256-token tiles of the fused kernel's work: the first, the middle and
    the last, so that the first, a middle and the last group of its schedule are covered whole."""
    n = M // tile
    return np.concatenate([np.arange(t * tile, (t + 1) * tile) for t in (0, n // 2, n - 1)])


def _run_large(full, B, T, seed, x_dist, mask_frac, model, want_kv=False):
    batch = synth.make_batch(G, B, T, seed, x_dist=x_dist, mask_frac=mask_frac)
    M = B * T
    x, tok = dev(batch.x), dev(batch.tokens)
    mask = None if batch.mask is None else dev(batch.mask)
    cache, length = full.new_cache(B, T)
    out = torch.full_like(x, 0x7FC1)
    gate = torch.full((M, 4), float("nan"), device="cuda")
    ids = torch.empty((B, T, 24), dtype=torch.int32, device="cuda")
    ws = full.workspace(M)
    kv = torch.empty((M, G.N), dtype=torch.int16, device="cuda") if want_kv else None
    eg.engram_forward(full.desc, full.tables, full.weights, x, tok, cache, length, mask, out, ws,
                      hash_ids_out=ids, gate_out=gate, kv_out=kv)
    assert eg.engram_check_errors() == 0
    ref_ids = oracle_state(model, B).push(batch.tokens)
    np.testing.assert_array_equal(host(ids), ref_ids)
    res = (batch, ref_ids.reshape(M, 24), host(out).reshape(M, 4, 5120), host(gate))
    return res + (host(kv),) if want_kv else res


def test_masked_b8_t8192_sampled(full):
    # the masked workload uses e8m0 scales 2^[-4,4]: same codes and weights, other scales
    model = synth.make_model(G, synth.BASE_SEED + 1, scale_mode="pow2")
    from tests.gpu_fixtures import DeviceModel
    dm = DeviceModel(model)
    B, T = 8, 8192
    M = B * T
    batch, ids, out, gate = _run_large(dm, B, T, synth.BASE_SEED + 103, "student_t3", 0.10, model)
    mask = batch.mask.reshape(M)
    x = batch.x.reshape(M, 4, 5120)
    assert 0.08 < (~mask).mean() < 0.12
    np.testing.assert_array_equal(out[~mask], x[~mask])          # every masked token, bit exact
    assert (gate[~mask] == 0).all() and ((gate[mask] > 0) & (gate[mask] < 1)).all()
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([rng.choice(np.nonzero(mask)[0], 96, replace=False),
                                    rng.choice(np.nonzero(~mask)[0], 16, replace=False),
                                    whole_tiles(M)]))
    check_tokens(dm, ids, x, mask, idx, out, gate)


def test_sweep_t1(full):
    batch, ids, out, gate, kv = _run_large(full, 1, 1, synth.BASE_SEED + 104, "normal", 0.0,
                                           full.model, want_kv=True)
    check_with_kv(full.model, ids, batch.x.reshape(1, 4, 5120), None, out, gate, kv)


def test_sweep_t65536_sampled(full):
    M = 65536
    batch, ids, out, gate = _run_large(full, 1, M, synth.BASE_SEED + 104, "normal", 0.0,
                                       full.model)
    idx = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(M).integers(0, M, 64),
                                    whole_tiles(M)]))
    check_tokens(full, ids, batch.x.reshape(M, 4, 5120), None, idx, out, gate)
    assert ((gate > 0) & (gate < 1)).all()
