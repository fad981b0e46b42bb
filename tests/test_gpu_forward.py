"""GPU parity of the whole forward (engram_forward) against the oracle.

Three checks per run:
  1. hash ids bit-exact, and the projection (kv_out) within one bf16 ulp of the oracle's;
  2. out and gate against the oracle's gate-and-add fed the GPU's own kv: within tolerance
     everywhere (this isolates the gate from f32-order flips of kv);
  3. gate and out against the oracle's full forward, allowing on top of the stage tolerances the
     difference that the GPU's kv (within its own tolerance) causes, as the oracle measures it.
"""
import numpy as np
import pytest
import torch

import deepseek_v4_engram_gb300 as eg
import synth
from oracle import engram as E
from oracle.numerics import bf16_to_f64, bf16_ulp
from tests.helpers import (GATE_ATOL, assert_gate_close, assert_kv_close, assert_out_close, dev,
                           empty_bf16, host, kv_flips, out_violations)

pytestmark = pytest.mark.gpu

FULLISH = synth.Geometry(dim=5120, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=64,
                         vocab=129280, n_compressed=100000, prime_floor=1 << 14)


@pytest.fixture(scope="module")
def tiny():
    from tests.gpu_fixtures import DeviceModel
    return DeviceModel(synth.make_model(synth.TINY, synth.BASE_SEED))


# dim 224 is not a multiple of the 256-column key tile: the forward takes the unfused path
ODD = synth.Geometry(dim=224, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=32, vocab=1000,
                     n_compressed=512, prime_floor=1009)


@pytest.fixture(scope="module")
def odd():
    from tests.gpu_fixtures import DeviceModel
    return DeviceModel(synth.make_model(ODD, synth.BASE_SEED + 11))


@pytest.fixture(scope="module")
def wide():
    from tests.gpu_fixtures import DeviceModel
    return DeviceModel(synth.make_model(FULLISH, synth.BASE_SEED + 9, scale_mode="pow2"))


def ws_for(dm, M, mode):
    """Workspace sized to select a path: "fastest" (the reported size), "kv" (room for a bf16 kv,
    no split-K partials), or "min" (rows + the fused kernel's scratch: the fused kernel)."""
    g = dm.geom
    r = lambda n: (n + 255) // 256 * 256
    base = r(M * g.K * 2)
    fused = eg.api.engram_wkv_gate_workspace_size(dm.desc, M)   # partial sums, gates, counters
    n = {"fastest": eg.engram_forward_workspace_size(dm.desc, M), "kv": base + r(M * g.N * 2),
         "min": base + fused}[mode]
    return torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")


def run_forward(dm, batch, cache=None, length=None, capacity=None, ws_mode="fastest"):
    B, T = batch.tokens.shape
    g = dm.geom
    if cache is None:
        cache, length = dm.new_cache(B, capacity or T)
    out = empty_bf16(B, T, g.hc_mult, g.dim)
    ids = torch.full((B, T, g.n_hash_cols), -1, dtype=torch.int32, device="cuda")
    gate = torch.full((B, T, g.hc_mult), float("nan"), device="cuda")
    kv = empty_bf16(B, T, g.N)
    ws = ws_for(dm, B * T, ws_mode)
    mask = None if batch.mask is None else dev(batch.mask)
    eg.engram_forward(dm.desc, dm.tables, dm.weights, dev(batch.x), dev(batch.tokens), cache,
                      length, mask, out, ws, hash_ids_out=ids, gate_out=gate, kv_out=kv)
    assert eg.engram_check_errors() == 0
    return dict(out=host(out), hash_ids=host(ids), gate=host(gate), kv=host(kv),
                cache=cache, length=length)


def check_against_oracle(dm, batch, r, state=None):
    B, T = batch.tokens.shape
    g, m = dm.geom, dm.model
    M = B * T
    st = state or E.NgramHashState(m.tables.token_map, m.tables.pad_id, m.tables.multipliers,
                                   m.tables.primes, m.tables.offsets, g.n_heads,
                                   g.max_ngram_size, B)
    ref = E.forward(st, m.table, m.scales, m.wkv, m.q, m.k, batch.x, batch.tokens, batch.mask,
                    m.eps)
    # 1. integer stages bit-exact, projection within one ulp
    np.testing.assert_array_equal(r["hash_ids"], ref["hash_ids"])
    A = ref["rows"].reshape(M, -1)
    assert_kv_close(r["kv"].reshape(M, -1), ref["kv"].reshape(M, -1), A, m.wkv)
    # 2. the gate stage alone, on the GPU's own kv
    mask = None if batch.mask is None else batch.mask.reshape(M)
    x = batch.x.reshape(M, g.hc_mult, g.dim)
    o2, g2 = E.gate_and_add(x, r["kv"].reshape(M, -1), m.q, m.k, mask, m.eps)
    assert_gate_close(r["gate"].reshape(M, -1), g2)
    value_gpu = r["kv"].reshape(M, -1)[:, g.hc_mult * g.dim:]
    assert_out_close(r["out"].reshape(M, g.hc_mult, g.dim), o2, value_gpu)
    # 3. end to end against the oracle's own kv. The GPU's kv may differ from the exact one
    #    (f32 accumulation): each such element must be a one-ulp flip at a rounding boundary
    #    (kv_flips). Every gate and output beyond the plain bar is counted and must trace to such
    #    a flip: a flipped value element of its column, or a flipped key element of its
    #    (token, stream) row; the size of the difference a flip may cause is measured by the
    #    oracle itself, evaluated on both kv inputs.
    flips = kv_flips(r["kv"].reshape(M, -1), A, m.wkv)
    key_rows = flips[:, : g.hc_mult * g.dim].reshape(M, g.hc_mult, g.dim).any(-1)   # [M, hc]
    value_cols = flips[:, g.hc_mult * g.dim:]                                         # [M, dim]
    value_ref = ref["kv"].reshape(M, -1)[:, g.hc_mult * g.dim:]
    plain = out_violations(r["out"].reshape(M, g.hc_mult, g.dim),
                           ref["out"].reshape(M, g.hc_mult, g.dim), value_ref)
    untraced = plain & ~(key_rows[:, :, None] | value_cols[:, None, :])
    gate_off = np.abs(r["gate"].reshape(M, -1).astype(np.float64) -
                      ref["gate"].reshape(M, -1)) > GATE_ATOL
    print(f"\n[{M} tokens] kv flips {int(flips.sum())} of {flips.size}; outputs beyond ulp + "
          f"2e-4|value| end to end: {int(plain.sum())} of {plain.size}; gates beyond 2e-4: "
          f"{int(gate_off.sum())}")
    assert not untraced.any(), f"{untraced.sum()} outputs off by more than the bar, no kv flip"
    assert not (gate_off & ~key_rows).any(), "a gate off by more than 2e-4 with no key flip"
    g_ref = ref["gate"].reshape(M, -1)
    dg_kv = np.abs(g2 - g_ref)
    dg = np.abs(r["gate"].reshape(M, -1).astype(np.float64) - g_ref)
    assert (dg <= GATE_ATOL + dg_kv).all(), f"gate error {dg.max():.3e} not explained by kv"
    o = bf16_to_f64(r["out"].reshape(M, g.hc_mult, g.dim))
    o_ref = bf16_to_f64(ref["out"].reshape(M, g.hc_mult, g.dim))
    vr = np.abs(bf16_to_f64(value_ref))[:, None, :]
    dv = np.abs(bf16_to_f64(value_gpu) - bf16_to_f64(value_ref))[:, None, :]
    tol = (2 * bf16_ulp(o_ref) + (GATE_ATOL + dg_kv[:, :, None]) * vr
           + r["gate"].reshape(M, -1)[:, :, None] * dv)
    bad = np.abs(o - o_ref) > tol
    assert not bad.any(), f"{bad.sum()} outputs not explained by kv; first {np.argwhere(bad)[:3]}"
    if mask is not None:
        np.testing.assert_array_equal(r["out"].reshape(M, g.hc_mult, g.dim)[~mask], x[~mask])
    return ref


@pytest.mark.parametrize("ws_mode", ["fastest", "kv", "min"])
@pytest.mark.parametrize("B,T", [(1, 16), (2, 17), (1, 129), (3, 100)])
def test_forward_tiny(tiny, B, T, ws_mode):
    batch = synth.make_batch(tiny.geom, B, T, synth.BASE_SEED + 100 + T)
    check_against_oracle(tiny, batch, run_forward(tiny, batch, ws_mode=ws_mode))


@pytest.mark.parametrize("B,T", [(1, 5), (2, 150)])
def test_forward_unfused_geometry(odd, B, T):
    batch = synth.make_batch(odd.geom, B, T, synth.BASE_SEED + 400 + T, mask_frac=0.2)
    check_against_oracle(odd, batch, run_forward(odd, batch))


@pytest.mark.parametrize("ws_mode", ["fastest", "kv", "min"])
@pytest.mark.parametrize("B,T,mask_frac", [(1, 1, 0.0), (2, 77, 0.0), (1, 300, 0.1),
                                           (4, 160, 0.1), (64, 1, 0.0), (1, 513, 0.1),
                                           (1, 700, 0.1)])
def test_forward_full_width(wide, B, T, mask_frac, ws_mode):
    batch = synth.make_batch(wide.geom, B, T, synth.BASE_SEED + 200 + T, x_dist="student_t3",
                             mask_frac=mask_frac)
    check_against_oracle(wide, batch, run_forward(wide, batch, ws_mode=ws_mode))


@pytest.mark.parametrize("B,T", [(1, 256), (2, 125), (1, 512), (1, 513), (1, 700), (2, 1024)])
def test_deferred_output_equals_fused(wide, B, T):
    # at 240-256 and 512-2048 tokens the fastest workspace runs the fused kernel with its output
    # deferred
    # (bf16 value rows, then out = x + gate * value in a second kernel); the minimum workspace runs
    # the fused kernel alone. Both round the value to bf16 and take one fma per element: equal bits.
    batch = synth.make_batch(wide.geom, B, T, synth.BASE_SEED + 260 + T, x_dist="student_t3",
                             mask_frac=0.1)
    deferred = run_forward(wide, batch, ws_mode="fastest")
    fused = run_forward(wide, batch, ws_mode="min")
    for key in ("out", "gate", "kv", "hash_ids"):
        np.testing.assert_array_equal(deferred[key], fused[key])


# Other shapes the kernels take: 1, 2 and 8 streams, 256-768 columns per stream, 2-5-grams,
# head_dim 32 and 64 (every projection path at each: decode, small-batch, deferred and fused)
OTHER = {
    "hc2_dim512": synth.Geometry(dim=512, hc_mult=2, n_heads=4, max_ngram_size=3, head_dim=32,
                                 vocab=3000, n_compressed=1500, prime_floor=2003),
    "hc8_dim256": synth.Geometry(dim=256, hc_mult=8, n_heads=8, max_ngram_size=4, head_dim=32,
                                 vocab=3000, n_compressed=1500, prime_floor=3001),
    "hc1_dim768": synth.Geometry(dim=768, hc_mult=1, n_heads=2, max_ngram_size=5, head_dim=64,
                                 vocab=3000, n_compressed=1500, prime_floor=4001),
}


@pytest.fixture(scope="module")
def others():
    from tests.gpu_fixtures import DeviceModel
    return {k: DeviceModel(synth.make_model(g, synth.BASE_SEED + 70 + i, scale_mode="pow2"))
            for i, (k, g) in enumerate(OTHER.items())}


@pytest.mark.parametrize("name", list(OTHER))
@pytest.mark.parametrize("B,T", [(8, 1), (1, 200), (2, 125), (1, 600), (1, 2100)])
def test_forward_other_geometries(others, name, B, T):
    dm = others[name]
    batch = synth.make_batch(dm.geom, B, T, synth.BASE_SEED + 280 + T, x_dist="student_t3",
                             mask_frac=0.1 if T > 1 else 0.0)
    r = run_forward(dm, batch)
    check_against_oracle(dm, batch, r)
    if B * T >= 200:   # and the fused kernel alone (the minimum workspace) gives the same bits as
        fused = run_forward(dm, batch, ws_mode="min")   # the fastest plan where that is fused
        if 240 <= B * T <= 256 or 512 <= B * T:
            for key in ("out", "gate", "kv", "hash_ids"):
                np.testing.assert_array_equal(r[key], fused[key])
        else:
            check_against_oracle(dm, batch, fused)


def test_prefill_then_decode_equals_one_prefill(wide):
    # the look-back cache carries across calls: prefill(T) == prefill(T-j) + j decode steps
    B, T, j = 3, 40, 4
    batch = synth.make_batch(wide.geom, B, T, synth.BASE_SEED + 300)
    whole = run_forward(wide, batch)
    cache, length = wide.new_cache(B, T)
    head = synth.Batch(batch.tokens[:, :T - j], batch.x[:, :T - j], None)
    parts = [run_forward(wide, head, cache, length)]
    for t in range(T - j, T):
        step = synth.Batch(batch.tokens[:, t:t + 1], batch.x[:, t:t + 1], None)
        parts.append(run_forward(wide, step, cache, length))
    # the hash is integer-exact across the split; out and kv of the split run come from other
    # projection kernels (token counts pick the path), so they are checked against the oracle
    np.testing.assert_array_equal(np.concatenate([p["hash_ids"] for p in parts], 1),
                                  whole["hash_ids"])
    np.testing.assert_array_equal(host(length), [T] * B)
    split = {k: np.concatenate([p[k] for p in parts], 1) for k in ("hash_ids", "out", "kv", "gate")}
    check_against_oracle(wide, batch, split)


# ------------------------------------------------------------------ forward from given hash ids


def run_forward_ids(dm, batch, ids, ws_mode):
    B, T = batch.tokens.shape
    g, M = dm.geom, batch.tokens.size
    out = empty_bf16(M, g.hc_mult, g.dim)
    gate = torch.full((M, g.hc_mult), float("nan"), device="cuda")
    kv = empty_bf16(M, g.N)
    mask = None if batch.mask is None else dev(batch.mask.reshape(M))
    eg.engram_forward_ids(dm.desc, dm.weights, dev(batch.x.reshape(M, g.hc_mult, g.dim)),
                          dev(np.ascontiguousarray(ids.reshape(M, -1), dtype=np.int32)), mask,
                          out, ws_for(dm, M, ws_mode), gate_out=gate, kv_out=kv)
    return host(out), host(gate), host(kv)


@pytest.mark.parametrize("ws_mode", ["fastest", "min"])
@pytest.mark.parametrize("B,T,mask_frac", [(1, 1, 0.0), (64, 1, 0.0), (2, 77, 0.1), (1, 300, 0.0),
                                           (1, 700, 0.1)])
def test_forward_ids_equals_forward(wide, B, T, mask_frac, ws_mode):
    # the same ids through engram_forward_ids and engram_forward take the same kernels after the
    # gather: bit-identical results; and both against the oracle
    batch = synth.make_batch(wide.geom, B, T, synth.BASE_SEED + 900 + T, mask_frac=mask_frac)
    r = run_forward(wide, batch, ws_mode=ws_mode)
    out, gate, kv = run_forward_ids(wide, batch, r["hash_ids"], ws_mode)
    assert eg.engram_check_errors() == 0
    M = B * T
    np.testing.assert_array_equal(out, r["out"].reshape(out.shape))
    np.testing.assert_array_equal(gate, r["gate"].reshape(gate.shape))
    np.testing.assert_array_equal(kv, r["kv"].reshape(kv.shape))
    check_against_oracle(wide, batch, dict(out=out, gate=gate, kv=kv, hash_ids=r["hash_ids"]))


@pytest.mark.parametrize("B,T", [(1, 5), (2, 150)])
def test_forward_ids_unfused_geometry_and_bad_id(odd, B, T):
    batch = synth.make_batch(odd.geom, B, T, synth.BASE_SEED + 950 + T, mask_frac=0.2)
    st = E.NgramHashState(odd.model.tables.token_map, odd.model.tables.pad_id,
                          odd.model.tables.multipliers, odd.model.tables.primes,
                          odd.model.tables.offsets, odd.geom.n_heads, odd.geom.max_ngram_size, B)
    ids = st.push(batch.tokens)
    out, gate, kv = run_forward_ids(odd, batch, ids, "fastest")
    assert eg.engram_check_errors() == 0
    check_against_oracle(odd, batch, dict(out=out, gate=gate, kv=kv, hash_ids=ids))
    # an id outside the table gathers a zero row and sets the error bit
    bad = ids.copy()
    bad[0, 0, 3] = odd.model.tables.num_embeddings
    run_forward_ids(odd, batch, bad, "fastest")
    assert eg.engram_check_errors() & 4


@pytest.mark.parametrize("B,T", [(64, 1), (1, 300), (1, 700)])
def test_forward_degenerate_masks(wide, B, T):
    # every token masked (an all-image batch): out is x bit for bit and every gate is 0; an
    # explicit all-True mask gives bit for bit what no mask gives. Decode, unfused and fused paths.
    import dataclasses
    batch = synth.make_batch(wide.geom, B, T, synth.BASE_SEED + 970 + T)
    none = run_forward(wide, batch)
    all_true = run_forward(wide, dataclasses.replace(batch, mask=np.ones((B, T), dtype=bool)))
    for key in ("out", "gate", "kv", "hash_ids"):
        np.testing.assert_array_equal(all_true[key], none[key])
    masked = run_forward(wide, dataclasses.replace(batch, mask=np.zeros((B, T), dtype=bool)))
    np.testing.assert_array_equal(masked["out"].reshape(batch.x.shape), batch.x)
    assert (masked["gate"] == 0).all()
    np.testing.assert_array_equal(masked["kv"], none["kv"])   # the projection ignores the mask
