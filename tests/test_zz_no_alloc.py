"""engram_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot hand this library a workspace: a runtime that owns all device memory and
passes a plugin only its input and output buffers, or a serving loop that must never call
cudaMalloc once it runs (cudaMalloc can synchronise the whole device). engram_forward_noalloc
serves them with the library's own fixed scratch array. It picks the fastest projection path whose
scratch fits that array, exactly as engram_forward does for a workspace of the same size, so
each call must give bit for bit what engram_forward gives with a workspace that admits only that
path; and every call reuses (and overwrites) the one array, so the calls are made in a row with
different sizes and paths.

This file is collected last on purpose, and builds everything it needs itself, so it also runs
alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import deepseek_v4_engram_gb300 as eg
import synth
from deepseek_v4_engram_gb300 import _lib
from tests.helpers import dev, empty_bf16, host

pytestmark = pytest.mark.gpu

WIDE = synth.Geometry(dim=5120, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=64,
                      vocab=129280, n_compressed=100000, prime_floor=1 << 14)


@pytest.fixture(scope="module")
def models():
    from tests.gpu_fixtures import DeviceModel
    return {"wide": DeviceModel(synth.make_model(WIDE, synth.BASE_SEED + 21, scale_mode="pow2")),
            "tiny": DeviceModel(synth.make_model(synth.TINY, synth.BASE_SEED + 22))}


def r256(n):
    return (n + 255) // 256 * 256


def reference_workspace_bytes(dm, M):
    """The workspace that makes engram_forward take the path engram_forward_noalloc takes: the
    fastest path's size when it fits the library's array, else the smallest workspace (rows and
    the fused kernel's scratch), which admits the fused path only."""
    fastest = eg.engram_forward_workspace_size(dm.desc, M)
    if fastest <= _lib.NOALLOC_SCRATCH_BYTES:
        return fastest, "fastest"
    return r256(M * dm.geom.K * 2) + eg.api.engram_wkv_gate_workspace_size(dm.desc, M), "fused"


def run(dm, batch, noalloc: bool):
    B, T = batch.tokens.shape
    g = dm.geom
    cache, length = dm.new_cache(B, T)
    out = empty_bf16(B, T, g.hc_mult, g.dim)
    ids = torch.full((B, T, g.n_hash_cols), -1, dtype=torch.int32, device="cuda")
    gate = torch.full((B, T, g.hc_mult), float("nan"), device="cuda")
    mask = None if batch.mask is None else dev(batch.mask)
    if noalloc:
        eg.api.engram_forward_noalloc(dm.desc, dm.tables, dm.weights, dev(batch.x),
                                      dev(batch.tokens), cache, length, mask, out,
                                      hash_ids_out=ids, gate_out=gate)
    else:
        n, _ = reference_workspace_bytes(dm, B * T)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        eg.engram_forward(dm.desc, dm.tables, dm.weights, dev(batch.x), dev(batch.tokens), cache,
                          length, mask, out, ws, hash_ids_out=ids, gate_out=gate)
    assert eg.engram_check_errors() == 0
    return host(out), host(ids), host(gate), host(length)


# (model, B, T, path engram_forward_noalloc takes at that size)
CALLS = [("wide", 64, 1, "fastest"),     # decode: weight-streaming projection, bf16 kv (~3.5 MB)
         ("tiny", 2, 150, "fastest"),    # 300 tokens at dim 256: projection GEMM, then the gate
         ("wide", 2, 256, "fastest"),    # 512 tokens: fused kernel, deferred output (~7.4 MB)
         ("wide", 1, 1024, "fused"),     # its deferred-output plan needs ~14.6 MB: the fused one
         ("wide", 3, 77, "fused")]       # its fastest path needs ~12.5 MB: the fused one fits


def test_noalloc_matches_workspace_forward_on_consecutive_calls(models):
    batches = []
    for i, (name, B, T, path) in enumerate(CALLS):
        dm = models[name]
        assert reference_workspace_bytes(dm, B * T)[1] == path
        batches.append((dm, synth.make_batch(dm.geom, B, T, synth.BASE_SEED + 500 + i,
                                             x_dist="student_t3", mask_frac=0.1)))
    # every call in a row through the shared array, then each against the workspace forward
    got = [run(dm, b, noalloc=True) for dm, b in batches]
    for (dm, b), g in zip(batches, got):
        ref = run(dm, b, noalloc=False)
        for a, r in zip(g, ref):
            np.testing.assert_array_equal(a, r)


def test_noalloc_rejects_more_tokens_than_its_scratch(models):
    wide = models["wide"]
    B, T = 1, 4096                                     # 4096 tokens need ~13 MB > 8 MiB
    x = torch.zeros((B, T, 4, 5120), dtype=torch.int16, device="cuda")
    out = torch.empty_like(x)
    tokens = torch.zeros((B, T), dtype=torch.int32, device="cuda")
    cache, length = wide.new_cache(B, T)
    with pytest.raises(eg.EngramError) as e:
        eg.api.engram_forward_noalloc(wide.desc, wide.tables, wide.weights, x, tokens, cache,
                                      length, None, out)
    assert e.value.code == _lib.ENGRAM_EINVAL and "scratch" in str(e.value)
    assert _lib.NOALLOC_SCRATCH_BYTES == 8 * 1024 * 1024
