"""engram_forward_noalloc: the forward for callers that cannot allocate device memory.

It runs the same kernels as engram_forward but keeps its scratch in a fixed array the library
owns, so it must give the same results as engram_forward with a caller workspace, on every call,
although every call reuses (and overwrites) that one array. This file is collected last on
purpose, and builds everything it needs itself, so it also runs alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import deepseek_v4_engram_gb300 as eg
import synth
from deepseek_v4_engram_gb300 import _lib
from tests.helpers import (assert_gate_close, assert_out_close, dev, empty_bf16, host)

pytestmark = pytest.mark.gpu

WIDE = synth.Geometry(dim=5120, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=64,
                      vocab=129280, n_compressed=100000, prime_floor=1 << 14)


@pytest.fixture(scope="module")
def wide():
    from tests.gpu_fixtures import DeviceModel
    return DeviceModel(synth.make_model(WIDE, synth.BASE_SEED + 21, scale_mode="pow2"))


def run(dm, batch, noalloc: bool):
    B, T = batch.tokens.shape
    g = dm.geom
    cache, length = dm.new_cache(B, T)
    out = empty_bf16(B, T, g.hc_mult, g.dim)
    ids = torch.full((B, T, g.n_hash_cols), -1, dtype=torch.int32, device="cuda")
    gate = torch.full((B, T, g.hc_mult), float("nan"), device="cuda")
    kv = None if noalloc else empty_bf16(B, T, g.N)
    mask = None if batch.mask is None else dev(batch.mask)
    if noalloc:
        eg.api.engram_forward_noalloc(dm.desc, dm.tables, dm.weights, dev(batch.x),
                                      dev(batch.tokens), cache, length, mask, out,
                                      hash_ids_out=ids, gate_out=gate)
    else:
        # the caller-workspace entry point, given a workspace as large as the library's own
        # scratch, so that both calls choose the same projection path
        ws = torch.empty(_lib.NOALLOC_SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
        eg.engram_forward(dm.desc, dm.tables, dm.weights, dev(batch.x), dev(batch.tokens), cache,
                          length, mask, out, ws, hash_ids_out=ids, gate_out=gate, kv_out=kv)
    assert eg.engram_check_errors() == 0
    return host(out), host(ids), host(gate), host(length), None if kv is None else host(kv)


def test_noalloc_matches_workspace_forward_on_consecutive_calls(wide):
    g = wide.geom
    # calls in a row with different inputs and sizes (the unfused projection at 600 tokens, the
    # small-batch one at 231, the fused kernel at 1024): each overwrites the previous one's
    # scratch; all must match engram_forward with a caller-provided workspace
    batches = [synth.make_batch(g, 2, 300, synth.BASE_SEED + 500, x_dist="student_t3",
                                mask_frac=0.1),
               synth.make_batch(g, 3, 77, synth.BASE_SEED + 501),
               synth.make_batch(g, 1, 1024, synth.BASE_SEED + 502, mask_frac=0.1)]
    got = [run(wide, b, noalloc=True) for b in batches]
    for b, (out, ids, gate, length, _) in zip(batches, got):
        ref_out, ref_ids, ref_gate, ref_len, ref_kv = run(wide, b, noalloc=False)
        M = b.tokens.size
        np.testing.assert_array_equal(ids, ref_ids)
        np.testing.assert_array_equal(length, ref_len)
        assert_gate_close(gate.reshape(M, -1), ref_gate.reshape(M, -1).astype(np.float64))
        value = ref_kv.reshape(M, -1)[:, g.hc_mult * g.dim:]
        assert_out_close(out.reshape(M, g.hc_mult, g.dim), ref_out.reshape(M, g.hc_mult, g.dim),
                         value)
        np.testing.assert_array_equal(out, ref_out)   # same kernels: bit for bit


def test_noalloc_rejects_more_tokens_than_its_scratch(wide):
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
