"""Host-side checks of the C ABI (no GPU): the library loads, exports every declared entry point,
and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from deepseek_v4_engram_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_entry_points():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"ENGRAM_API\s+[\w\s\*]+?\b(engram_\w+)\s*\(", src)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"
    assert lib.engram_abi_version() == 1


def desc(**kw):
    d = dict(dim=256, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=32, reserved=0,
             num_embeddings=25874, norm_eps=1e-6)
    d.update(kw)
    return _lib.EngramDesc(**d)


def test_wkv_validation(lib):
    assert lib.engram_wkv(None, None, None, 16, 1280, 768, None) == _lib.ENGRAM_EINVAL
    assert lib.engram_wkv(None, None, None, 16, 1280, 760, None) == _lib.ENGRAM_EUNSUPPORTED
    assert lib.engram_wkv(None, None, None, -1, 1280, 768, None) == _lib.ENGRAM_EINVAL
    assert lib.engram_wkv(None, None, None, 0, 1280, 768, None) == _lib.ENGRAM_OK   # empty
    assert lib.engram_wkv(8, 0x1000000, 0x4000000, 16, 1280, 768, None) == _lib.ENGRAM_EINVAL
    assert b"aligned" in lib.engram_last_error()


@pytest.mark.parametrize("bad", [dict(head_dim=48), dict(dim=0), dict(max_ngram_size=1),
                                 dict(num_embeddings=1 << 31), dict(norm_eps=-1.0),
                                 dict(dim=260)])
def test_desc_validation(lib, bad):
    d = desc(**bad)
    assert lib.engram_embed_rows(ctypes.byref(d), 16, 16, 16, 4, 16, None) == _lib.ENGRAM_EINVAL
    assert lib.engram_forward_workspace_size(ctypes.byref(d), 16) == 0


def test_shard_rows_validation(lib):
    d = desc()
    n = d.num_embeddings
    f = lib.engram_embed_rows_shard
    # the shard must lie in [0, num_embeddings)
    assert f(ctypes.byref(d), 16, 16, -1, 10, 16, 4, 16, None) == _lib.ENGRAM_EINVAL
    assert f(ctypes.byref(d), 16, 16, n - 5, 10, 16, 4, 16, None) == _lib.ENGRAM_EINVAL
    assert b"shard" in lib.engram_last_error()
    # NULL ids, a misaligned shard; nothing to do for 0 ids
    assert f(ctypes.byref(d), 16, 16, 0, 10, None, 4, 16, None) == _lib.ENGRAM_EINVAL
    assert f(ctypes.byref(d), 24, 16, 0, 10, 16, 4, 16, None) == _lib.ENGRAM_EINVAL
    assert f(ctypes.byref(d), None, None, 0, 0, None, 0, None, None) == _lib.ENGRAM_OK


def test_stream_probe_validation(lib):
    f = lib.engram_probe_stream_read
    assert f(16, 64, 3, None) == _lib.ENGRAM_EINVAL            # no such method
    assert f(16, 40, 0, None) == _lib.ENGRAM_EINVAL            # not a multiple of 16 bytes
    assert f(24, 64, 1, None) == _lib.ENGRAM_EINVAL            # misaligned
    assert f(None, 64, 0, None) == _lib.ENGRAM_EINVAL
    assert f(None, 0, 0, None) == _lib.ENGRAM_OK               # nothing to read


def test_graph_handle_validation(lib):
    d = desc()
    t = _lib.EngramTables(0x1000, 1000, 0, 0x2000, 0x3000, 0x4000)
    w = _lib.EngramWeights()
    # no place for the handle: rejected before any CUDA call
    assert lib.engram_forward_graph_create(ctypes.byref(d), ctypes.byref(t), ctypes.byref(w), 16,
                                           16, 1, 1, 16, 16, 8, None, 16, None, None, None, 256,
                                           1 << 20, None) == _lib.ENGRAM_EINVAL
    assert lib.engram_graph_launch(None, None) == _lib.ENGRAM_EINVAL
    assert b"graph" in lib.engram_last_error()
    assert lib.engram_graph_destroy(None) == _lib.ENGRAM_OK


def test_forward_workspace_is_the_deferred_plans_exactly_in_its_ranges(lib):
    # the fastest workspace holds the gathered rows, the fused kernel's scratch and the bf16 value
    # rows exactly where engram_forward takes the deferred-output plan: 240-256 and 512-2048 tokens
    # at the full geometry
    d = desc(dim=5120, head_dim=64, num_embeddings=1 << 20)
    r = lambda n: (n + 255) // 256 * 256
    for M in (200, 239, 240, 250, 256, 257, 384, 511, 512, 700, 2048, 2049, 4096):
        ws = lib.engram_forward_workspace_size(ctypes.byref(d), M)
        deferred = (r(M * 1536 * 2) + r(lib.engram_wkv_gate_workspace_size(ctypes.byref(d), M))
                    + r(M * 5120 * 2))
        assert (ws == deferred) == (240 <= M <= 256 or 512 <= M <= 2048), M


def test_gate_rejects_aliasing_and_misalignment(lib):
    d = desc()
    x = 0x10000
    # out overlapping x
    rc = lib.engram_gate_and_add(ctypes.byref(d), x, 0x900000, 0x2000, 0x4000, None, x + 256,
                                 None, 4, None)
    assert rc == _lib.ENGRAM_EINVAL and b"overlaps" in lib.engram_last_error()
    rc = lib.engram_gate_and_add(ctypes.byref(d), x + 2, 0x900000, 0x2000, 0x4000, None,
                                 0x800000, None, 4, None)
    assert rc == _lib.ENGRAM_EINVAL and b"aligned" in lib.engram_last_error()
    assert lib.engram_gate_and_add(ctypes.byref(d), None, None, None, None, None, None, None, 0,
                                   None) == _lib.ENGRAM_OK


def test_hash_validation(lib):
    d = desc()
    t = _lib.EngramTables(0x1000, 1000, 0, 0x2000, 0x3000, 0x4000)
    args = [ctypes.byref(d), ctypes.byref(t), 0x5000, 2, 3, 0x6000, 0x7000, 8, 0x8000, None]
    bad = list(args)
    bad[3] = -1
    assert lib.engram_hash(*bad) == _lib.ENGRAM_EINVAL
    bad = list(args)
    bad[8] = None
    assert lib.engram_hash(*bad) == _lib.ENGRAM_EINVAL
    t2 = _lib.EngramTables(0x1000, 1000, -3, 0x2000, 0x3000, 0x4000)
    bad = list(args)
    bad[1] = ctypes.byref(t2)
    assert lib.engram_hash(*bad) == _lib.ENGRAM_EINVAL
    # ids overlapping the cache
    bad = list(args)
    bad[8] = 0x6000
    assert lib.engram_hash(*bad) == _lib.ENGRAM_EINVAL
    bad = list(args)
    bad[3] = 0
    assert lib.engram_hash(*bad) == _lib.ENGRAM_OK          # nothing to do


def test_forward_workspace_and_validation(lib):
    d = desc()
    n16 = lib.engram_forward_workspace_size(ctypes.byref(d), 16)
    n32 = lib.engram_forward_workspace_size(ctypes.byref(d), 32)
    assert n16 > 0 and n32 > n16 and n16 % 256 == 0
    t = _lib.EngramTables(0x1000, 1000, 0, 0x2000, 0x3000, 0x4000)
    w = _lib.EngramWeights(0x10000, 0x20000, 0x30000, 0x40000, 0x50000)
    # workspace too small
    rc = lib.engram_forward(ctypes.byref(d), ctypes.byref(t), ctypes.byref(w), 0x100000, 0x5000,
                            1, 16, 0x6000, 0x7000, 16, None, 0x900000, None, None, None,
                            0x1000000, 64, None)
    assert rc == _lib.ENGRAM_EINVAL and b"workspace" in lib.engram_last_error()
    # weights missing
    rc = lib.engram_forward(ctypes.byref(d), ctypes.byref(t), None, 0x100000, 0x5000, 1, 16,
                            0x6000, 0x7000, 16, None, 0x900000, None, None, None, 0x1000000,
                            n16, None)
    assert rc == _lib.ENGRAM_EINVAL


def test_hash_rows_layers_validation(lib):
    d = desc()
    t = _lib.EngramTables(0x1000, 1000, 0, None, None, None)   # per-layer constants not read

    def layer(**kw):
        f = dict(multipliers=0x2000, primes=0x3000, offsets=0x4000, num_embeddings=25874,
                 table=0x10000, scales=0x20000, rows=0x40000, hash_ids=None)
        f.update(kw)
        return _lib.EngramLayerHash(**f)

    def call(layers, n=None, B=2, T=3, cache=0x6000, cap=8):
        arr = (_lib.EngramLayerHash * max(len(layers), 1))(*layers)
        return lib.engram_hash_rows_layers(ctypes.byref(d), ctypes.byref(t), arr,
                                           len(layers) if n is None else n, 0x5000, B, T, cache,
                                           0x7000, cap, None)

    ok = [layer(), layer(num_embeddings=30000, rows=0x80000)]
    assert call(ok, B=0) == _lib.ENGRAM_OK                       # nothing to do
    assert call(ok, n=0) == _lib.ENGRAM_EINVAL
    assert call([layer()] * 17) == _lib.ENGRAM_EINVAL            # above ENGRAM_MAX_HASH_LAYERS
    assert call([layer(), layer(table=None)]) == _lib.ENGRAM_EINVAL
    assert b"layer 1" in lib.engram_last_error()
    assert call([layer(rows=None)]) == _lib.ENGRAM_EINVAL
    assert call([layer(rows=None)], B=0) == _lib.ENGRAM_OK       # no output when empty
    assert call([layer(rows=0x40008)]) == _lib.ENGRAM_EINVAL     # rows not 16-byte aligned
    assert call([layer(num_embeddings=1 << 31)]) == _lib.ENGRAM_EINVAL
    assert call([layer(rows=0x6000)]) == _lib.ENGRAM_EINVAL      # rows overlap the cache
    assert call([layer(hash_ids=0x6010)]) == _lib.ENGRAM_EINVAL  # ids overlap the cache
    assert call(ok, B=-1) == _lib.ENGRAM_EINVAL
    assert lib.engram_hash_rows_layers(ctypes.byref(d), ctypes.byref(t), None, 1, 0x5000, 2, 3,
                                       0x6000, 0x7000, 8, None) == _lib.ENGRAM_EINVAL


def test_forward_ids_validation(lib):
    d = desc()
    w = _lib.EngramWeights(0x10000, 0x20000, 0x30000, 0x40000, 0x50000)
    n16 = lib.engram_forward_workspace_size(ctypes.byref(d), 16)

    def call(ids=0x8000, M=16, ws=0x1000000, nbytes=None, wts=w):
        return lib.engram_forward_ids(ctypes.byref(d), None if wts is None else ctypes.byref(wts),
                                      0x100000, ids, M, None, 0x900000, None, None, ws,
                                      n16 if nbytes is None else nbytes, None)

    assert call(M=-1) == _lib.ENGRAM_EINVAL
    assert call(wts=None) == _lib.ENGRAM_EINVAL
    assert call(nbytes=64) == _lib.ENGRAM_EINVAL and b"workspace" in lib.engram_last_error()
    assert call(ids=None) == _lib.ENGRAM_EINVAL and b"hash_ids" in lib.engram_last_error()
    assert call(ids=0x8002) == _lib.ENGRAM_EINVAL                       # misaligned ids
    assert call(ids=0x1000000) == _lib.ENGRAM_EINVAL                    # ids inside the workspace
    assert call(M=0, ids=None) == _lib.ENGRAM_OK                        # nothing to do
