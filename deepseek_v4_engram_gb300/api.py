"""Thin Python binding of libengram.so: the entry points of include/engram.h under the same names.

Argument marshalling only. Tensors must be CUDA tensors, contiguous, of the element size the C
ABI expects (bf16 may be passed as torch.bfloat16 or as int16/uint16 bits). Every computation
runs in the library's kernels; if the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field

import torch

from . import _lib
from ._lib import EngramDesc, EngramLayerHash, EngramTables, EngramWeights


class EngramError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"engram status {code}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    return _lib.load()


def _check(rc: int) -> None:
    if rc != _lib.ENGRAM_OK:
        raise EngramError(rc, lib().engram_last_error().decode())


_ITEMSIZE = {"bf16": 2, "u8": 1, "i32": 4, "u64": 8, "i64": 8, "f32": 4}


def _ptr(t: torch.Tensor | None, kind: str, name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (the library takes device pointers)")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.element_size() != _ITEMSIZE[kind]:
        raise ValueError(f"{name}: element size {t.element_size()} != {_ITEMSIZE[kind]} ({kind})")
    return t.data_ptr()


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_desc(dim, hc_mult, n_heads, max_ngram_size, head_dim, num_embeddings,
              norm_eps=1e-6) -> EngramDesc:
    return EngramDesc(dim, hc_mult, n_heads, max_ngram_size, head_dim, 0, num_embeddings,
                      norm_eps)


@dataclass
class DeviceTables:
    """Hash tables on the device plus the C struct pointing at them (keeps the tensors alive)."""

    token_map: torch.Tensor
    pad_id: int
    multipliers: torch.Tensor
    primes: torch.Tensor
    offsets: torch.Tensor
    c: EngramTables = field(init=False)

    def __post_init__(self):
        self.c = EngramTables(_ptr(self.token_map, "i32", "token_map"), self.token_map.numel(),
                              self.pad_id, _ptr(self.multipliers, "u64", "multipliers"),
                              _ptr(self.primes, "u64", "primes"),
                              _ptr(self.offsets, "i64", "offsets"))


@dataclass
class DeviceWeights:
    """Layer parameters on the device plus the C struct pointing at them."""

    table: torch.Tensor
    scales: torch.Tensor
    wkv: torch.Tensor
    q_weight: torch.Tensor
    k_weight: torch.Tensor
    c: EngramWeights = field(init=False)

    def __post_init__(self):
        self.c = EngramWeights(_ptr(self.table, "u8", "table"), _ptr(self.scales, "u8", "scales"),
                               _ptr(self.wkv, "bf16", "wkv"), _ptr(self.q_weight, "bf16", "q"),
                               _ptr(self.k_weight, "bf16", "k"))


def engram_check_errors(stream=None) -> int:
    """Synchronise the stream; return the device error word (cleared). Raises on CUDA failure."""
    bits = ctypes.c_uint32(0)
    rc = lib().engram_check_errors(_stream(stream), ctypes.byref(bits))
    if rc in (_lib.ENGRAM_OK, _lib.ENGRAM_EDEVICE, _lib.ENGRAM_ECAPACITY):
        return bits.value
    _check(rc)
    return bits.value


def engram_hash(desc, tables: DeviceTables, tokens, cache, cache_len, hash_ids, stream=None):
    B, T = tokens.shape
    _check(lib().engram_hash(ctypes.byref(desc), ctypes.byref(tables.c),
                             _ptr(tokens, "i32", "tokens"), B, T, _ptr(cache, "i32", "cache"),
                             _ptr(cache_len, "i32", "cache_len"), cache.shape[1],
                             _ptr(hash_ids, "i32", "hash_ids"), _stream(stream)))


@dataclass
class DeviceLayerHash:
    """One Engram layer's hash constants, table and outputs for engram_hash_rows_layers."""

    multipliers: torch.Tensor
    primes: torch.Tensor
    offsets: torch.Tensor
    table: torch.Tensor
    scales: torch.Tensor
    rows: torch.Tensor
    hash_ids: torch.Tensor | None = None
    c: EngramLayerHash = field(init=False)

    def __post_init__(self):
        self.c = EngramLayerHash(_ptr(self.multipliers, "u64", "multipliers"),
                                 _ptr(self.primes, "u64", "primes"),
                                 _ptr(self.offsets, "i64", "offsets"), self.table.shape[0],
                                 _ptr(self.table, "u8", "table"), _ptr(self.scales, "u8", "scales"),
                                 _ptr(self.rows, "bf16", "rows"),
                                 _ptr(self.hash_ids, "i32", "hash_ids"))


def engram_hash_rows_layers(desc, tables: DeviceTables, layers, tokens, cache, cache_len,
                            stream=None):
    """Stages 1 + 2 for several layers (a list of DeviceLayerHash) in one launch."""
    B, T = tokens.shape
    arr = (EngramLayerHash * max(len(layers), 1))(*[lh.c for lh in layers])
    _check(lib().engram_hash_rows_layers(
        ctypes.byref(desc), ctypes.byref(tables.c), arr, len(layers),
        _ptr(tokens, "i32", "tokens"), B, T, _ptr(cache, "i32", "cache"),
        _ptr(cache_len, "i32", "cache_len"), cache.shape[1], _stream(stream)))


def engram_embed_rows(desc, table, scales, ids, out, stream=None):
    _check(lib().engram_embed_rows(ctypes.byref(desc), _ptr(table, "u8", "table"),
                                   _ptr(scales, "u8", "scales"), _ptr(ids, "i32", "ids"),
                                   ids.numel(), _ptr(out, "bf16", "out"), _stream(stream)))


def engram_embed_rows_shard(desc, table_shard, scales_shard, row_begin: int, ids, out,
                            stream=None):
    shard_rows = 0 if table_shard is None else table_shard.shape[0]
    _check(lib().engram_embed_rows_shard(ctypes.byref(desc), _ptr(table_shard, "u8", "table_shard"),
                                         _ptr(scales_shard, "u8", "scales_shard"), row_begin,
                                         shard_rows, _ptr(ids, "i32", "ids"), ids.numel(),
                                         _ptr(out, "bf16", "out"), _stream(stream)))


def engram_probe_stream_read(buf, method: int, stream=None):
    """One read of `buf` (a contiguous CUDA tensor) over every SM: 0 bulk copies, 1 plain loads,
    2 bulk copies with an L2 evict-first policy."""
    if not (isinstance(buf, torch.Tensor) and buf.is_cuda and buf.is_contiguous()):
        raise TypeError("buf: expected a contiguous CUDA tensor")
    _check(lib().engram_probe_stream_read(ctypes.c_void_p(buf.data_ptr()),
                                          buf.numel() * buf.element_size(), method,
                                          _stream(stream)))


def engram_wkv(a, w, kv, stream=None):
    M, K = a.shape
    N = w.shape[0]
    _check(lib().engram_wkv(_ptr(a, "bf16", "a"), _ptr(w, "bf16", "w"), _ptr(kv, "bf16", "kv"),
                            M, N, K, _stream(stream)))


def engram_gate_and_add(desc, x, kv, q_weight, k_weight, token_mask, out, gate_out=None,
                        stream=None):
    M = x.shape[0]
    _check(lib().engram_gate_and_add(ctypes.byref(desc), _ptr(x, "bf16", "x"),
                                     _ptr(kv, "bf16", "kv"), _ptr(q_weight, "bf16", "q"),
                                     _ptr(k_weight, "bf16", "k"),
                                     _ptr(token_mask, "u8", "token_mask"), _ptr(out, "bf16", "out"),
                                     _ptr(gate_out, "f32", "gate_out"), M, _stream(stream)))


def engram_wkv_gate_workspace_size(desc, M: int) -> int:
    return int(lib().engram_wkv_gate_workspace_size(ctypes.byref(desc), M))


def engram_wkv_gate(desc, rows, wkv, x, q_weight, k_weight, token_mask, out, gate_out=None,
                    kv_out=None, workspace=None, stream=None):
    """Stages 3 + 4 in one kernel. `workspace` (uint8 CUDA tensor) defaults to a fresh one."""
    M = x.shape[0]
    if workspace is None:
        workspace = torch.empty(max(engram_wkv_gate_workspace_size(desc, M), 256),
                                dtype=torch.uint8, device=x.device)
    _check(lib().engram_wkv_gate(ctypes.byref(desc), _ptr(rows, "bf16", "rows"),
                                 _ptr(wkv, "bf16", "wkv"), _ptr(x, "bf16", "x"),
                                 _ptr(q_weight, "bf16", "q"), _ptr(k_weight, "bf16", "k"),
                                 _ptr(token_mask, "u8", "token_mask"), _ptr(out, "bf16", "out"),
                                 _ptr(gate_out, "f32", "gate_out"), _ptr(kv_out, "bf16", "kv_out"),
                                 M, _ptr(workspace, "u8", "workspace"), workspace.numel(),
                                 _stream(stream)))


def engram_forward_workspace_size(desc, M: int) -> int:
    return int(lib().engram_forward_workspace_size(ctypes.byref(desc), M))


def engram_forward(desc, tables: DeviceTables, weights: DeviceWeights, x, tokens, cache,
                   cache_len, token_mask, out, workspace, hash_ids_out=None, gate_out=None,
                   kv_out=None, stream=None):
    B, T = tokens.shape
    _check(lib().engram_forward(
        ctypes.byref(desc), ctypes.byref(tables.c), ctypes.byref(weights.c), _ptr(x, "bf16", "x"),
        _ptr(tokens, "i32", "tokens"), B, T, _ptr(cache, "i32", "cache"),
        _ptr(cache_len, "i32", "cache_len"), cache.shape[1],
        _ptr(token_mask, "u8", "token_mask"), _ptr(out, "bf16", "out"),
        _ptr(hash_ids_out, "i32", "hash_ids_out"), _ptr(gate_out, "f32", "gate_out"),
        _ptr(kv_out, "bf16", "kv_out"), _ptr(workspace, "u8", "workspace"), workspace.numel(),
        _stream(stream)))


class EngramGraph:
    """engram_forward captured once as a library-owned CUDA graph (engram_forward_graph_create);
    launch() replays it. The tensors given at creation are kept referenced: refill x and tokens
    in place between launches."""

    def __init__(self, desc, tables: DeviceTables, weights: DeviceWeights, x, tokens, cache,
                 cache_len, token_mask, out, workspace, hash_ids_out=None, gate_out=None,
                 kv_out=None):
        B, T = tokens.shape
        handle = ctypes.c_void_p()
        _check(lib().engram_forward_graph_create(
            ctypes.byref(desc), ctypes.byref(tables.c), ctypes.byref(weights.c),
            _ptr(x, "bf16", "x"), _ptr(tokens, "i32", "tokens"), B, T,
            _ptr(cache, "i32", "cache"), _ptr(cache_len, "i32", "cache_len"), cache.shape[1],
            _ptr(token_mask, "u8", "token_mask"), _ptr(out, "bf16", "out"),
            _ptr(hash_ids_out, "i32", "hash_ids_out"), _ptr(gate_out, "f32", "gate_out"),
            _ptr(kv_out, "bf16", "kv_out"), _ptr(workspace, "u8", "workspace"),
            workspace.numel(), ctypes.byref(handle)))
        self._handle = handle
        self._keep = (desc, tables, weights, x, tokens, cache, cache_len, token_mask, out,
                      workspace, hash_ids_out, gate_out, kv_out)

    def launch(self, stream=None):
        if not self._handle:
            raise EngramError(_lib.ENGRAM_EINVAL, "graph destroyed")
        _check(lib().engram_graph_launch(self._handle, _stream(stream)))

    def destroy(self):
        if self._handle:
            lib().engram_graph_destroy(self._handle)
            self._handle = ctypes.c_void_p()
            self._keep = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def engram_forward_ids(desc, weights: DeviceWeights, x, hash_ids, token_mask, out, workspace,
                       gate_out=None, kv_out=None, stream=None):
    """Stages 2-4 from given hash ids [M, n_hash_cols] (the listing's forward(x, hash_ids, mask))."""
    M = hash_ids.shape[0]
    _check(lib().engram_forward_ids(
        ctypes.byref(desc), ctypes.byref(weights.c), _ptr(x, "bf16", "x"),
        _ptr(hash_ids, "i32", "hash_ids"), M, _ptr(token_mask, "u8", "token_mask"),
        _ptr(out, "bf16", "out"), _ptr(gate_out, "f32", "gate_out"),
        _ptr(kv_out, "bf16", "kv_out"), _ptr(workspace, "u8", "workspace"), workspace.numel(),
        _stream(stream)))


def engram_forward_noalloc(desc, tables: DeviceTables, weights: DeviceWeights, x, tokens, cache,
                           cache_len, token_mask, out, hash_ids_out=None, gate_out=None,
                           kv_out=None, stream=None):
    """engram_forward with the library's own fixed scratch instead of a workspace argument."""
    B, T = tokens.shape
    _check(lib().engram_forward_noalloc(
        ctypes.byref(desc), ctypes.byref(tables.c), ctypes.byref(weights.c), _ptr(x, "bf16", "x"),
        _ptr(tokens, "i32", "tokens"), B, T, _ptr(cache, "i32", "cache"),
        _ptr(cache_len, "i32", "cache_len"), cache.shape[1],
        _ptr(token_mask, "u8", "token_mask"), _ptr(out, "bf16", "out"),
        _ptr(hash_ids_out, "i32", "hash_ids_out"), _ptr(gate_out, "f32", "gate_out"),
        _ptr(kv_out, "bf16", "kv_out"), _stream(stream)))
