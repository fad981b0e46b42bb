"""ctypes view of libengram.so: the structs and entry points of include/engram.h, nothing more."""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libengram.so")

ENGRAM_OK = 0
ENGRAM_EINVAL = 1
ENGRAM_ECAPACITY = 2
ENGRAM_ECUDA = 3
ENGRAM_EDEVICE = 4
ENGRAM_EUNSUPPORTED = 5

DEVERR_TOKEN_RANGE = 1
DEVERR_CACHE_FULL = 2
DEVERR_ID_RANGE = 4
DEVERR_WAIT_TIMEOUT = 8


class EngramDesc(ctypes.Structure):
    _fields_ = [("dim", ctypes.c_int32), ("hc_mult", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("max_ngram_size", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("num_embeddings", ctypes.c_int64), ("norm_eps", ctypes.c_float)]


class EngramTables(ctypes.Structure):
    _fields_ = [("token_map", ctypes.c_void_p), ("vocab", ctypes.c_int32),
                ("pad_id", ctypes.c_int32), ("multipliers", ctypes.c_void_p),
                ("primes", ctypes.c_void_p), ("offsets", ctypes.c_void_p)]


class EngramWeights(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("wkv", ctypes.c_void_p), ("q_weight", ctypes.c_void_p),
                ("k_weight", ctypes.c_void_p)]


class EngramLayerHash(ctypes.Structure):
    _fields_ = [("multipliers", ctypes.c_void_p), ("primes", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("num_embeddings", ctypes.c_int64),
                ("table", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("rows", ctypes.c_void_p), ("hash_ids", ctypes.c_void_p)]


MAX_HASH_LAYERS = 16

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_DESC = ctypes.POINTER(EngramDesc)
_TAB = ctypes.POINTER(EngramTables)
_WTS = ctypes.POINTER(EngramWeights)

# name -> (restype, argtypes); the same names as include/engram.h
SIGNATURES = {
    "engram_last_error": (ctypes.c_char_p, []),
    "engram_abi_version": (_I32, []),
    "engram_check_errors": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "engram_hash": (ctypes.c_int, [_DESC, _TAB, _P, _I32, _I32, _P, _P, _I32, _P, _P]),
    "engram_hash_rows_layers": (ctypes.c_int, [_DESC, _TAB, ctypes.POINTER(EngramLayerHash), _I32,
                                               _P, _I32, _I32, _P, _P, _I32, _P]),
    "engram_embed_rows": (ctypes.c_int, [_DESC, _P, _P, _P, _I64, _P, _P]),
    "engram_embed_rows_shard": (ctypes.c_int, [_DESC, _P, _P, _I64, _I64, _P, _I64, _P, _P]),
    "engram_probe_stream_read": (ctypes.c_int, [_P, _SZ, _I32, _P]),
    "engram_forward_graph_create": (ctypes.c_int, [_DESC, _TAB, _WTS, _P, _P, _I32, _I32, _P, _P,
                                                   _I32, _P, _P, _P, _P, _P, _P, _SZ,
                                                   ctypes.POINTER(ctypes.c_void_p)]),
    "engram_graph_launch": (ctypes.c_int, [_P, _P]),
    "engram_graph_destroy": (ctypes.c_int, [_P]),
    "engram_wkv": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _I32, _P]),
    "engram_gate_and_add": (ctypes.c_int, [_DESC, _P, _P, _P, _P, _P, _P, _P, _I64, _P]),
    "engram_wkv_gate_workspace_size": (_SZ, [_DESC, _I64]),
    "engram_wkv_gate": (ctypes.c_int, [_DESC, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _SZ,
                                       _P]),
    "engram_forward_workspace_size": (_SZ, [_DESC, _I64]),
    "engram_forward": (ctypes.c_int, [_DESC, _TAB, _WTS, _P, _P, _I32, _I32, _P, _P, _I32, _P,
                                      _P, _P, _P, _P, _P, _SZ, _P]),
    "engram_forward_ids": (ctypes.c_int, [_DESC, _WTS, _P, _P, _I64, _P, _P, _P, _P, _P, _SZ,
                                          _P]),
    "engram_forward_noalloc": (ctypes.c_int, [_DESC, _TAB, _WTS, _P, _P, _I32, _I32, _P, _P,
                                              _I32, _P, _P, _P, _P, _P, _P]),
}

NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the in-tree library (build it with deepseek_v4_engram_gb300.build first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: the Engram CUDA library is not built "
            "(run `python -m deepseek_v4_engram_gb300.build`). There is no fallback path.")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
