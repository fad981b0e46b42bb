"""GB300 (sm_103a) Engram forward path of DeepSeek V4.1 behind a C ABI (libengram.so).

Importing the package loads nothing; the library is loaded on the first call and must have been
built (``python -m deepseek_v4_engram_gb300.build``). There is no CPU fallback.
"""
from .api import (DeviceLayerHash, DeviceTables, DeviceWeights, EngramError, EngramGraph,  # noqa: F401,E501
                  engram_check_errors, engram_embed_rows, engram_embed_rows_shard,
                  engram_forward, engram_forward_ids,
                  engram_forward_noalloc,
                  engram_forward_workspace_size, engram_gate_and_add, engram_hash,
                  engram_hash_rows_layers, engram_wkv, engram_wkv_gate,
                  engram_wkv_gate_workspace_size, make_desc)
from .shard import embed_rows_sharded, exchange_rows, row_owner, table_shard_range  # noqa: F401
