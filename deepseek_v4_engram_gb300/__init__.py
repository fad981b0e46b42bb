"""GB300 (sm_103a) Engram forward path of DeepSeek V4.1 behind a C ABI (libengram.so).

Importing the package loads nothing; the library is loaded on the first call and must have been
built (``python -m deepseek_v4_engram_gb300.build``). There is no CPU fallback.
"""
from .api import (DeviceTables, DeviceWeights, EngramError, engram_check_errors,  # noqa: F401
                  engram_embed_rows, engram_forward, engram_forward_workspace_size, engram_gate_and_add,
                  engram_hash, engram_wkv, engram_wkv_gate, make_desc)
