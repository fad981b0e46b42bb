"""Device-side copies of synthetic models and batches for the GPU tests and the benchmark."""
from __future__ import annotations

import numpy as np
import torch

import deepseek_v4_engram_gb300 as eg
import synth

from tests.helpers import dev


class DeviceModel:
    def __init__(self, model: synth.Model):
        g = model.geom
        t = model.tables
        self.model = model
        self.geom = g
        self.desc = eg.make_desc(g.dim, g.hc_mult, g.n_heads, g.max_ngram_size, g.head_dim,
                                 t.num_embeddings, model.eps)
        self.tables = eg.DeviceTables(dev(t.token_map), t.pad_id, dev(t.multipliers),
                                      dev(t.primes), dev(t.offsets))
        self.weights = eg.DeviceWeights(dev(model.table), dev(model.scales), dev(model.wkv),
                                        dev(model.q), dev(model.k))

    def new_cache(self, B: int, capacity: int):
        cache = torch.zeros((B, capacity), dtype=torch.int32, device="cuda")
        length = torch.zeros(B, dtype=torch.int32, device="cuda")
        return cache, length

    def workspace(self, M: int) -> torch.Tensor:
        n = eg.engram_forward_workspace_size(self.desc, M)
        return torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
