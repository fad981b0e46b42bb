"""GPU: engram_forward captured as a library-owned CUDA graph (engram_forward_graph_create,
engram_graph_launch). A replay must do exactly what one engram_forward call with the creation's
arguments does: the same bits in out, gate and hash ids, and the same cache and cache lengths,
step after step with the inputs refilled in place."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import deepseek_v4_engram_gb300 as eg
import synth
from tests.helpers import dev, empty_bf16, host

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WIDE = synth.Geometry(dim=5120, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=64,
                      vocab=129280, n_compressed=100000, prime_floor=1 << 14)


@pytest.fixture(scope="module")
def wide():
    from tests.gpu_fixtures import DeviceModel
    return DeviceModel(synth.make_model(WIDE, synth.BASE_SEED + 51, scale_mode="pow2"))


class Step:
    """The buffers of one engram_forward step shape."""

    def __init__(self, dm, B, T, cache, length):
        g = dm.geom
        self.x = torch.empty((B, T, g.hc_mult, g.dim), dtype=torch.int16, device="cuda")
        self.tokens = torch.empty((B, T), dtype=torch.int32, device="cuda")
        self.mask = torch.ones((B, T), dtype=torch.uint8, device="cuda")
        self.out = empty_bf16(B, T, g.hc_mult, g.dim)
        self.ids = torch.full((B, T, g.n_hash_cols), -1, dtype=torch.int32, device="cuda")
        self.gate = torch.full((B, T, g.hc_mult), float("nan"), device="cuda")
        self.ws = dm.workspace(B * T)
        self.cache, self.length = cache, length

    def fill(self, batch):
        self.x.copy_(dev(batch.x))
        self.tokens.copy_(dev(batch.tokens))
        self.mask.copy_(dev(batch.mask.astype(np.uint8)))

    def args(self):
        return (self.x, self.tokens, self.cache, self.length, self.mask, self.out, self.ws)

    def result(self):
        return [host(t) for t in (self.out, self.ids, self.gate, self.cache, self.length)]


def prefilled(dm, B, prefill, capacity, seed):
    cache, length = dm.new_cache(B, capacity)
    if prefill:
        b = synth.make_batch(dm.geom, B, prefill, seed)
        out = empty_bf16(B, prefill, dm.geom.hc_mult, dm.geom.dim)
        eg.engram_forward(dm.desc, dm.tables, dm.weights, dev(b.x), dev(b.tokens), cache, length,
                          None, out, dm.workspace(B * prefill))
    return cache, length


@pytest.mark.parametrize("B,T,prefill,steps", [(64, 1, 40, 5), (3, 1, 0, 4), (1, 700, 5, 2),
                                               (2, 150, 0, 2)])
def test_graph_replays_equal_forward_calls(wide, B, T, prefill, steps):
    dm = wide
    cap = prefill + T * steps + 3
    graph_step = Step(dm, B, T, *prefilled(dm, B, prefill, cap, synth.BASE_SEED + 600))
    call_step = Step(dm, B, T, *prefilled(dm, B, prefill, cap, synth.BASE_SEED + 600))
    x, tok, cache, length, mask, out, ws = graph_step.args()
    g = eg.EngramGraph(dm.desc, dm.tables, dm.weights, x, tok, cache, length, mask, out, ws,
                       hash_ids_out=graph_step.ids, gate_out=graph_step.gate)
    try:
        for i in range(steps):
            batch = synth.make_batch(dm.geom, B, T, synth.BASE_SEED + 610 + i, mask_frac=0.2)
            graph_step.fill(batch)
            g.launch()
            call_step.fill(batch)
            x, tok, cache, length, mask, out, ws = call_step.args()
            eg.engram_forward(dm.desc, dm.tables, dm.weights, x, tok, cache, length, mask, out,
                              ws, hash_ids_out=call_step.ids, gate_out=call_step.gate)
            assert eg.engram_check_errors() == 0
            for a, r in zip(graph_step.result(), call_step.result()):
                np.testing.assert_array_equal(a, r)
        np.testing.assert_array_equal(host(graph_step.length), prefill + T * steps)
    finally:
        g.destroy()


def test_graph_creation_validates_like_forward(wide):
    dm = wide
    st = Step(dm, 2, 1, *dm.new_cache(2, 4))
    x, tok, cache, length, mask, out, ws = st.args()
    with pytest.raises(eg.EngramError) as e:   # a workspace too small for any path
        eg.EngramGraph(dm.desc, dm.tables, dm.weights, x, tok, cache, length, mask, out, ws[:64])
    assert e.value.code == 1
    g = eg.EngramGraph(dm.desc, dm.tables, dm.weights, x, tok, cache, length, mask, out, ws)
    g.destroy()
    with pytest.raises(eg.EngramError):
        g.launch()
    assert eg.engram_check_errors() == 0
    np.testing.assert_array_equal(host(length), [0, 0])   # creation runs no kernel


def test_graph_as_first_call_of_a_process():
    # creating the graph is the first thing the process does with the library (nothing loaded)
    code = (
        "import numpy as np, torch, synth, deepseek_v4_engram_gb300 as eg\n"
        "from tests.gpu_fixtures import DeviceModel\n"
        "from tests.helpers import dev\n"
        "dm = DeviceModel(synth.make_model(synth.TINY, synth.BASE_SEED))\n"
        "b = synth.make_batch(dm.geom, 2, 3, synth.BASE_SEED + 7)\n"
        "x, tok = dev(b.x), dev(b.tokens)\n"
        "cache, length = dm.new_cache(2, 8)\n"
        "out = torch.empty_like(x)\n"
        "g = eg.EngramGraph(dm.desc, dm.tables, dm.weights, x, tok, cache, length, None, out,\n"
        "                   dm.workspace(6))\n"
        "g.launch()\n"
        "assert eg.engram_check_errors() == 0\n"
        "assert length.tolist() == [3, 3]\n"
        "g.destroy()\n"
        "print('ok')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-2000:]
