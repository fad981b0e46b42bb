"""Host checks of the benchmark (no GPU): the reference arm's JSON line, the roofline arithmetic and
the tie between the recorded DRAM traffic and the sources of the kernel it was measured on."""
import json
import os
import shutil
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PEAKS = {"hbm_gbs": 6701.8, "bf16_tflops": 1921.1, "bf16_tflops_sustained": 1731.1}


def test_reference_arm_prints_one_json_line_with_the_contract_keys():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert (d["steps"], d["warmup"]) == (1, 0)
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["seq_len"] == 4096 and d["config"]["global_batch"] == 1


def test_roofline_bound_switches_at_the_crossover():
    # time = max(FLOP / bf16 peak, bytes / HBM peak); the bound is whichever is larger
    per_tok_flop = bench.FLOPS_PER_TOKEN / (PEAKS["bf16_tflops"] * 1e12)
    per_tok_byte = bench.BYTES_PER_TOKEN / (PEAKS["hbm_gbs"] * 1e9)
    w = bench.WKV_BYTES / (PEAKS["hbm_gbs"] * 1e9)
    cross = w / (per_tok_flop - per_tok_byte)     # tokens where the two times meet
    assert 400 < cross < 420                      # 412 at these peaks
    lo, hi = int(cross) - 5, int(cross) + 5
    assert bench.roofline_of(lo, 1.0, PEAKS)[0] == "hbm"
    assert bench.roofline_of(hi, 1.0, PEAKS)[0] == "tensor"
    # a step that takes exactly the roofline time is at fraction 1
    for M in (1, 64, 4096):
        t = max(per_tok_flop * M, per_tok_byte * M + w)
        assert abs(bench.roofline_of(M, t * 1e3, PEAKS)[1] - 1.0) < 1e-9


def test_traffic_record_is_tied_to_the_kernel_sources(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    sources = rec["engram_fused_kernel"]["sources"]
    # a copy of the sources and the record: the record applies while they are unchanged
    for src in sources + ["profiles/ncu_traffic.json"]:
        dst = tmp_path / src
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(ROOT, src), dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    got = bench.kernel_traffic("engram_fused_kernel")
    assert got == {"bytes_per_launch": rec["engram_fused_kernel"]["bytes_per_launch"],
                   "tokens_per_launch": rec["engram_fused_kernel"]["tokens"]}
    # any change to a source file voids it
    with open(tmp_path / sources[0], "a") as f:
        f.write("\n")
    assert bench.kernel_traffic("engram_fused_kernel") is None
    assert bench.kernel_traffic("no_such_kernel") is None
