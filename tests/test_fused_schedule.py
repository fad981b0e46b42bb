"""Host check of the fused kernel's work-item order (no GPU): the header is compiled with g++ into a
small program that enumerates the order for many shapes and checks that it is a permutation of
every (token tile, column tile) item and that every value item comes after all the key items of
its token tile (the only wait in the kernel: a value item needs that tile's gates). With that, a
persistent grid whose pairs take items in order cannot deadlock."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "deepseek_v4_engram_gb300", "csrc")

PROGRAM = r"""
#define __host__
#define __device__
#include "fused_schedule.cuh"
#include <cstdio>
#include <vector>
using namespace engram;

static long check(int mt, int nk, int nv, int pairs) {
  FusedSchedule s = make_fused_schedule(mt, nk, nv, pairs);
  if (s.items != (long)mt * (nk + nv)) return 1;
  std::vector<long> pos((size_t)mt * (nk + nv), -1), last_key(mt, -1), first_val(mt, 1L << 60);
  long bad = 0;
  for (long i = 0; i < s.items; ++i) {
    FusedItem it = fused_item_at(s, i);
    if (it.mt < 0 || it.mt >= mt || it.col < 0 || it.col >= (it.value ? nv : nk)) {
      if (bad++ < 3) printf("bad item %ld\n", i);
      continue;
    }
    long& p = pos[(size_t)it.mt * (nk + nv) + (it.value ? nk + it.col : it.col)];
    if (p >= 0 && bad++ < 3) printf("item repeated at %ld\n", i);
    p = i;
    if (it.value) { if (i < first_val[it.mt]) first_val[it.mt] = i; }
    else last_key[it.mt] = i;
  }
  for (long p : pos) if (p < 0) ++bad;
  for (int t = 0; t < mt; ++t)
    if (first_val[t] <= last_key[t] && bad++ < 3) printf("tile %d: value before key\n", t);
  return bad;
}

int main() {
  long bad = 0, cases = 0;
  for (int mt : {1, 2, 3, 5, 8, 9, 16, 17, 31, 33, 64, 256})
    for (int hc : {1, 2, 4, 8})
      for (int nv : {1, 3, 20})
        for (int pairs : {1, 7, 76}) {
          bad += check(mt, hc * nv, nv, pairs);
          ++cases;
        }
  FusedSchedule s = make_fused_schedule(16, 80, 20, 76);
  printf("cases=%ld bad=%ld group=%d groups=%d items=%ld\n", cases, bad, s.group, s.groups,
         (long)s.items);
  return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_fused_item_order_is_a_valid_permutation(tmp_path):
    src = tmp_path / "check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "check"
    subprocess.run(["g++", "-std=c++17", "-O2", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    fields = dict(kv.split("=") for kv in r.stdout.split())
    assert fields["bad"] == "0"
    # 4096 tokens at hc 4, dim 5120 on 76 pairs: two groups of eight 256-token tiles
    assert (fields["group"], fields["groups"], fields["items"]) == ("8", "2", "1600")
