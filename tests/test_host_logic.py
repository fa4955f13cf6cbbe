"""Host-side rules of the CUDA library that need no GPU, compiled with g++
from the library's own internal header: the backward's super-batch size (how
many (batch, kv head) groups fa_bwd_main runs together, key tile slowest
within each)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tiled_attention_05_gb300", "csrc")
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")

PROGRAM = r"""
#include <cstdio>
#include "fa_internal.h"
int main() {
  const int sms_list[] = {1, 148, 152, 200};
  const int kv_list[] = {1, 2, 3, 16, 63, 64, 100, 256};
  for (int sms : sms_list)
    for (int kv : kv_list)
      for (int g = 1; g <= 300; ++g) std::printf("%d %d %d %d\n", g, kv, sms, fa::super_batch_groups(g, kv, sms));
  return 0;
}
"""


@pytest.fixture(scope="module")
def rule_table(tmp_path_factory):
    if shutil.which("g++") is None or not os.path.exists(os.path.join(CUDA_INC, "cuda.h")):
        pytest.skip("needs g++ and the CUDA headers")
    d = tmp_path_factory.mktemp("host_logic")
    src, exe = d / "rule.cpp", d / "rule"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-std=c++17", "-O1", f"-I{CSRC}", f"-I{CUDA_INC}", str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return [tuple(map(int, ln.split())) for ln in out.splitlines()]


def test_super_batch_divides_the_group_count(rule_table):
    for g, kv, sms, s in rule_table:
        assert 1 <= s <= g and g % s == 0, (g, kv, sms, s)


def test_super_batch_fills_the_gpu_and_is_the_smallest_such_divisor(rule_table):
    for g, kv, sms, s in rule_table:
        want = (3 * sms + 1) // 2          # 1.5 CTAs per SM, rounded up
        s_min = max(1, -(-want // kv))     # fewest groups whose key tiles reach it
        fits = [x for x in range(s_min, min(g - 1, 4 * s_min) + 1) if g % x == 0]
        if fits:
            assert s == fits[0], (g, kv, sms, s)
            assert s * kv >= want
        else:
            assert s == g, (g, kv, sms, s)  # one super-batch: every group at once


def test_super_batch_on_the_measured_workloads(rule_table):
    table = {(g, kv, sms): s for g, kv, sms, s in rule_table}
    assert table[(16, 64, 152)] == 4    # B=2, Hkv=8, T=8192: 4 of 16 groups at a time
    assert table[(16, 256, 152)] == 1   # B=1, Hkv=16, T=32768: one group fills the GPU
    assert table[(64, 16, 152)] == 16   # B=4, H=16, T=2048
    assert table[(8, 64, 152)] == 4     # sliding window, B=1, Hkv=8, T=8192
    assert table[(1, 2, 152)] == 1
