"""Host logic of the persistent kernels' unit order: the head-group size that the
launchers choose (grid_aligned_group in csrc/fa_internal.h), compiled here with g++
against the real header and checked against hand-worked cases and its defining
property.  No GPU is needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_io_aware_05_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

CASES = [(24, 16, 152), (40, 16, 152), (20, 32, 152), (12, 32, 152), (2, 32, 64), (1, 32, 152),
         (0, 32, 152), (256, 32, 152), (5, 256, 152), (7, 10, 35), (9, 4, 0)]

PROGRAM = r"""
#include "fa_internal.h"
#include <cstdio>
int main() {
    const int cases[][3] = {%s};
    for (const auto &c : cases)
        std::printf("%%d\n", fa::grid_aligned_group(c[0], c[1], c[2]));
    return 0;
}
"""


@pytest.fixture(scope="module")
def chosen(tmp_path_factory):
    if shutil.which("g++") is None or not os.path.isdir(CUDA_INC):
        pytest.skip("g++ or the CUDA headers are not available")
    d = tmp_path_factory.mktemp("sched")
    src = d / "sched.cpp"
    src.write_text(PROGRAM % ", ".join("{%d, %d, %d}" % c for c in CASES))
    exe = d / "sched"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, "-I", CUDA_INC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    return dict(zip(CASES, map(int, out)))


def test_worked_cases(chosen):
    # B8 H32 N4096 d128: forward levels = 16 query-tile pairs, backward levels = 32 key blocks
    assert chosen[(24, 16, 152)] == 19     # 19 * 16 = 304 = 2 passes of 152
    assert chosen[(40, 16, 152)] == 38     # 38 * 16 = 608 = 4 passes
    assert chosen[(20, 32, 152)] == 19     # 19 * 32 = 608
    assert chosen[(12, 32, 152)] == 12     # no size in [6, 12] is a whole number of passes
    assert chosen[(2, 32, 64)] == 2
    assert chosen[(1, 32, 152)] == 1
    assert chosen[(0, 32, 152)] == 1       # at least one head per group
    assert chosen[(256, 32, 152)] == 247   # 247 * 32 = 7904 = 52 passes
    assert chosen[(9, 4, 0)] == 9          # no grid: the budget's size


def test_defining_property(chosen):
    for (gmax, levels, grid), g in chosen.items():
        top = max(gmax, 1)
        aligned = [c for c in range(top, 0, -1) if 2 * c >= top and grid > 0 and (c * levels) % grid == 0]
        assert g == (aligned[0] if aligned else top), (gmax, levels, grid, g)
