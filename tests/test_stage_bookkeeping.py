"""Host-side unit test of the staging-ring bookkeeping the tcgen05 multi-token kernel
uses when it stops early: for each stage, which fill was issued last and which mbarrier
phase parity that fill completes.  The header is compiled with g++ into a small program
and its answers are checked against a direct simulation of the ring."""
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "paged_kv_cache_197_gb300" / "csrc" / "pa_stages.h"

PROGRAM = r"""
#include <cstdio>
#include "pa_stages.h"
int main() {
    for (int stages = 1; stages <= 6; ++stages)
        for (int issued = 0; issued <= 40; ++issued)
            for (int st = -1; st <= stages; ++st) {
                pa::StageFill f = pa::last_fill(issued, stages, st);
                std::printf("%d %d %d %d %u\n", stages, issued, st, f.any ? 1 : 0, f.parity);
            }
    return 0;
}
"""


def simulate(stages, issued, st):
    """Issue tiles 0..issued-1 into the ring; each fill of a stage flips its phase."""
    if st < 0 or st >= stages:
        return 0, 0
    fills = [t // stages for t in range(issued) if t % stages == st]
    if not fills:
        return 0, 0
    return 1, fills[-1] & 1


def test_last_fill_matches_simulation(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("needs a C++ compiler")
    src = tmp_path / "stages.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "stages"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", str(HEADER.parent), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    rows = [list(map(int, line.split())) for line in out.splitlines()]
    assert len(rows) == sum(41 * (s + 2) for s in range(1, 7))
    for stages, issued, st, anyf, parity in rows:
        assert (anyf, parity) == simulate(stages, issued, st), (stages, issued, st)
