"""Host check of the tensor-core sweeps' work-unit schedule.

`sched_check.cpp` includes the schedule header the kernel uses
(`all_pairs_distance_gb300/csrc/tc_schedule.h`), enumerates every unit of the
count's triangle, the union's distance bands (three, or one for small
problems) and the border's rectangle, with one and with two row blocks per
unit, over tile counts that span several column chunks (512 tiles; 128 in the
union's last band over at most 2,048 tiles) and ragged tails, and checks that
each tile pair the sweep must evaluate is evaluated exactly once (the union
leaves out the diagonal, which the tile-local union covers) and no other pair
is.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_unit_schedule_covers_every_tile_pair_once(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "sched_check")
    subprocess.run([cxx, "-O2", "-std=c++17", "-o", exe, os.path.join(HERE, "sched_check.cpp")],
                   check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
