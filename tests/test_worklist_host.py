"""Host check of the expert kernels' work lists: the C++ program worklist_check.cpp expands
random routings through the same header the kernels use (pw_internal.h) and checks that the
lists cover every shared and routed (row tile, token chunk) exactly once, in the order the
kernels rely on, with non-empty K ranges."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_work_lists_cover_every_tile_once(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    exe = tmp_path / "worklist_check"
    subprocess.run([gxx, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "any_precision_bit_gb300", "csrc"),
                    os.path.join(HERE, "worklist_check.cpp"), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip() == "ok"
