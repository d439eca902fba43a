"""The workspace layout and the row-statistics chunk plan, checked on the host (no GPU).

Compiles tests/native/chunk_plan_check.cu (which includes the statistics
translation unit) against the library's other objects with nvcc and runs it:
the workspace regions must be aligned, ordered and large enough for every
shape tried; every row's chunks, found as the merge kernel finds them, must
cover the row's stages once and in order, and the plan must fit the
workspace's partial area.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_chunk_plan_covers_every_row_once(tmp_path):
    from reject_row_vocab_gb300 import _build
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    _build.build()
    objs = [os.path.join(_build.BUILD, s.replace(".cu", ".o")) for s in _build.SOURCES if s != "sv_stats.cu"]
    exe = str(tmp_path / "chunk_plan_check")
    cmd = [_build.nvcc()] + _build.ARCH + ["-O1", "-std=c++17", "-I", _build.INCLUDE, "-I", _build.CSRC,
                                          os.path.join(ROOT, "tests", "native", "chunk_plan_check.cu")] + objs + \
        ["-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-3000:]
    assert "layout: " in r.stdout and r.stdout.count(" 0 failures") == 2, r.stdout
