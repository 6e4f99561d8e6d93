"""Host check (no GPU): the dense tensor-core kernel walks only the live tiles
of a mask through closed-form ranges (live_query_tiles / live_key_tiles in
csrc/mask.h); they must name exactly the tiles tile_any classifies as live.
The check is a small C++ program compiled here with the host compiler."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_live_tile_ranges_match_tile_classes(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "tile_ranges_check"
    src = os.path.join(ROOT, "tests", "native", "tile_ranges_check.cpp")
    inc = os.path.join(ROOT, "attention_backward_attn_gb300", "csrc")
    subprocess.run([cxx, "-O1", "-std=c++17", "-I", inc, src, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout
    assert out.stdout.startswith("ok ")
