"""Host check of how an attention launch cuts its tile list into units of work (each
warp's static share and the pool chunks claimed at run time): compiles
tests/cpp/work_units_check.cpp against the kernel's own header with the host compiler and
runs it. No GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "cpp", "work_units_check.cpp")


def test_work_units_tile_the_list_and_name_each_chunk_once(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "work_units_check")
    subprocess.run([cxx, "-O2", "-std=c++17", "-Wall", "-Werror", SRC, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
