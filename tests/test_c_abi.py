"""The C ABI from a plain C program (tests/c_abi/host_steps.c): it includes
only include/dms.h and links only libdms.so.  Built here with gcc (no GPU
needed); run on a GPU, where it checks exact first-step outputs and the convex
range of later ones (see the program's header)."""
import os
import shutil
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "learned_kv_cache_eviction_b300")
SRC = os.path.join(ROOT, "tests", "c_abi", "host_steps.c")


def _build(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    lib = os.path.join(LIBDIR, "libdms.so")
    if not os.path.exists(lib):
        pytest.skip("libdms.so not built")
    exe = os.path.join(str(tmp_path), "host_steps")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), SRC, lib,
           f"-Wl,-rpath,{LIBDIR}", "-lm", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_builds_against_the_header_and_library(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_client_runs_host_buffer_steps(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")
