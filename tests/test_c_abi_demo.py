"""A plain C program against include/mp.h and libmp.so (tests/c/mp_abi_demo.c):
it compiles as C11 here, and on a GPU it runs the pages' worked example, a
permute/unpermute roundtrip and an error path through the C ABI alone."""
from __future__ import annotations

import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "mp_abi_demo.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _flags():
    return ["-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
            "-I", os.path.join(CUDA, "include")]


def test_demo_compiles_as_c(tmp_path):
    if not os.path.isdir(os.path.join(CUDA, "include")):
        pytest.skip("no CUDA headers")
    subprocess.run(["gcc", *_flags(), "-c", SRC, "-o", str(tmp_path / "demo.o")], check=True)


@pytest.mark.gpu
def test_demo_runs_through_the_c_abi(tmp_path):
    from unpermute_routing_indices_gb300 import library_path
    lib = library_path()
    exe = tmp_path / "demo"
    subprocess.run(["gcc", *_flags(), SRC, "-o", str(exe), lib,
                    "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                    "-Wl,-rpath," + os.path.dirname(lib),
                    "-Wl,-rpath," + os.path.join(CUDA, "lib64")], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
