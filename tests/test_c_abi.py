"""The boundary from plain C: every public header is valid C99, and small C
programs linked against libhoc.so use it without Python (host-only entry
points on any machine; an allreduce and an all-gather on the GPU)."""
import glob
import os
import shutil
import subprocess

import pytest

from collective_communication_schedules_gb300 import hoc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.dirname(hoc.LIB_PATH)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

needs_gcc = pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")


@needs_gcc
@pytest.mark.parametrize("header", sorted(glob.glob(os.path.join(INCLUDE, "*.h"))), ids=os.path.basename)
def test_header_is_c99(header):
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", INCLUDE, "-x", "c", header], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _build_and_run(src, out, extra):
    if not os.path.exists(hoc.LIB_PATH):
        pytest.skip("libhoc.so is not built")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, src, "-L", LIBDIR, "-lhoc",
           f"-Wl,-rpath,{LIBDIR}", "-o", out] + extra
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return subprocess.run([out], capture_output=True, text=True, timeout=120)


@needs_gcc
def test_host_entry_points_from_c(tmp_path):
    r = _build_and_run(os.path.join(ROOT, "tests", "c", "abi_host.c"), str(tmp_path / "abi_host"), [])
    assert r.returncode == 0 and "ABI OK" in r.stdout, r.stdout + r.stderr


@pytest.mark.gpu
@needs_gcc
def test_collectives_from_c(tmp_path):
    extra = ["-I", os.path.join(CUDA, "include"), "-L", os.path.join(CUDA, "lib64"), "-lcudart",
             f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = _build_and_run(os.path.join(ROOT, "tests", "c", "abi_gpu.c"), str(tmp_path / "abi_gpu"), extra)
    assert r.returncode == 0 and "ABI GPU OK" in r.stdout, r.stdout + r.stderr
