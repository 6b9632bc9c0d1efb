"""The C ABI used from plain C (`tests/c/abi_smoke.c`): the header compiles as
C99 and the program links against the library with no Python in the way
(here); on a GPU the program runs one decode step and checks it (`-m gpu`)."""
import os
import shutil
import subprocess

import pytest

import paged_kv_cache_156_gb300 as pkv
from paged_kv_cache_156_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_smoke.c")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_program(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = _build.build()
    exe = str(tmp_path / "abi_smoke")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA_HOME, "include"), SRC, "-L", os.path.dirname(lib), "-lpkv",
           "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.dirname(lib), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    exe = build_program(tmp_path)
    assert os.path.exists(exe)


@pytest.mark.gpu
@pytest.mark.parametrize("nvtx", [False, True])
def test_c_program_runs_one_decode_step(tmp_path, nvtx):
    """nvtx: with PKV_NVTX set every launching call opens an NVTX range (a no-op without a tool)."""
    exe = build_program(tmp_path)
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = os.path.dirname(pkv.LIB_PATH) + os.pathsep + env.get("LD_LIBRARY_PATH", "")
    if nvtx:
        env["PKV_NVTX"] = "1"
    else:
        env.pop("PKV_NVTX", None)
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and "abi_smoke ok" in r.stdout, r.stdout + r.stderr
