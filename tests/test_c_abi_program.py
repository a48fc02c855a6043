"""The C ABI used from a plain C program (tests/c_abi/route_from_c.c): it compiles and links
against include/moe_route.h and the library on any machine, and on a GB300 it runs route ->
dispatch -> combine and route + dispatch as one call on cudaMalloc'd buffers, checking the
results with no oracle (see the program's header comment)."""
import os
import subprocess

import pytest
import torch

import combine_moe_route_02_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    moe.build()
    libdir = os.path.dirname(moe.lib()._name)
    exe = str(tmp_path / "route_from_c")
    cmd = ["gcc", "-std=c11", "-O1", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c_abi", "route_from_c.c"),
           "-o", exe, "-L", libdir, "-lmoe_route_gb300", "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-3000:]
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_program_runs_the_path(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    exe = _build(tmp_path)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout + out.stderr
    print(out.stdout.strip())
