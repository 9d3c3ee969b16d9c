"""The library called from plain C: a program compiled against
include/mxfp4.h and linked to libmxfp4_gb300.so.  Compiling and linking run on
the CPU (the header's declarations must match the exported symbols); running
it needs the GPU."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "tests", "c_abi", "quantize_worked_block.c")


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    import mxfp4_block_quantization_gb300 as mx
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    out = str(tmp_path_factory.mktemp("cabi") / "quantize_worked_block")
    libdir = os.path.dirname(mx.LIB_PATH)
    cmd = [os.environ.get("CC", "gcc"), "-std=c11", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"), SRC,
           "-o", out, "-L", libdir, "-lmxfp4_gb300", "-L", os.path.join(cuda, "lib64"),
           "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    if shutil.which(cmd[0]) is None:
        pytest.skip("no C compiler")
    if not os.path.exists(os.path.join(libdir, "libmxfp4_gb300.so")):
        pytest.skip("library not built")
    # the linker wants the conventional file name
    subprocess.run(cmd, check=True)
    return out


def test_c_program_compiles_and_links(program):
    assert os.path.exists(program)


@pytest.mark.gpu
def test_c_program_runs(program):
    r = subprocess.run([program], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "match" in r.stdout
