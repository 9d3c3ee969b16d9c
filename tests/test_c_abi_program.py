"""The library called from plain C: programs compiled against
include/mxfp4.h and linked to libmxfp4_gb300.so (the second one also to the
CPU oracle, which only this test program links, to compare every byte).
Compiling and linking run on the CPU (the header's declarations must match
the exported symbols); running them needs the GPU."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT

PROGRAMS = {
    "quantize_worked_block": False,   # expected bytes derived by hand
    "moe_calls_vs_oracle": True,      # expected bytes from the oracle
}


@pytest.fixture(scope="module", params=sorted(PROGRAMS))
def program(request, tmp_path_factory):
    import mxfp4_block_quantization_gb300 as mx
    name = request.param
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    out = str(tmp_path_factory.mktemp("cabi") / name)
    libdir = os.path.dirname(mx.LIB_PATH)
    cmd = [os.environ.get("CC", "gcc"), "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_abi", name + ".c"), "-o", out,
           "-L", libdir, "-lmxfp4_gb300", f"-Wl,-rpath,{libdir}"]
    if PROGRAMS[name]:
        import oracle
        oracle.lib()
        odir = os.path.join(ROOT, "oracle")
        cmd += ["-I", odir, "-L", odir, "-loracle_mxfp4", f"-Wl,-rpath,{odir}"]
    cmd += ["-L", os.path.join(cuda, "lib64"), "-lcudart",
            f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    if shutil.which(cmd[0]) is None:
        pytest.skip("no C compiler")
    if not os.path.exists(os.path.join(libdir, "libmxfp4_gb300.so")):
        pytest.skip("library not built")
    subprocess.run(cmd, check=True)
    return out


def test_c_program_compiles_and_links(program):
    assert os.path.exists(program)


@pytest.mark.gpu
def test_c_program_runs(program):
    r = subprocess.run([program], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "match" in r.stdout
