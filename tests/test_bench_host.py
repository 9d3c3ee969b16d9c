"""Host-side checks of bench.py: the algorithmic byte counts its GB/s figures
divide by, and the reference arm (the CPU oracle), which must print the
contract's JSON line without mapping any part of the CUDA library."""
import json
import os
import subprocess
import sys

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_of_the_configurations():
    # BF16 in + codes + tiled scales (pad rows and pad columns counted as written)
    assert bench.quant_bytes(128, 256) == 128 * 256 * 2 + 128 * 128 + 128 * 8
    assert bench.quant_bytes(4096, 7168) == 74_317_824
    assert bench.quant_bytes(1000, 2880) == 7_294_208          # 1024 x 92 scale bytes
    assert bench.quant_bytes(196_608, 2048) == 1_019_215_872   # w13
    assert bench.quant_bytes(262_144, 768) == 509_607_936      # w2
    assert bench.dequant_bytes(4096, 7168) == bench.quant_bytes(4096, 7168)


def test_reference_arm_line_without_the_cuda_library():
    code = (
        "import io, contextlib, json, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import bench\n"
        "buf = io.StringIO()\n"
        "with contextlib.redirect_stdout(buf):\n"
        "    bench.main(['--impl', 'reference', '--steps', '1', '--warmup', '3'])\n"
        "maps = open('/proc/self/maps').read()\n"
        "print(json.dumps({'line': buf.getvalue().strip().splitlines()[-1],\n"
        "                  'product': 'libmxfp4_gb300' in maps,\n"
        "                  'oracle': 'liboracle_mxfp4' in maps}))\n")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    res = json.loads(out.stdout.strip().splitlines()[-1])
    assert res["oracle"] and not res["product"], "the reference arm mapped the CUDA library"
    line = json.loads(res["line"])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["steps"] == 1 and line["warmup"] == 3 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    rows = int(line["config"]["workload"].split("first ")[1].split(" rows")[0])
    assert 1 <= rows <= 4096 and line["config"]["bytes_per_step"] == bench.quant_bytes(rows, 7168)
