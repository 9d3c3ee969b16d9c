"""Build step of libmxfp4_gb300.so (sm_103a only) and of its bounds-checking
twin libmxfp4_gb300_debug.so (-DMXFP4_DEBUG_BOUNDS).

Compiles every ``csrc/*.cu`` translation unit of both variants in parallel
with nvcc into ``_build/`` and links the shared libraries in-tree, beside this
file.  A variant is rebuilt only when a source or header is newer than it.
No fast-math, no flush-to-zero: the kernels rely on IEEE float32 division
and subnormals.
"""
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(HERE, "libmxfp4_gb300.so")
DEBUG_LIBRARY = os.path.join(HERE, "libmxfp4_gb300_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-Werror", "all-warnings"]
# A register spill in the normal build is an error; the bounds-checking build
# carries extra live ranges and may spill.
VARIANTS = {
    "release": (LIBRARY, BUILD_DIR, ["-Xptxas", "-warn-spills"]),
    "debug": (DEBUG_LIBRARY, os.path.join(BUILD_DIR, "debug"), ["-DMXFP4_DEBUG_BOUNDS"]),
}


def _nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)])


def needs_build(library: str = LIBRARY) -> bool:
    if not os.path.exists(library):
        return True
    built = os.path.getmtime(library)
    return any(os.path.getmtime(p) > built for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link every variant that is missing or stale; returns the
    path of the normal library."""
    todo = [(name, v) for name, v in VARIANTS.items() if force or needs_build(v[0])]
    if not todo:
        return LIBRARY
    nvcc = _nvcc()
    procs, links = [], []
    for name, (library, build_dir, defines) in todo:
        os.makedirs(build_dir, exist_ok=True)
        objs = []
        for src in sources():
            obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defines, *extra_flags, "-c", src, "-o", obj]
            if verbose:
                cmd += ["-Xptxas", "-v"]
            procs.append((f"{name}:{os.path.basename(src)}",
                          subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        links.append((library, objs))
    failed = []
    for tag, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode:
            failed.append(tag)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    for library, objs in links:
        tmp = library + f".tmp{os.getpid()}"
        subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, library)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
