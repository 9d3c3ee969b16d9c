"""Build step of the CPU oracle (test infrastructure only).

Compiles ``mxfp4_oracle.c`` into ``liboracle_mxfp4.so`` beside it with the
host C compiler.  Strict IEEE arithmetic: no fast-math, no FP contraction.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "mxfp4_oracle.c")
HEADER = os.path.join(HERE, "mxfp4_oracle.h")
LIBRARY = os.path.join(HERE, "liboracle_mxfp4.so")


def needs_build() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    built = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(p) > built for p in (SOURCE, HEADER))


def build(force: bool = False) -> str:
    """Compile the oracle if it is missing or older than its sources."""
    if force or needs_build():
        tmp = LIBRARY + f".tmp{os.getpid()}"
        cmd = [
            os.environ.get("CC", "gcc"), "-std=c11", "-O2", "-Wall", "-Wextra",
            "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
            SOURCE, "-o", tmp, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True))
