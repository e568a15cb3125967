"""Compile the fp64 C oracle into ``oracle/_build/liboracle.so`` with gcc.

Test infrastructure: building the checker is not using it.  Plain ``-O2``,
no fast-math, so that every floating-point operation is the IEEE binary64
operation written in the source.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off",
                    "-std=c99", "-Wall", "-shared", "-fPIC", SRC, "-o", tmp,
                    "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


def build_variant(src_text: str, name: str) -> str:
    """Compile a modified copy of the oracle source (used by tests that
    plant a mistake in the oracle to check that the pins catch it)."""
    os.makedirs(OUT_DIR, exist_ok=True)
    src = os.path.join(OUT_DIR, f"{name}.c")
    lib = os.path.join(OUT_DIR, f"lib{name}.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off",
                    "-std=c99", "-w", "-shared", "-fPIC", src, "-o", lib,
                    "-lm"], check=True)
    return lib


if __name__ == "__main__":
    print(build(force=True))
