"""Build step for the fp64 CPU oracle (test infrastructure only).

Compiles ``attn_oracle.c`` into ``liboracle.so`` next to this file with the
host C compiler.  Only the tests, the smoke check and the CPU-baseline leg
of the benchmark load the result; the CUDA library never does.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build_oracle(force: bool = False) -> str:
    """Compile the oracle if the shared object is missing or stale; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + ".tmp.%d" % os.getpid()
    # -ffp-contract=off keeps every multiply and add separately rounded, so
    # x86 and Arm hosts produce the same fp64 results.
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
