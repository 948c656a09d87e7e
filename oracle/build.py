"""TEST INFRASTRUCTURE ONLY: compiles the C oracle with gcc (fp64, OpenMP).

Building the checker is not using it: ``__graft_entry__.build()`` calls
``build_oracle()`` so that the GPU machine has the library before the tests run.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "paged_attention_ref.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle_attn.so")


def build_oracle(force: bool = False) -> str:
    """Compile ``paged_attention_ref.c`` into ``_build/liboracle_attn.so``."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
