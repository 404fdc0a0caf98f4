"""Build the fp64 CPU oracle (plain C, gcc) into oracle/libmla_oracle.so.

Test infrastructure: compiled by ``__graft_entry__.build()`` and on demand by
``oracle.load()``.  OpenMP is used when the compiler supports it.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mla_oracle.c")
LIB = os.path.join(HERE, "libmla_oracle.so")


def build_oracle(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
