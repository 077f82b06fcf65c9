"""Compile the oracle (test infrastructure) into oracle/libdlo_oracle.so.

Plain g++, no architecture-specific flags, so the same source builds on the
x86 development host and on the Arm GPU host.  Floating-point contraction is
off so that each multiply and add is rounded separately, as written.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dlo_oracle.cpp")
LIB = os.path.join(HERE, "libdlo_oracle.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.check_call([
        "g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-ffp-contract=off",
        "-pthread", "-o", tmp, SRC])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
