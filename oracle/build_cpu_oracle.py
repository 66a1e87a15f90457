"""Builds the C++ CPU oracle (cpu_oracle.cpp) into liboracle_cpu.so beside it with g++.

TEST INFRASTRUCTURE: building the checker is not using it. Plain C++17 and std::thread,
no architecture flags, so the same source builds on x86-64 and on Arm hosts;
-ffp-contract=off keeps every float32 and double operation rounded on its own.
"""
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cpu_oracle.cpp")
LIB = os.path.join(HERE, "liboracle_cpu.so")


def build(force=False):
    """Compile the oracle if its library is missing or older than its source; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("no C++ compiler found for the CPU oracle")
    tmp = LIB + ".tmp"
    cmd = [cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o", tmp, SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the CPU oracle failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
