"""Compile the CPU oracle (plain C++) into oracle/_build/libsmoe_oracle.so.

Test infrastructure: called by ``__graft_entry__.build()`` and on first use of the
``oracle`` package.  No fused multiply-add contraction (-ffp-contract=off), no fast-math,
no architecture-specific flags, so the same sums come out on x86-64 and aarch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "smoe_oracle.cpp")
OUT_DIR = os.path.join(HERE, "_build")
OUT = os.path.join(OUT_DIR, "libsmoe_oracle.so")


def build(force: bool = False, sanitize: bool = False) -> str:
    out = OUT if not sanitize else os.path.join(OUT_DIR, "libsmoe_oracle_san.so")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    os.makedirs(OUT_DIR, exist_ok=True)
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-Wall", "-Wextra", SRC, "-o", out + ".tmp"]
    if sanitize:
        cmd[1:2] = ["-O1", "-g", "-fsanitize=address,undefined", "-fno-omit-frame-pointer"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, sanitize="--sanitize" in sys.argv))
