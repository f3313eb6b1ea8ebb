"""Builds the plain-C oracle into a shared library (test infrastructure only).

The library is written to oracle/_lib/. A build with `mutant=n` plants the known
mistake n (see colimoe_oracle.c); `sanitize=True` adds ASan and UBSan.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "colimoe_oracle.c")
LIB_DIR = os.path.join(HERE, "_lib")


def lib_path(mutant: int = 0, sanitize: bool = False, openmp: bool = True, out_dir: str = LIB_DIR) -> str:
    tag = f"_m{mutant}" if mutant else ""
    tag += "_san" if sanitize else ""
    tag += "" if openmp else "_serial"
    return os.path.join(out_dir, f"libcolimoe_oracle{tag}.so")


def build(mutant: int = 0, sanitize: bool = False, openmp: bool = True, out_dir: str = LIB_DIR,
          force: bool = False) -> str:
    out = lib_path(mutant, sanitize, openmp, out_dir)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(SRC),
                                             os.path.getmtime(os.path.join(HERE, "colimoe_oracle.h")))):
        return out
    os.makedirs(out_dir, exist_ok=True)
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-Wall", "-Wextra", "-Wno-unused-parameter", f"-DCOLI_ORACLE_MUTANT={int(mutant)}"]
    if openmp:
        cmd.append("-fopenmp")
    if sanitize:
        cmd += ["-fsanitize=address,undefined", "-fno-omit-frame-pointer", "-g"]
    tmp = out + f".tmp{os.getpid()}"
    cmd += [SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
