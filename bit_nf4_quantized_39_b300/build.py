"""Build step of libqlora_nf4.so: one nvcc invocation for sm_103a, in-tree.

Usage: ``python -m bit_nf4_quantized_39_b300.build`` (or ``__graft_entry__.build()``).
The library is written next to this file so that it travels with the source
tree; nothing is installed into site-packages.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "api.cu")
OUT = os.path.join(HERE, "libqlora_nf4.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def command(out: str = OUT, extra=()) -> list:
    return [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
            "-I", os.path.join(ROOT, "include"), "-Xptxas", "-v", *extra, "-o", out, SRC]


def sources():
    d = os.path.join(HERE, "csrc")
    return [os.path.join(d, f) for f in sorted(os.listdir(d))] + [os.path.join(ROOT, "include", "qlora_nf4.h")]


def up_to_date(out: str = OUT) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(s) <= t for s in sources())


def build(force: bool = False, verbose: bool = False, log: str | None = None) -> str:
    if not force and up_to_date():
        return OUT
    cmd = command()
    res = subprocess.run(cmd, capture_output=True, text=True)
    text = res.stdout + res.stderr
    if log:
        with open(log, "w") as f:
            f.write(" ".join(cmd) + "\n" + text)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + "\n".join(l for l in text.splitlines() if "error" in l)[:4000])
    if verbose:
        print(text)
    return OUT


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(OUT)
