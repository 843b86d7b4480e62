"""Builds the fp64 CPU oracle (``libgn_oracle.so``) with gcc.

Test infrastructure only.  ``build(mutant=k)`` compiles a copy with one planted
mistake (see ``gn_oracle.c``) into a separate file; only the mutation test asks
for that.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gn_oracle.c")


def lib_path(mutant: int = 0, outdir: str | None = None) -> str:
    name = "libgn_oracle.so" if mutant == 0 else f"libgn_oracle_m{mutant}.so"
    return os.path.join(outdir or HERE, name)


def build(mutant: int = 0, outdir: str | None = None, force: bool = False) -> str:
    out = lib_path(mutant, outdir)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SRC)):
        return out
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
           f"-DGNO_MUTANT={int(mutant)}", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(int(sys.argv[1]) if len(sys.argv) > 1 else 0, force=True))
