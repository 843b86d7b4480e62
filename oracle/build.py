"""Builds the fp64 CPU oracles with gcc: ``libgn_oracle.so`` (GroupNorm,
``gn_oracle.c``) and ``librow_oracle.so`` (LayerNorm / RMSNorm over rows,
``row_oracle.c``).

Test infrastructure only.  ``build(mutant=k)`` compiles a copy with one planted
mistake (see the C sources) into a separate file; only the mutation tests ask
for that.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = {"gn": ("gn_oracle.c", "GNO_MUTANT"), "row": ("row_oracle.c", "RNO_MUTANT")}


def lib_path(mutant: int = 0, outdir: str | None = None, which: str = "gn") -> str:
    stem = {"gn": "libgn_oracle", "row": "librow_oracle"}[which]
    name = f"{stem}.so" if mutant == 0 else f"{stem}_m{mutant}.so"
    return os.path.join(outdir or HERE, name)


def build(mutant: int = 0, outdir: str | None = None, force: bool = False,
          which: str = "gn") -> str:
    src, macro = SOURCES[which]
    src = os.path.join(HERE, src)
    out = lib_path(mutant, outdir, which)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
           f"-D{macro}={int(mutant)}", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build_all(force: bool = False) -> list:
    return [build(0, force=force, which=w) for w in SOURCES]


if __name__ == "__main__":
    print(build_all(force=True))
