"""Compile the C oracle (test infrastructure) into oracle/liboracle.so with gcc.

Building the checker is not using it: ``__graft_entry__.build()`` calls this so
that the tests find the library ready on a fresh machine.
"""
from __future__ import annotations

import os
import subprocess
import tempfile

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qwp_oracle.c")


def library_path() -> str:
    return os.path.join(_HERE, "liboracle.so")


def is_stale() -> bool:
    lib = library_path()
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(_SRC)


def build(verbose: bool = False) -> str:
    out = library_path()
    tmp = tempfile.NamedTemporaryFile(suffix=".so", dir=_HERE, delete=False).name
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    # OpenMP over output rows when the compiler supports it; plain serial C otherwise.
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            break
        if verbose:
            print(r.stderr)
    else:
        os.unlink(tmp)
        raise RuntimeError("failed to compile the oracle: " + r.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True))
