"""Build and run dispatch_cost.c against the in-tree libgranikv.so: the host cost of one
granikv_dispatch call, timed from C on this machine's CPU ("B.5 Per-Step Dispatch Overhead").

  python -m shared_prefix_kv_decode_gb300.dispatch_cost [B ...]     (default: 1 64 1024)
"""

from __future__ import annotations

import os
import platform
import subprocess
import sys

from . import build as _build


def main(argv=None):
    args = list(argv if argv is not None else sys.argv[1:]) or ["1", "64", "1024"]
    lib = _build.build()
    here = os.path.dirname(os.path.abspath(__file__))
    exe = os.path.join(_build.BUILD, "dispatch_cost")
    os.makedirs(_build.BUILD, exist_ok=True)
    subprocess.run(["gcc", "-O2", "-I" + _build.INCLUDE, os.path.join(here, "dispatch_cost.c"), "-o", exe,
                    "-L" + os.path.dirname(lib), "-lgranikv", "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    print(f"# {platform.machine()} host, {os.cpu_count()} cores")
    return subprocess.run([exe] + args).returncode


if __name__ == "__main__":
    sys.exit(main())
