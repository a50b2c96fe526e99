"""Build and run stream_floor.cu: the read-bandwidth floor of a kernel that only stages bytes
through shared memory the way the decode kernels do (one CTA per SM, a ring of bulk-copied
stages), for one layer's 16K-token prefix (67 MB) as a cold single launch and as a chain of
back-to-back launches, and for 1 GB.  It bounds what a decode-attention launch of that size can
reach on this GPU.

  python -m shared_prefix_kv_decode_gb300.stream_floor
"""

from __future__ import annotations

import json
import os
import subprocess
import sys

from . import build as _build


def main(argv=None):
    here = os.path.dirname(os.path.abspath(__file__))
    exe = os.path.join(_build.BUILD, "stream_floor")
    os.makedirs(_build.BUILD, exist_ok=True)
    subprocess.run([_build._nvcc(), *_build.ARCH, "-O3", "-std=c++17", "-o", exe,
                    os.path.join(here, "stream_floor.cu")], check=True)
    peak = 0.0
    path = os.path.join(os.path.dirname(here), "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            peak = float(json.load(f).get("hbm_gbs", 0.0))
    return subprocess.run([exe, str(peak)]).returncode


if __name__ == "__main__":
    sys.exit(main())
