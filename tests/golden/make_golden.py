"""Write tests/golden/oracle_tiny.json: a small oracle result kept as a regression fixture.

The pages print no worked example with values, so this fixture is not a pin against the pages; it
freezes the oracle (already pinned by tests/test_oracle.py) so that later edits to it show up.
It calls only the oracle.  Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import swa_oracle as orc  # noqa: E402


def tiny_inputs():
    """B=1, Hq=2, Hkv=1, N=6, D=4 with entries on a coarse grid (exact in bf16)."""
    rng = np.random.default_rng(2024)
    shape_q, shape_kv = (1, 2, 6, 4), (1, 1, 6, 4)
    q = np.round(rng.standard_normal(shape_q) * 4) / 4
    k = np.round(rng.standard_normal(shape_kv) * 4) / 4
    v = np.round(rng.standard_normal(shape_kv) * 4) / 4
    do = np.round(rng.standard_normal(shape_q) * 4) / 4
    return q, k, v, do


def main():
    q, k, v, do = tiny_inputs()
    W, scale = 3, 0.5
    out = orc.oracle_backward(q, k, v, do, W, scale)
    record = {
        "what": "oracle forward+backward, B=1 Hq=2 Hkv=1 N=6 D=4, window 3, scale 0.5",
        "source": "written by tests/golden/make_golden.py from oracle/ only",
        "window": W,
        "scale": scale,
        "inputs": {"q": q.tolist(), "k": k.tolist(), "v": v.tolist(), "do": do.tolist()},
        "outputs": {key: out[key].tolist() for key in ("o", "lse", "dq", "dk", "dv")},
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json")
    with open(path, "w") as f:
        json.dump(record, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
