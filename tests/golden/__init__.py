"""Readers for the hand-worked fixtures in this folder."""
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def mx_blocks():
    """Parse mx_blocks.txt -> list of (name, inputs fp64[32], scale byte, codes uint8[32])."""
    out = []
    cur = None
    with open(os.path.join(HERE, "mx_blocks.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, rest = line.partition(" ")
            if key == "block":
                cur = {"name": rest.strip()}
                out.append(cur)
            elif key == "in":
                v = [float.fromhex(t) for t in rest.split()]
                cur["in"] = np.array(v + [0.0] * (32 - len(v)), dtype=np.float64)
            elif key == "scale":
                cur["scale"] = int(rest, 16)
            elif key == "q":
                q = [int(t, 16) for t in rest.split()]
                cur["q"] = np.array(q + [0] * (32 - len(q)), dtype=np.uint8)
    return [(b["name"], b["in"], b["scale"], b["q"]) for b in out]
