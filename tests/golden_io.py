"""Readers for the hand-written fixtures under tests/golden/."""
import os

import numpy as np

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(HERE, name), encoding="utf-8") as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                yield line


def layout():
    out = {}
    for line in _lines("layout.txt"):
        k, v = [s.strip() for s in line.split("=", 1)]
        vals = [float(x) for x in v.split()]
        out[k] = vals if len(vals) > 1 else vals[0]
    return out


def hand_row():
    """-> dict(latent float64 [512], rope float64 [64], row uint8 [352],
    codes {g: [16]}, groups [g...])."""
    latent = np.zeros(512)
    rope = np.zeros(64)
    row = np.zeros(352, dtype=np.uint8)
    codes = {}
    groups = []
    rope_vals = rope_bytes = None
    for line in _lines("hand_row.txt"):
        head, body = [s.strip() for s in line.split(":", 1)]
        parts = head.split()
        if parts[0] == "group":
            g, what = int(parts[1]), parts[2]
            if what == "values":
                latent[16 * g:16 * g + 16] = [float(x) for x in body.split()]
                groups.append(g)
            elif what == "scale":
                row[256 + g] = int(body, 16)
            elif what == "codes":
                codes[g] = [int(x) for x in body.split()]
            elif what == "bytes":
                row[8 * g:8 * g + 8] = [int(x, 16) for x in body.split()]
        elif parts[0] == "rope" and parts[1] == "values":
            rope_vals = [float(x) for x in body.split()]
        elif parts[0] == "rope" and parts[1] == "bytes":
            rope_bytes = [int(x, 16) for x in body.split()]
    rope[:len(rope_vals)] = rope_vals
    row[288:288 + len(rope_bytes)] = rope_bytes
    return {"latent": latent, "rope": rope, "row": row, "codes": codes, "groups": groups}
