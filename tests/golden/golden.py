"""Reader for the hand-worked text fixtures in this folder."""
from __future__ import annotations

import os
import struct

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def _float(tok: str) -> np.float32:
    if tok.lower().startswith("0x"):
        return np.frombuffer(struct.pack("<I", int(tok, 16)), dtype=np.float32)[0]
    return np.float32(float(tok))


def q8_hand_blocks():
    """Yields dicts: name, K, stride, row_blocks, x (float32 [1, stride]), blocks {b: (d, s, q[32])}."""
    case = None
    with open(os.path.join(HERE, "q8_hand_blocks.txt")) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            head, _, rest = line.partition(" ")
            if head == "case":
                case = {"name": rest.strip(), "xs": {}, "blocks": {}}
            elif head == "K":
                t = rest.split()
                case["K"], case["stride"], case["row_blocks"] = int(t[0]), int(t[2]), int(t[4])
            elif head == "x":
                for tok in rest.split():
                    i, v = tok.split("=")
                    case["xs"][int(i)] = _float(v)
            elif head == "block":
                t = rest.split()
                b = int(t[0])
                d = int(t[1].split("=")[1], 16)
                s = int(t[2].split("=")[1], 16)
                q = np.zeros(32, dtype=np.int8)
                qspec = t[3].split("=", 1)[1] if len(t) > 3 else ""
                for item in filter(None, qspec.split(",")):
                    i, v = item.split(":")
                    q[int(i)] = int(v)
                case["blocks"][b] = (d, s, q)
            elif head == "end":
                x = np.zeros((1, case["stride"]), dtype=np.float32)
                for i, v in case["xs"].items():
                    x[0, i] = v
                case["x"] = x
                yield case
                case = None


def block_bytes(d: int, s: int, q: np.ndarray) -> bytes:
    return struct.pack("<HH", d, s) + q.astype(np.int8).tobytes()
