"""Reader for the hand-derived block probes under tests/golden/."""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
QK = {"q8_0": 32, "q4_k": 256, "q6_k": 256}
BB = {"q8_0": 34, "q4_k": 144, "q6_k": 210}


def load(fmt: str):
    """Yield (name, K, raw_bytes_of_one_row, expected_weights[K])."""
    path = os.path.join(GOLDEN, f"{fmt}_probes.txt")
    probes = []
    cur = None
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "probe":
                K = int(tok[2].split("=")[1])
                nb = (K + QK[fmt] - 1) // QK[fmt]
                cur = {"name": tok[1], "K": K, "raw": np.zeros(nb * BB[fmt], np.uint8),
                       "exp": np.zeros(K, np.float64)}
            elif tok[0] == "set":
                cur["raw"][int(tok[1])] = int(tok[2], 16)
            elif tok[0] == "fill":
                cur["raw"][int(tok[1]):int(tok[2]) + 1] = int(tok[3], 16)
            elif tok[0] == "expect":
                cur["exp"][int(tok[1])] = _val(tok[2])
            elif tok[0] == "expect_range":
                cur["exp"][int(tok[1]):int(tok[2]) + 1] = _val(tok[3])
            elif tok[0] == "end":
                probes.append((cur["name"], cur["K"], cur["raw"], cur["exp"]))
                cur = None
            else:
                raise ValueError(f"bad fixture line: {line}")
    return probes


def _val(s: str) -> float:
    if "0x" in s.lower():
        return float.fromhex(s)
    return float(s)
