"""Parser for tests/golden/worked_examples.txt (hand-worked reads)."""
from __future__ import annotations

import os

import numpy as np

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.txt")


def load_cases(path: str = PATH):
    cases, cur = [], None
    with open(path) as fh:
        for raw in fh:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0], "w": [], "src": [], "expect": [], "w_all": None}
            elif key == "end":
                cur["w"] = np.array(cur["w"], dtype=np.float64)
                cur["src"] = np.array(cur["src"], dtype=np.float64)
                cur["expect"] = np.array(cur["expect"], dtype=np.float64)
                cases.append(cur)
                cur = None
            elif key == "kind":
                cur["kind"] = vals[0]
                if vals[0] == "block":
                    cur["N"], cur["S"] = int(vals[1]), int(vals[2])
            elif key in ("d",):
                cur[key] = int(vals[0])
            elif key in ("eps", "tol"):
                cur[key] = float(vals[0])
            elif key == "w":
                cur["w"].append([float(v) for v in vals])
            elif key == "w*":
                cur["w_all"] = [float(v) for v in vals]
            elif key == "gamma":
                cur["gamma"] = np.array([float(v) for v in vals], dtype=np.float64)
            elif key in ("src", "expect"):
                cur[key].append([float(v) for v in vals])
            else:
                raise ValueError(f"unknown key {key!r} in {path}")
    return cases
