"""Reader for the small text fixtures in this folder (values printed on the pages)."""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def _value(tok: str) -> float:
    if tok.startswith("ln"):
        return math.log(float(Fraction(tok[2:])))
    if tok in ("-inf", "inf"):
        return float(tok)
    return float(Fraction(tok))


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(HERE, name), encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rhs = line.partition("=")
            rows = [[_value(t) for t in r.split()] for r in rhs.split(";")]
            arr = np.array(rows, dtype=np.float64)
            if arr.shape[0] == 1:
                arr = arr[0]
                if arr.size == 1:
                    arr = arr[0]
            out[key.strip()] = arr
    return out
