"""Reader for the small text fixtures under tests/golden/."""

import math
import os
from fractions import Fraction

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _value(expr: str) -> float:
    expr = expr.strip()
    if expr == "ln2":
        return math.log(2.0)
    return float(Fraction(expr))


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, expr = line.split("=", 1)
            out[key.strip()] = _value(expr)
    return out
