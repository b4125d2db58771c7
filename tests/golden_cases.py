"""Parser for tests/golden/hand_worked_cases.txt (hand-derived closed forms)."""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_worked_cases.txt")
POISON = 1.0e30


def load_cases(path: str = GOLDEN) -> dict[str, dict]:
    cases: dict[str, dict] = {}
    cur = None
    with open(path) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("case "):
                cur = cases.setdefault(line[5:].strip(), {})
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            cur[key] = json.loads(val)
    return cases


def _expand(x, D):
    """Nested lists with "P" (a whole row of poison) -> float list."""
    if x == "P":
        return [POISON] * D
    if isinstance(x, list):
        return [_expand(e, D) for e in x]
    return float(x)


def pool_tensor(case: dict, key: str) -> torch.Tensor:
    return torch.tensor(_expand(case[key], case["D"]), dtype=torch.float32)


def scale_of(case: dict) -> float:
    s = case["scale"]
    return math.log(3.0) if s == "ln3" else float(s)


def expected_of(case: dict) -> torch.Tensor:
    def conv(x):
        if isinstance(x, list):
            return [conv(e) for e in x]
        return float(Fraction(x))
    return torch.tensor(conv(case["expected"]), dtype=torch.float64)
