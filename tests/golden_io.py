"""Readers for the text fixtures under tests/golden (page-printed values)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def sections(name: str) -> dict:
    """Parse '[section]' blocks of one value per line ('#' lines are citations)."""
    out, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = line[1:-1]
                out[cur] = []
            else:
                out[cur].append(line)
    return out


def records(name: str) -> list:
    """Whitespace-separated records, one per non-comment line."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def f32_bits(values) -> np.ndarray:
    return np.array([np.float32(v) for v in values], dtype=np.float32).view(np.uint32)
