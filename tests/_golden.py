"""Loading of the hand-derived fixtures under tests/golden/."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f32(rows):
    conv = {"nan": np.nan, "-0": -0.0}
    return np.array([[conv.get(v, v) if isinstance(v, str) else v for v in r] for r in rows],
                    np.float32)


def bf16_bits(a):
    """Exact bf16 values -> bit patterns (fixture values are exact in bf16)."""
    f = np.asarray(a, np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "fixture value not exact in bf16"
    return (u >> 16).astype(np.uint16)
