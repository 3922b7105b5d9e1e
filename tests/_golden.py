"""Loading helpers for the hand-worked fixtures in tests/golden/."""
import json
import os

import numpy as np
import torch

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def hexbytes(lst):
    return np.array([int(v, 16) for v in lst], dtype=np.uint8)


def bf16_exact_bits(values):
    """bf16 bits of decimal values that bf16 represents exactly (asserted)."""
    f = [(-0.0 if v == "-0" else float(v)) for v in values]
    t = torch.tensor(f, dtype=torch.float64)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.double(), t), "fixture value not exact in bf16"
    return b.view(torch.int16).numpy().view(np.uint16)
