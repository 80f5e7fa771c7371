"""The oracle reproduces its committed snapshot (tests/golden/make_golden.py)."""
import os

import numpy as np

from oracle import ref
from packed_linear_attention_gb300 import inputs as I

HERE = os.path.dirname(os.path.abspath(__file__))


def load_samples():
    out = []
    with open(os.path.join(HERE, "golden", "tiny_f32_samples.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            out.append((parts[0], tuple(int(x) for x in parts[1:-1]), float(parts[-1])))
    return out


def test_oracle_matches_snapshot():
    o, ck, fin = ref.prefill(I.tiny_f32(seed=0))
    arrays = {"o": o, "ckpt": ck, "final": fin}
    samples = load_samples()
    assert len(samples) == 300
    for name, idx, val in samples:
        np.testing.assert_allclose(arrays[name][idx], val, rtol=1e-12, atol=1e-15)
