"""Writes tests/golden/tiny_f32_samples.txt from the fp64 oracle only.

The fixture is a regression snapshot of the oracle on the seeded 4-prompt fp32 workload
(lengths 17, 64, 100, 255; H_k=2, H_v=4, d=64; checkpoints at multiples of 64): a few
hundred sampled output, checkpoint and final-state entries. It guards the oracle against
accidental edits; its correctness rests on the pin tests, not on this file.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import ref  # noqa: E402
from packed_linear_attention_gb300 import inputs  # noqa: E402


def sample_indices(shape, count, seed):
    rng = np.random.default_rng(seed)
    return [tuple(int(rng.integers(s)) for s in shape) for _ in range(count)]


def main():
    p = inputs.tiny_f32(seed=0)
    o, ck, fin = ref.prefill(p, threads=1)
    lines = ["# oracle snapshot: workload tiny_f32 seed 0 (see make_golden.py)",
             "# kind index... value"]
    for name, arr, seed in (("o", o, 1), ("ckpt", ck, 2), ("final", fin, 3)):
        for idx in sample_indices(arr.shape, 100, seed):
            lines.append(f"{name} {' '.join(map(str, idx))} {float(arr[idx])!r}")
    with open(os.path.join(HERE, "tiny_f32_samples.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
