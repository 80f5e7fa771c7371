"""Seeded random packs through every prefill kernel: lengths from 0 to a few hundred tokens
(chunk boundaries, single tokens and empty prompts included), GQA groups of 1, 2 and 4,
zero or nonzero initial states, random checkpoint sets on the chunk grid plus the prompt
end, direct or raw gates, strong or slow decay. On each pack the two chunked schedules must
agree bit for bit, and the throughput schedule and the token-serial kernel must match the
fp64 oracle on every prompt and value head."""
import numpy as np
import pytest

from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import compare_units, run, torch_cuda

pytestmark = pytest.mark.gpu


def _random_pack(seed):
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 7))
    pool = [0, 1, 2, 63, 64, 65, 127, 128, 129, 191, 256]
    lengths = [int(rng.choice(pool)) if rng.random() < 0.4 else int(rng.integers(1, 320))
               for _ in range(n)]
    hk = int(rng.choice([1, 2, 4]))
    group = int(rng.choice([1, 2, 4]))
    hv = min(hk * group, 8)
    if hv % hk:
        hv = hk
    ck = []
    for L in lengths:
        grid = [x for x in range(64, L + 1, 64)]
        pick = sorted(set(int(x) for x in rng.choice(grid, size=min(len(grid), 2), replace=False))) \
            if grid and rng.random() < 0.7 else []
        if L > 0 and (L % 64 or rng.random() < 0.5) and rng.random() < 0.7 and L not in pick:
            pick.append(L)
        ck.append(sorted(pick))
    init_std = float(rng.choice([0.0, 0.02, 0.05]))
    decay = float(rng.choice([1.0, 0.05, 4.0]))
    p = I.make_pack(lengths, num_k_heads=hk, num_v_heads=hv, head_dim=128, io_dtype="bf16",
                    seed=2000 + seed, init_std=init_std if init_std > 0 else None,
                    ckpt_lists=ck, decay_scale=decay)
    if rng.random() < 0.3:
        p = I.with_raw_gates(p, seed=seed)
    return p


@pytest.mark.parametrize("seed", range(40))
def test_random_pack(seed):
    torch_cuda()
    p = _random_pack(seed)
    pipe = run(p, gdn.KERNEL_CHUNKED_PIPELINED)
    thr = run(p, gdn.KERNEL_CHUNKED_THROUGHPUT)
    for x, y, what in zip(pipe, thr, ("o", "ckpt", "final")):
        np.testing.assert_array_equal(x, y, err_msg=what)
    seqs = list(range(p.num_seqs))
    heads = list(range(p.a.shape[1]))
    compare_units(p, thr, seqs, heads, per_item=False)
    compare_units(p, run(p, gdn.KERNEL_RECURRENT), seqs, heads, per_item=False)
