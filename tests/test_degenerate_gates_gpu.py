"""Degenerate inputs against the oracle, in every kernel. The gates: no decay (a = 0,
g = 1) with full writes (beta = 1); pure decay (beta = 0, the state only shrinks); a
memoryless token (a = -inf, g = 0: the state restarts from that token's write); and decays
strong enough that exp(a) underflows fp32 (a = -120). Gated Delta Networks (Yang, Kautz &
Hatamizadeh, 2024) define the update for every g in [0, 1] and beta in [0, 1]. The keys
and queries: no in-kernel L2 norm (rows normalised upstream), and all-zero rows (norm 0,
the epsilon under the root)."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import compare_units, run

pytestmark = pytest.mark.gpu

KERNELS = [gdn.KERNEL_CHUNKED_PIPELINED, gdn.KERNEL_CHUNKED_THROUGHPUT, gdn.KERNEL_RECURRENT]
CFG = dict(num_k_heads=2, num_v_heads=4, head_dim=128)
LENS = [200, 64, 131, 1, 0, 257]  # chunk edges, a tail, one token, an empty prompt


def _pack(case: str) -> I.Pack:
    p = I.make_pack(LENS, **CFG, io_dtype="bf16", seed=51, init_std=0.02,
                    ckpt_lists=[[64, 192], [64], [128, 131], [1], [], [256, 257]])
    a, beta = p.a.copy(), p.beta.copy()
    rng = np.random.default_rng(7)
    if case == "no_decay_full_write":
        a[:] = 0.0
        beta[:] = 1.0
    elif case == "pure_decay":  # weak decay, so that the states stay inside fp32's range
        a *= 0.01
        beta[:] = 0.0
    elif case == "memoryless_tokens":  # g = 0 at about one token in twenty
        a[rng.random(a.shape) < 0.05] = -np.inf
    elif case == "underflowing_decay":  # exp(a) = 0 in fp32 at about one token in ten
        a[rng.random(a.shape) < 0.1] = -120.0
    else:
        raise ValueError(case)
    return dataclasses.replace(p, a=a.astype(np.float32), beta=beta.astype(np.float32),
                               name=f"{p.name}_{case}")


@pytest.mark.parametrize("case", ["no_decay_full_write", "pure_decay", "memoryless_tokens",
                                  "underflowing_decay"])
@pytest.mark.parametrize("pref", KERNELS)
def test_degenerate_gates(case, pref):
    p = _pack(case)
    got = run(p, pref)
    assert all(np.isfinite(x).all() for x in got), "non-finite output"
    compare_units(p, got, list(range(len(LENS))), list(range(CFG["num_v_heads"])))


def _qk_pack(case: str) -> I.Pack:
    p = I.make_pack(LENS, **CFG, io_dtype="bf16", seed=53, init_std=0.02,
                    ckpt_lists=[[64, 192], [64], [128, 131], [1], [], [256, 257]])
    if case == "no_l2norm":  # q and k normalised upstream (the generator's own rows)
        return dataclasses.replace(p, qk_l2norm=False, name=f"{p.name}_{case}")
    if case == "zero_rows":  # all-zero q and k rows (norm 0: the epsilon under the root)
        q, k = p.q.copy(), p.k.copy()
        rng = np.random.default_rng(9)
        zq = rng.random(q.shape[:2]) < 0.05
        zk = rng.random(k.shape[:2]) < 0.05
        q[zq] = 0
        k[zk] = 0
        return dataclasses.replace(p, q=q, k=k, name=f"{p.name}_{case}")
    raise ValueError(case)


@pytest.mark.parametrize("case", ["no_l2norm", "zero_rows"])
@pytest.mark.parametrize("pref", KERNELS)
def test_qk_without_norm_and_zero_rows(case, pref):
    p = _qk_pack(case)
    got = run(p, pref)
    assert all(np.isfinite(x).all() for x in got), "non-finite output"
    compare_units(p, got, list(range(len(LENS))), list(range(CFG["num_v_heads"])))
