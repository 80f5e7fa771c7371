"""Degenerate inputs against the oracle, in every kernel. The gates: no decay (a = 0,
g = 1) with full writes (beta = 1); pure decay (beta = 0, the state only shrinks); a
memoryless token (a = -inf, g = 0: the state restarts from that token's write); and decays
strong enough that exp(a) underflows fp32 (a = -120). Gated Delta Networks (Yang, Kautz &
Hatamizadeh, 2024) define the update for every g in [0, 1] and beta in [0, 1]. The keys
and queries: no in-kernel L2 norm (rows normalised upstream), and all-zero rows (norm 0,
the epsilon under the root). Sequence splitting over memoryless tokens, and the decode
step with such inputs."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

from oracle import ref
from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import assert_close, compare_units, handle, run, torch_cuda

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


def test_split_with_memoryless_tokens():
    """Sequence splitting over memoryless tokens: the segment maps (zero and identity
    starts) restart at a = -inf inside a segment, and their composition stays exact."""
    torch = torch_cuda()
    h = handle()
    p = _pack("memoryless_tokens")
    buf = gdn.to_device(p)
    gdn.prefill_split(h, buf, 64)  # the 257-token prompt in five segments
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status(buf.split_workspace) == 0
    got = (buf.o.float().cpu().numpy().astype(np.float64),
           buf.ckpt.cpu().numpy().astype(np.float64),
           buf.final.cpu().numpy().astype(np.float64))
    assert all(np.isfinite(x).all() for x in got), "non-finite output"
    compare_units(p, got, list(range(len(LENS))), list(range(CFG["num_v_heads"])))


def test_decode_step_degenerate_inputs():
    """One decode token with a = -inf (the stored state is dropped), beta = 0 (only the
    decay applies) and all-zero q or k rows, against the oracle."""
    torch = torch_cuda()
    ms = I.mixed_step()
    B = ms.dec_q.shape[0]
    q, k, a, b = ms.dec_q.copy(), ms.dec_k.copy(), ms.dec_a.copy(), ms.dec_beta.copy()
    a[0::4] = -np.inf
    b[1::4] = 0.0
    q[2::4, 0] = 0
    k[3::4, 1] = 0
    cfg = gdn.make_config(16, 32, 128)
    slots = np.arange(B, dtype=np.int32)[::-1].copy()
    pool_np = np.ascontiguousarray(ms.dec_states[::-1])
    pool = torch.from_numpy(pool_np.copy()).cuda()
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    dev = lambda x: torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)  # noqa
    gdn.gdn_decode_step(handle(), cfg, B, dev(q), dev(k), dev(ms.dec_v), torch.from_numpy(a).cuda(),
                        torch.from_numpy(b).cuda(), pool, B, torch.from_numpy(slots).cuda(), o)
    torch.cuda.synchronize()
    f = I.bf16_bits_to_f32
    ro, rpool = ref.decode(f(q), f(k), f(ms.dec_v), a, b, pool_np, slots, scale=128 ** -0.5)
    go = o.float().cpu().numpy().astype(np.float64)
    gp = pool.cpu().numpy().astype(np.float64)
    assert np.isfinite(go).all() and np.isfinite(gp).all()
    assert_close(go, ro, "bf16", "decode o")
    assert_close(gp, rpool, "bf16", "decode states")
