"""GPU parity with raw gate inputs (GDN_GATES_RAW): the kernels turn the raw projections
a_raw, b_raw and the per-head A_log, dt_bias into log-decay and write strength
(a = -exp(A_log) softplus(a_raw + dt_bias), beta = sigmoid(b_raw), the gating of the
Gated DeltaNet layer in the Qwen3.5-style hybrid models) before the recurrence. The
oracle applies the same transform in fp64 and then runs its usual recurrence."""
import numpy as np
import pytest

from oracle import ref
from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import assert_close, compare_units, handle, run, torch_cuda

pytestmark = pytest.mark.gpu

KERNELS = [gdn.KERNEL_AUTO, gdn.KERNEL_RECURRENT]


@pytest.mark.parametrize("pref", KERNELS)
def test_raw_gates_tiny_f32(pref):
    torch_cuda()
    p = I.with_raw_gates(I.tiny_f32(), seed=1)
    o, ck, fin = run(p, pref)
    ro, rck, rfin = ref.prefill(p)
    assert_close(o, ro, "f32", "o")
    assert_close(ck, rck, "f32", "ckpt")
    assert_close(fin, rfin, "f32", "final")


@pytest.mark.parametrize("pref", KERNELS + [gdn.KERNEL_CHUNKED_PIPELINED,
                                            gdn.KERNEL_CHUNKED_THROUGHPUT])
def test_raw_gates_edge_lengths_bf16_d128(pref):
    torch_cuda()
    lengths = [1, 0, 63, 64, 65, 129, 200, 3]
    ck = [[x for x in range(64, n + 1, 64)] + ([n] if n % 64 and n > 0 else []) for n in lengths]
    base = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                       seed=5, init_std=0.02, ckpt_lists=ck)
    p = I.with_raw_gates(base, seed=2)
    got = run(p, pref)
    compare_units(p, got, list(range(len(lengths))), list(range(4)))


def test_raw_gates_equal_precomputed_gates_within_tolerance():
    """The raw-gate call and a direct-gate call fed the oracle's fp64 gates (rounded to
    fp32) agree within the bf16 tolerance: the in-kernel transform is the only difference."""
    torch_cuda()
    lengths = [300, 77, 128]
    base = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                       seed=6, init_std=0.02)
    raw = I.with_raw_gates(base, seed=3)
    a, beta = ref.gates_from_raw(raw.a, raw.beta, raw.a_log, raw.dt_bias)
    direct = I.Pack(**{f: getattr(raw, f) for f in raw.__dataclass_fields__})
    direct.a, direct.beta = a.astype(np.float32), beta.astype(np.float32)
    direct.a_log = direct.dt_bias = None
    g_raw, g_dir = run(raw), run(direct)
    for x, y, what in zip(g_raw, g_dir, ("o", "ckpt", "final")):
        assert_close(x, y, "bf16", what)


def test_raw_gates_decode_step():
    torch = torch_cuda()
    ms = I.mixed_step(seed=4)
    B, Hv = ms.dec_a.shape
    rng = np.random.default_rng(9)
    a_raw = rng.standard_normal((B, Hv)).astype(np.float32)
    b_raw = rng.standard_normal((B, Hv)).astype(np.float32)
    a_log = np.log(rng.uniform(1.0, 16.0, Hv)).astype(np.float32)
    dt_bias = rng.uniform(-7.0, -2.0, Hv).astype(np.float32)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    bf = lambda x: dev(x.view(np.int16)).view(torch.bfloat16)
    a_log_d, dt_bias_d = dev(a_log), dev(dt_bias)
    cfg = gdn.make_config(16, 32, 128, a_log=a_log_d, dt_bias=dt_bias_d)
    pool = dev(ms.dec_states.copy())
    slots = dev(np.arange(B, dtype=np.int32))
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_step(handle(), cfg, B, bf(ms.dec_q), bf(ms.dec_k), bf(ms.dec_v), dev(a_raw),
                        dev(b_raw), pool, B, slots, o)
    torch.cuda.synchronize()
    a, beta = ref.gates_from_raw(a_raw, b_raw, a_log, dt_bias)
    f = I.bf16_bits_to_f32
    ro, rst = ref.decode(f(ms.dec_q), f(ms.dec_k), f(ms.dec_v), a, beta, ms.dec_states,
                         np.arange(B), scale=128 ** -0.5)
    assert_close(o.float().cpu().numpy().astype(np.float64), ro, "bf16", "decode o")
    assert_close(pool.cpu().numpy().astype(np.float64), rst, "bf16", "decode states")
