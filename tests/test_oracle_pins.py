"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test would fail for a plausible slip in the oracle: decay applied after the write,
the output taken from the old state, a sign flip in the delta, a wrong GQA head map, a
checkpoint taken one token early, or the pack offsets mixed up.

The gated delta rule (Gated Delta Networks, Yang, Kautz & Hatamizadeh, 2024):
S_t = g_t S_{t-1} - beta_t (g_t S_{t-1} k_t - v_t) k_t^T, o_t = scale S_t q_t.
Packing, initial states and checkpoints follow sparkinfer v0.6.28's release notes
(packed passes, prefix-cache checkpoints, pack_ckpt_check).
"""
from fractions import Fraction as Fr

import numpy as np
import pytest
import torch

from oracle import ref
from packed_linear_attention_gb300 import inputs as I


def _run(cu, q, k, v, a, beta, init=None, ckpt_cu=None, ckpt_pos=None, scale=1.0, l2norm=False):
    return ref.prefill_arrays(cu, q, k, v, a, beta, init, ckpt_cu, ckpt_pos, scale=scale,
                              l2norm=l2norm, threads=2)


# ---- P1: brute force over exact rationals, product form --------------------------------

def _mat_mul(A, B):
    return [[sum(A[i][t] * B[t][j] for t in range(len(B))) for j in range(len(B[0]))]
            for i in range(len(A))]


def _product_form(S0, ks, vs, gs, bs, T):
    """S_T = S0 A_1...A_T + sum_i beta_i v_i k_i^T A_{i+1}...A_T, A_t = g_t (I - beta_t k_t k_t^T)."""
    dk = len(ks[0])
    I_ = [[Fr(int(i == j)) for j in range(dk)] for i in range(dk)]

    def A(t):
        return [[gs[t] * (I_[i][j] - bs[t] * ks[t][i] * ks[t][j]) for j in range(dk)]
                for i in range(dk)]

    def chain(lo):  # A_lo ... A_{T-1} (0-based)
        M = I_
        for t in range(lo, T):
            M = _mat_mul(M, A(t))
        return M

    S = _mat_mul(S0, chain(0))
    for i in range(T):
        outer = [[bs[i] * vs[i][r] * ks[i][c] for c in range(dk)] for r in range(len(vs[0]))]
        term = _mat_mul(outer, chain(i + 1))
        S = [[S[r][c] + term[r][c] for c in range(dk)] for r in range(len(S))]
    return S


@pytest.mark.parametrize("dk,dv,T", [(2, 2, 5), (3, 2, 6), (2, 3, 4)])
def test_p1_exact_rational_product_form(dk, dv, T):
    rng = np.random.default_rng(10 + dk * 7 + T)
    # rational unit keys: Pythagorean pairs embedded in dk dims
    pairs = [(Fr(3, 5), Fr(4, 5)), (Fr(-4, 5), Fr(3, 5)), (Fr(5, 13), Fr(12, 13)),
             (Fr(8, 17), Fr(-15, 17)), (Fr(1), Fr(0)), (Fr(0), Fr(-1))]
    ks = []
    for t in range(T):
        x, y = pairs[int(rng.integers(len(pairs)))]
        vec = [Fr(0)] * dk
        i0 = int(rng.integers(dk - 1))
        vec[i0], vec[i0 + 1] = x, y
        ks.append(vec)
    qs = [[Fr(int(rng.integers(-4, 5)), 4) for _ in range(dk)] for _ in range(T)]
    vs = [[Fr(int(rng.integers(-8, 9)), 8) for _ in range(dv)] for _ in range(T)]
    gs = [Fr(int(rng.integers(1, 9)), 8) for _ in range(T)]
    bs = [Fr(int(rng.integers(0, 5)), 4) for _ in range(T)]
    S0 = [[Fr(int(rng.integers(-4, 5)), 16) for _ in range(dk)] for _ in range(dv)]
    scale = Fr(1, 2)

    f = lambda M: np.array([[float(x) for x in row] for row in M])
    q = f(qs)[:, None, :]
    k = f(ks)[:, None, :]
    v = f(vs)[:, None, :]
    a = np.log(np.array([float(g) for g in gs]))[:, None]
    beta = np.array([float(b) for b in bs])[:, None]
    init = f(S0)[None, None]
    cu = np.array([0, T], np.int32)
    ckpt_cu = np.array([0, T], np.int32)
    ckpt_pos = np.arange(1, T + 1, dtype=np.int32)
    o, ck, fin = _run(cu, q, k, v, a, beta, init, ckpt_cu, ckpt_pos, scale=0.5)

    for t in range(1, T + 1):
        St = _product_form(S0, ks, vs, gs, bs, t)
        np.testing.assert_allclose(ck[t - 1, 0], f(St), rtol=1e-13, atol=1e-15)
        ot = [scale * sum(St[r][c] * qs[t - 1][c] for c in range(dk)) for r in range(dv)]
        np.testing.assert_allclose(o[t - 1, 0], [float(x) for x in ot], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(fin[0, 0], f(_product_form(S0, ks, vs, gs, bs, T)),
                               rtol=1e-13, atol=1e-15)


def test_p1_python_transcription_matches_c():
    p = I.make_pack([5, 9, 1, 0, 12], num_k_heads=2, num_v_heads=4, head_dim=8, io_dtype="f32",
                    seed=3, init_std=0.3, ckpt_lists=[[2, 5], [9], [1], [], [4, 12]])
    args = (p.cu_seqlens, p.as_f32("q"), p.as_f32("k"), p.as_f32("v"), p.a, p.beta, p.init,
            p.ckpt_cu, p.ckpt_pos)
    o1, c1, f1 = ref.prefill_arrays(*args, scale=p.scale, threads=3)
    o2, c2, f2 = ref.prefill_py(*args, scale=p.scale)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(c1, c2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(f1, f2, rtol=1e-13, atol=1e-15)


# ---- P2: closed form -- the delta rule stores associations -----------------------------

def test_p2_orthonormal_keys_store_values_exactly():
    rng = np.random.default_rng(7)
    d, m = 8, 6
    basis = np.eye(d)[rng.permutation(d)[:m]]            # exactly orthonormal keys
    signs = rng.choice([-1.0, 1.0], size=(m, 1))
    keys = basis * signs
    vals = rng.integers(-16, 17, size=(m, d)) / 16.0
    # query token t with key i(t) <= t
    qidx = [0, 1, 0, 3, 2, 5]
    q = keys[qidx][:, None, :]
    k = keys[:, None, :]
    v = vals[:, None, :]
    a = np.zeros((m, 1))
    beta = np.ones((m, 1))
    o, _, fin = _run(np.array([0, m], np.int32), q, k, v, a, beta, scale=0.25)
    S = fin[0, 0]
    np.testing.assert_array_equal(S, vals.T @ keys)        # S = sum v_i k_i^T
    np.testing.assert_array_equal(S @ keys.T, vals.T)      # S k_i = v_i
    for t, i in enumerate(qidx):
        np.testing.assert_array_equal(o[t, 0], 0.25 * vals[i])


def test_p2_overwrite_replaces_old_value():
    """beta = 1, g = 1, the same key written twice: the second value replaces the first."""
    k = np.array([[[0.6, 0.8]], [[0.6, 0.8]]])
    v = np.array([[[1.0, -2.0]], [[3.0, 0.5]]])
    q = k.copy()
    o, _, fin = _run(np.array([0, 2], np.int32), q, k, v, np.zeros((2, 1)), np.ones((2, 1)))
    np.testing.assert_allclose(fin[0, 0] @ k[1, 0], v[1, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(o[1, 0], v[1, 0], rtol=0, atol=1e-15)


# ---- P3: special cases -------------------------------------------------------------------

def test_p3_zero_beta_is_pure_decay():
    rng = np.random.default_rng(11)
    T, d = 7, 5
    q = rng.standard_normal((T, 1, d))
    k = rng.standard_normal((T, 1, d))
    v = rng.standard_normal((T, 1, d))
    a = -rng.random((T, 1))
    S0 = rng.standard_normal((1, 1, d, d))
    o, _, fin = _run(np.array([0, T], np.int32), q, k, v, a, np.zeros((T, 1)), S0, scale=0.5,
                     l2norm=True)
    cum = np.cumsum(a[:, 0])
    np.testing.assert_allclose(fin[0, 0], np.exp(cum[-1]) * S0[0, 0], rtol=1e-13)
    qn = q[:, 0] / np.sqrt(np.sum(q[:, 0] ** 2, axis=1, keepdims=True) + 1e-6)
    for t in range(T):
        np.testing.assert_allclose(o[t, 0], 0.5 * np.exp(cum[t]) * S0[0, 0] @ qn[t], rtol=1e-12)


def test_p3_zero_decay_is_memoryless():
    rng = np.random.default_rng(12)
    T, d = 6, 4
    q = rng.standard_normal((T, 1, d))
    k = rng.standard_normal((T, 1, d))
    v = rng.standard_normal((T, 1, d))
    beta = rng.random((T, 1))
    a = np.full((T, 1), -np.inf)                           # g = 0
    S0 = rng.standard_normal((1, 1, d, d))
    ckpt_cu = np.array([0, T], np.int32)
    ckpt_pos = np.arange(1, T + 1, dtype=np.int32)
    o, ck, _ = _run(np.array([0, T], np.int32), q, k, v, a, beta, S0, ckpt_cu, ckpt_pos)
    for t in range(T):
        np.testing.assert_allclose(ck[t, 0], beta[t, 0] * np.outer(v[t, 0], k[t, 0]), rtol=1e-14)
        np.testing.assert_allclose(o[t, 0], beta[t, 0] * v[t, 0] * np.dot(k[t, 0], q[t, 0]),
                                   rtol=1e-13)


def test_p3_scalar_state_sum_of_products():
    """d_k = d_v = 1: s_T = s_0 prod_j c_j + sum_i beta_i v_i k_i prod_{j>i} c_j,
    with c_j = g_j (1 - beta_j k_j^2)."""
    rng = np.random.default_rng(13)
    T = 9
    k = rng.uniform(-1, 1, T)
    v = rng.standard_normal(T)
    g = rng.uniform(0.2, 1.0, T)
    b = rng.uniform(0, 1, T)
    s0 = 0.7
    c = g * (1 - b * k * k)
    expect = s0 * np.prod(c) + sum(b[i] * v[i] * k[i] * np.prod(c[i + 1:]) for i in range(T))
    _, _, fin = _run(np.array([0, T], np.int32), np.ones((T, 1, 1)), k[:, None, None],
                     v[:, None, None], np.log(g)[:, None], b[:, None], np.full((1, 1, 1, 1), s0))
    np.testing.assert_allclose(fin[0, 0, 0, 0], expect, rtol=1e-13)


def test_l2norm_matches_prenormalised_keys():
    """With l2norm on, k = c (3, 4) behaves as (3/5, 4/5) up to the 1e-6 under the root."""
    rng = np.random.default_rng(14)
    T = 4
    k_raw = np.array([[3.0, 4.0], [-8.0, 6.0], [5.0, -12.0], [1.0, 0.0]])[:, None, :] * 2.0
    q_raw = np.array([[0.0, 2.0], [3.0, 4.0], [1.0, 1.0], [-6.0, 8.0]])[:, None, :]
    v = rng.standard_normal((T, 1, 2))
    a = -rng.random((T, 1))
    beta = rng.random((T, 1))
    nrm = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    o1, _, f1 = _run(np.array([0, T], np.int32), q_raw, k_raw, v, a, beta, l2norm=True)
    o2, _, f2 = _run(np.array([0, T], np.int32), nrm(q_raw), nrm(k_raw), v, a, beta, l2norm=False)
    np.testing.assert_allclose(o1, o2, rtol=1e-6)
    np.testing.assert_allclose(f1, f2, rtol=1e-6)


# ---- P4: packing -------------------------------------------------------------------------

def test_p4_packed_equals_alone_bitwise():
    p = I.make_pack([17, 64, 100, 1, 0, 33], num_k_heads=2, num_v_heads=4, head_dim=16,
                    io_dtype="bf16", seed=5, init_std=0.02,
                    ckpt_lists=[[17], [64], [64, 100], [1], [], [32]])
    o, ck, fin = ref.prefill(p, threads=4)
    for n in range(p.num_seqs):
        s = I.sub_pack(p, [n])
        o1, ck1, fin1 = ref.prefill(s, threads=1)
        np.testing.assert_array_equal(o[p.cu_seqlens[n]:p.cu_seqlens[n + 1]], o1)
        np.testing.assert_array_equal(ck[p.ckpt_cu[n]:p.ckpt_cu[n + 1]], ck1)
        np.testing.assert_array_equal(fin[n], fin1[0])


# ---- P5: GQA head map ---------------------------------------------------------------------

def test_p5_gqa_equals_duplicated_keys():
    p = I.make_pack([20, 7], num_k_heads=2, num_v_heads=4, head_dim=8, io_dtype="f32", seed=6)
    o, _, fin = ref.prefill(p)
    # same problem with one key head per value head: value head h gets key head h // 2
    q4 = np.repeat(p.as_f32("q"), 2, axis=1)
    k4 = np.repeat(p.as_f32("k"), 2, axis=1)
    o4, _, fin4 = ref.prefill_arrays(p.cu_seqlens, q4, k4, p.as_f32("v"), p.a, p.beta, None,
                                     None, None, scale=p.scale)
    np.testing.assert_array_equal(o, o4)
    np.testing.assert_array_equal(fin, fin4)
    # and a wrong map (h % H_k) would differ
    q_bad = np.stack([p.as_f32("q")[:, h % 2] for h in range(4)], axis=1)
    k_bad = np.stack([p.as_f32("k")[:, h % 2] for h in range(4)], axis=1)
    o_bad, _, _ = ref.prefill_arrays(p.cu_seqlens, q_bad, k_bad, p.as_f32("v"), p.a, p.beta,
                                     None, None, None, scale=p.scale)
    assert not np.array_equal(o, o_bad)


# ---- P6: resume from a checkpoint ----------------------------------------------------------

@pytest.mark.parametrize("cut", [1, 64, 100, 191])
def test_p6_resume_from_checkpoint_bitwise(cut):
    L = 192
    p = I.make_pack([L], num_k_heads=1, num_v_heads=2, head_dim=16, io_dtype="bf16", seed=8,
                    init_std=0.02, ckpt_lists=[[cut]])
    o, ck, fin = ref.prefill(p)
    rest = I.Pack(name="rest", cu_seqlens=np.array([0, L - cut], np.int32),
                  q=p.q[cut:], k=p.k[cut:], v=p.v[cut:], a=p.a[cut:], beta=p.beta[cut:],
                  init=ck.astype(np.float64), ckpt_cu=np.zeros(2, np.int32),
                  ckpt_pos=np.zeros(0, np.int32), num_k_heads=1, num_v_heads=2, head_dim=16,
                  io_dtype="bf16", scale=p.scale)
    o2, _, fin2 = ref.prefill(rest)
    np.testing.assert_array_equal(o[cut:], o2)
    np.testing.assert_array_equal(fin, fin2)


def test_checkpoint_is_state_after_p_tokens():
    """A checkpoint at p equals the final state of the first p tokens run alone."""
    p = I.make_pack([50], num_k_heads=1, num_v_heads=1, head_dim=8, io_dtype="f32", seed=9,
                    ckpt_lists=[[10, 37, 50]])
    _, ck, fin = ref.prefill(p)
    for j, pos in enumerate([10, 37, 50]):
        head = I.make_pack([pos], num_k_heads=1, num_v_heads=1, head_dim=8, io_dtype="f32")
        head.q, head.k, head.v = p.q[:pos], p.k[:pos], p.v[:pos]
        head.a, head.beta = p.a[:pos], p.beta[:pos]
        _, _, f = ref.prefill(head)
        np.testing.assert_array_equal(ck[j], f[0])
    np.testing.assert_array_equal(ck[2], fin[0])


# ---- P8: decode is a one-token prefill ------------------------------------------------------

def test_p8_decode_equals_one_token_prefill():
    rng = np.random.default_rng(15)
    B, Hk, Hv, d = 5, 2, 4, 8
    q = rng.standard_normal((B, Hk, d))
    k = rng.standard_normal((B, Hk, d))
    v = rng.standard_normal((B, Hv, d))
    a = -rng.random((B, Hv))
    beta = rng.random((B, Hv))
    pool = rng.standard_normal((9, Hv, d, d))
    slots = np.array([4, 0, 8, 2, 5], np.int32)
    o, new = ref.decode(q, k, v, a, beta, pool, slots, scale=0.3)
    cu = np.arange(B + 1, dtype=np.int32)
    o2, _, fin = ref.prefill_arrays(cu, q, k, v, a, beta, pool[slots], None, None, scale=0.3)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(new[slots], fin)
    untouched = [s for s in range(9) if s not in set(slots.tolist())]
    np.testing.assert_array_equal(new[untouched], pool[untouched])


# ---- argument checks of the oracle itself ---------------------------------------------------

def test_oracle_rejects_bad_checkpoints():
    p = I.make_pack([10], num_k_heads=1, num_v_heads=1, head_dim=4, io_dtype="f32",
                    ckpt_lists=[[11]])
    with pytest.raises(ValueError):
        ref.prefill(p)


# ---- raw gate inputs: the GDN layer's gating from its projections -------------------------

def test_raw_gates_special_values():
    """a = -exp(A_log) softplus(a_raw + dt_bias), beta = sigmoid(b_raw) at points where the
    functions have exact or limiting values."""
    a_raw = np.array([[0.0, 0.0, 50.0, -50.0]])
    b_raw = np.array([[0.0, 40.0, -40.0, 0.0]])
    a_log = np.array([0.0, np.log(2.0), 0.0, 0.0])
    dt_bias = np.array([0.0, 0.0, 0.0, 0.0])
    a, beta = ref.gates_from_raw(a_raw, b_raw, a_log, dt_bias)
    np.testing.assert_allclose(a[0, 0], -np.log(2.0), rtol=1e-15)        # softplus(0) = ln 2
    np.testing.assert_allclose(a[0, 1], -2.0 * np.log(2.0), rtol=1e-15)  # exp(A_log) = 2
    np.testing.assert_allclose(a[0, 2], -50.0, rtol=1e-15)               # softplus(x) ~ x
    np.testing.assert_allclose(a[0, 3], -np.exp(-50.0), rtol=1e-12)      # ~ exp(x) far left
    np.testing.assert_allclose(beta[0], [0.5, 1.0, np.exp(-40.0), 0.5], rtol=1e-12)
    # dt_bias shifts the softplus argument
    a2, _ = ref.gates_from_raw(np.array([[1.5]]), np.array([[0.0]]), np.array([0.0]),
                               np.array([-1.5]))
    np.testing.assert_allclose(a2[0, 0], -np.log(2.0), rtol=1e-15)


def test_raw_gates_match_library_routines():
    F = torch.nn.functional
    rng = np.random.default_rng(16)
    a_raw = rng.standard_normal((50, 6)) * 4
    b_raw = rng.standard_normal((50, 6)) * 4
    a_log = rng.uniform(-2, 3, 6)
    dt_bias = rng.uniform(-5, 1, 6)
    a, beta = ref.gates_from_raw(a_raw, b_raw, a_log, dt_bias)
    x = torch.from_numpy(a_raw + dt_bias)
    want_a = -torch.exp(torch.from_numpy(a_log)) * F.softplus(x, beta=1.0, threshold=1e9)
    np.testing.assert_allclose(a, want_a.numpy(), rtol=1e-14)
    np.testing.assert_allclose(beta, torch.sigmoid(torch.from_numpy(b_raw)).numpy(), rtol=1e-14)


def test_raw_gate_pack_runs_the_same_recurrence():
    p = I.make_pack([33, 70], num_k_heads=1, num_v_heads=2, head_dim=8, io_dtype="f32", seed=17)
    r = I.with_raw_gates(p, seed=3)
    o, _, f = ref.prefill(r)
    a, beta = ref.gates_from_raw(r.a, r.beta, r.a_log, r.dt_bias)
    o2, _, f2 = ref.prefill_arrays(r.cu_seqlens, r.as_f32("q"), r.as_f32("k"), r.as_f32("v"),
                                   a, beta, None, None, None, scale=r.scale)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(f, f2)
    assert np.all(a < 0) and np.all((beta > 0) & (beta < 1))
