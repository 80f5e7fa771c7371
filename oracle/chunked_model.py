"""NumPy model of the chunked (UT / WY) form of the gated delta rule (TEST INFRASTRUCTURE).

This is not the oracle: it is the algebra that the GPU kernel evaluates, written in fp64
with plain matrix products so that a test can check the decomposition against the
token-by-token oracle (they agree to ~1e-12), and so that the effect of rounding each
tensor-core operand to bf16 can be measured on the CPU before any kernel is written.
It shares no code with the CUDA library.

Per prompt and value head, for a chunk of L <= C tokens starting from state S0
(d_v x d_k), with G_i = a_1 + ... + a_i (chunk-local inclusive cumulative log-decay) and
k_i, q_i L2-normalised:

  A_ij   = beta_i exp(G_i - G_j) (k_i . k_j)      for j < i, else 0
  T      = (I + A)^{-1}                           unit lower triangular
  U      = T diag(beta) V
  W      = T diag(beta exp(G)) K
  Delta  = U - W S0^T                             row i is the delta written at token i
  O      = scale [diag(exp(G)) Q S0^T + (exp(G_i - G_j) (q_i . k_j))_{j <= i} Delta]
  S_L    = exp(G_L) S0 + Delta^T diag(exp(G_L - G)) K

Derivation: unrolling S_t = g_t S_{t-1} + delta_t k_t^T inside the chunk gives
S_t = exp(G_t) S0 + sum_{j<=t} exp(G_t - G_j) delta_j k_j^T; substituting into
delta_t = beta_t (v_t - g_t S_{t-1} k_t) gives (I + A) Delta = diag(beta)(V - diag(exp G) K S0^T).
All exponents are <= 0, so no term can overflow.

The L2 norms are folded into diagonal factors, so the raw input rows of K and Q are the
only operands that meet the norms (as the kernel does, keeping those operands exact).
"""
from __future__ import annotations

import numpy as np

L2NORM_EPS = 1e-6


# ---- operand rounding models (for precision studies) -------------------------------------

def _bf16(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + (((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF))) & np.uint32(0xFFFF0000)
    return r.view(np.float32).astype(np.float64)


def _tf32(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + (((u >> 13) & np.uint32(1)) + np.uint32(0xFFF))) & np.uint32(0xFFFFE000)
    return r.view(np.float32).astype(np.float64)


def operand(x: np.ndarray, mode: str) -> list[np.ndarray]:
    """Split an operand the way a tensor-core product would consume it: a list of parts
    whose products are summed. 'f64': exact; 'f32': fp32; 'bf16': one rounding;
    'bf16x2': hi + lo bf16 pair; 'tf32': one tf32 rounding; 'f16': one
    IEEE half rounding."""
    if mode == "f64":
        return [np.asarray(x, dtype=np.float64)]
    if mode == "f32":
        return [np.asarray(x, dtype=np.float32).astype(np.float64)]
    if mode == "bf16":
        return [_bf16(x)]
    if mode == "bf16x2":
        hi = _bf16(x)
        return [hi, _bf16(np.asarray(x, np.float64) - hi)]
    if mode == "tf32":
        return [_tf32(x)]
    if mode == "f16":
        return [np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)]
    raise ValueError(mode)


def mm(a: np.ndarray, b: np.ndarray, ma: str = "f64", mb: str = "f64",
       drop_lo_lo: bool = True) -> np.ndarray:
    """a @ b with each operand split per its mode (lo*lo terms dropped, as a kernel would)."""
    pa, pb = operand(a, ma), operand(b, mb)
    out = np.zeros((a.shape[0], b.shape[1]))
    for i, x in enumerate(pa):
        for j, y in enumerate(pb):
            if drop_lo_lo and i > 0 and j > 0:
                continue
            out += x @ y
    return out


# Default: everything exact (the P7 check). A precision study passes a dict overriding
# some of these keys with 'bf16', 'bf16x2', 'tf32' or 'f32'.
EXACT = dict(T=("f64", "f64"), WK=("f64", "f64"), US=("f64", "f64"), QS=("f64", "f64"),
             PD=("f64", "f64"), DK=("f64", "f64"), inv="f64")


def _chunk(S0, Kr, Qr, V, a, beta, scale, l2norm, prec):
    """One chunk; returns (O, S_end). Kr, Qr are the raw (un-normalised) rows."""
    L = Kr.shape[0]
    if l2norm:
        rk = 1.0 / np.sqrt(np.sum(Kr * Kr, axis=1) + L2NORM_EPS)
        rq = 1.0 / np.sqrt(np.sum(Qr * Qr, axis=1) + L2NORM_EPS)
    else:
        rk = np.ones(L)
        rq = np.ones(L)
    G = np.cumsum(a)
    gam = np.exp(G)
    diff = G[:, None] - G[None, :]
    lower = np.tril(np.ones((L, L), dtype=bool), -1)
    incl = np.tril(np.ones((L, L), dtype=bool), 0)
    Gam_strict = np.where(lower, np.exp(np.where(lower, diff, 0.0)), 0.0)
    Gam_incl = np.where(incl, np.exp(np.where(incl, diff, 0.0)), 0.0)

    KK = mm(Kr, Kr.T)                        # raw K K^T (exact operands: bf16 inputs)
    QK = mm(Qr, Kr.T)
    A = (beta * rk)[:, None] * Gam_strict * KK * rk[None, :]
    P = rq[:, None] * Gam_incl * QK * rk[None, :]
    I = np.eye(L)
    if prec["inv"] == "f32":
        T = np.linalg.inv((I + A).astype(np.float32)).astype(np.float64)
    else:
        T = np.linalg.inv(I + A)
    T = np.tril(T)
    # W = T diag(beta gamma / |k|) K_raw ; U = T diag(beta) V
    W = mm(T * (beta * gam * rk)[None, :], Kr, *prec["WK"])
    U = mm(T * beta[None, :], V, *prec["T"])
    # Delta = U - W S0^T
    Delta = U - mm(W, S0.T, *prec["US"])
    # O = scale [diag(gamma / |q|) Q_raw S0^T + P Delta]
    O = scale * ((gam * rq)[:, None] * mm(Qr, S0.T, "f64", prec["QS"][1]) +
                 mm(P, Delta, *prec["PD"]))
    # S_L = gamma_L S0 + Delta^T diag(exp(G_L - G) / |k|) K_raw
    decay_to_end = np.exp(G[-1] - G) * rk
    S_end = gam[-1] * S0 + mm(Delta.T * decay_to_end[None, :], Kr, *prec["DK"])
    return O, S_end


def prefill(cu_seqlens, q, k, v, a, beta, init, ckpt_cu, ckpt_pos, *, scale, chunk=64,
            l2norm=True, prec=None, heads=None):
    """Chunked evaluation over a pack. Shapes as the oracle's. Checkpoint positions must
    be multiples of `chunk` or equal to the prompt length. Returns (o, ckpt, final)."""
    p = dict(EXACT)
    if prec:
        p.update(prec)
    cu = [int(x) for x in cu_seqlens]
    q, k, v, a, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, a, beta))
    N = len(cu) - 1
    T_, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    G = Hv // Hk
    o = np.zeros((T_, Hv, dv))
    C = 0 if ckpt_cu is None else int(ckpt_cu[-1])
    ck = np.zeros((C, Hv, dv, dk))
    fin = np.zeros((N, Hv, dv, dk))
    for n in range(N):
        s, e = cu[n], cu[n + 1]
        want = {} if ckpt_cu is None else {
            int(ckpt_pos[j]): j for j in range(int(ckpt_cu[n]), int(ckpt_cu[n + 1]))}
        for pos in want:
            if pos % chunk and pos != e - s:
                raise ValueError("checkpoint off the chunk grid")
        for h in (range(Hv) if heads is None else heads):
            S = np.zeros((dv, dk)) if init is None else np.array(init[n, h], dtype=np.float64)
            for c0 in range(s, e, chunk):
                c1 = min(c0 + chunk, e)
                O, S = _chunk(S, k[c0:c1, h // G], q[c0:c1, h // G], v[c0:c1, h],
                              a[c0:c1, h], beta[c0:c1, h], scale, l2norm, p)
                o[c0:c1, h] = O
                if (c1 - s) in want:
                    ck[want[c1 - s], h] = S
            fin[n, h] = S
    return o, ck, fin
