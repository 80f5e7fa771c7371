"""Python entry to the fp64 CPU oracle (TEST INFRASTRUCTURE ONLY).

Only tests, the smoke check and the benchmark's CPU-baseline leg may import this module.
It builds and loads ``oracle/gdn_ref.c`` (plain C, gcc) and feeds it the exact fp64
widening of the values the library reads (bf16 or fp32). It shares no code with the CUDA
library and never imports it.

Functions:
  * ``prefill(pack)`` -- the token-by-token gated delta rule over a packed batch
    (Gated Delta Networks' recurrence; packed prompts, initial states and prefix-cache
    checkpoints as in sparkinfer v0.6.28's release notes).
  * ``decode(...)`` -- one token per sequence, the same recurrence applied once.
  * ``prefill_py(...)`` -- the same definition in pure Python/NumPy loops, for tiny cases.

Every function here is pinned by tests that do not reuse its formula (brute force over
exact rationals, closed forms, special cases, packing/resume identities).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdn_ref.c")
LIB = os.path.join(HERE, "libgdn_ref.so")
L2NORM_EPS = 1e-6

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_ref.c into libgdn_ref.so next to it (gcc -O2, no target-specific flags)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, SRC, "-lm", "-lpthread"])
        os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIB)
            P = ctypes.c_void_p
            i32, f64 = ctypes.c_int32, ctypes.c_double
            lib.gdn_ref_prefill.restype = ctypes.c_int
            lib.gdn_ref_prefill.argtypes = [i32, P, i32, i32, i32, i32, f64, i32, f64,
                                            P, P, P, P, P, P, P, P, P, P, P, i32]
            lib.gdn_ref_decode.restype = ctypes.c_int
            lib.gdn_ref_decode.argtypes = [i32, i32, i32, i32, i32, f64, i32, f64,
                                           P, P, P, P, P, P, P, P]
            _lib = lib
    return _lib


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def _f64(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float64)


def gates_from_raw(a_raw, b_raw, a_log, dt_bias):
    """Gates of the Qwen3.5/3.6-style GDN layer from its raw projections, in fp64: per value
    head h, log-decay a = -exp(A_log[h]) * softplus(a_raw + dt_bias[h]) (so g = exp(a))
    and write strength beta = sigmoid(b_raw). a_raw, b_raw: [T, H_v]; a_log, dt_bias: [H_v]."""
    a_raw = np.asarray(a_raw, dtype=np.float64)
    b_raw = np.asarray(b_raw, dtype=np.float64)
    x = a_raw + np.asarray(dt_bias, dtype=np.float64)[None, :]
    softplus = np.logaddexp(0.0, x)
    a = -np.exp(np.asarray(a_log, dtype=np.float64))[None, :] * softplus
    beta = 1.0 / (1.0 + np.exp(-b_raw))
    return a, beta


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def prefill_arrays(cu_seqlens, q, k, v, a, beta, init, ckpt_cu, ckpt_pos, *, scale,
                   l2norm=True, eps=L2NORM_EPS, threads=None):
    """Run the oracle on fp64-convertible arrays. Shapes: q, k [T, H_k, d_k];
    v [T, H_v, d_v]; a, beta [T, H_v]; init [N, H_v, d_v, d_k] or None.
    Returns (o [T, H_v, d_v], ckpt [C, H_v, d_v, d_k], final [N, H_v, d_v, d_k]) in fp64."""
    lib = _load()
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    N = cu.shape[0] - 1
    q, k, v, a, beta, init = map(_f64, (q, k, v, a, beta, init))
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    assert k.shape == q.shape and v.shape[0] == T and a.shape == (T, Hv) == beta.shape
    if ckpt_cu is None:
        ckpt_cu = np.zeros(N + 1, dtype=np.int32)
        ckpt_pos = np.zeros(0, dtype=np.int32)
    ckpt_cu = np.ascontiguousarray(ckpt_cu, dtype=np.int32)
    ckpt_pos = np.ascontiguousarray(ckpt_pos, dtype=np.int32)
    C = int(ckpt_cu[-1])
    o = np.zeros((T, Hv, dv), dtype=np.float64)
    ck = np.zeros((C, Hv, dv, dk), dtype=np.float64)
    fin = np.zeros((N, Hv, dv, dk), dtype=np.float64)
    if init is not None:
        assert init.shape == (N, Hv, dv, dk)
    rc = lib.gdn_ref_prefill(N, _ptr(cu), Hk, Hv, dk, dv, float(scale), int(bool(l2norm)),
                             float(eps), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta),
                             _ptr(init), _ptr(ckpt_cu), _ptr(ckpt_pos) if C else None,
                             _ptr(o), _ptr(ck) if C else None, _ptr(fin),
                             int(threads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")
    return o, ck, fin


def prefill(pack, threads=None):
    """Oracle over a ``Pack`` from ``packed_linear_attention_gb300.inputs`` (raw gate
    inputs, when the pack has them, are turned into gates by gates_from_raw first)."""
    a, beta = pack.a, pack.beta
    if getattr(pack, "a_log", None) is not None:
        a, beta = gates_from_raw(pack.a, pack.beta, pack.a_log, pack.dt_bias)
    return prefill_arrays(pack.cu_seqlens, pack.as_f32("q"), pack.as_f32("k"),
                          pack.as_f32("v"), a, beta, pack.init, pack.ckpt_cu,
                          pack.ckpt_pos, scale=pack.scale, l2norm=pack.qk_l2norm,
                          threads=threads)


def decode(q, k, v, a, beta, states, slots, *, scale, l2norm=True, eps=L2NORM_EPS):
    """One decode token per batch row. q, k [B, H_k, d]; v [B, H_v, d]; a, beta [B, H_v];
    states [S, H_v, d_v, d_k] (a copy is updated and returned); slots [B] int.
    Returns (o [B, H_v, d_v], new_states) in fp64."""
    lib = _load()
    q, k, v, a, beta = map(_f64, (q, k, v, a, beta))
    st = np.array(states, dtype=np.float64, copy=True, order="C")
    slots = np.ascontiguousarray(slots, dtype=np.int32)
    B, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    o = np.zeros((B, Hv, dv), dtype=np.float64)
    rc = lib.gdn_ref_decode(B, Hk, Hv, dk, dv, float(scale), int(bool(l2norm)), float(eps),
                            _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(st),
                            _ptr(slots), _ptr(o))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")
    return o, st


def prefill_py(cu_seqlens, q, k, v, a, beta, init, ckpt_cu, ckpt_pos, *, scale,
               l2norm=True, eps=L2NORM_EPS):
    """The same definition as gdn_ref.c written with NumPy row operations; slow, for tiny
    cases. Kept so the C build can be checked against an independent transcription."""
    cu = [int(x) for x in cu_seqlens]
    q, k, v, a, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, a, beta))
    N = len(cu) - 1
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    G = Hv // Hk
    o = np.zeros((T, Hv, dv))
    C = 0 if ckpt_cu is None else int(ckpt_cu[-1])
    ck = np.zeros((C, Hv, dv, dk))
    fin = np.zeros((N, Hv, dv, dk))
    for n in range(N):
        for h in range(Hv):
            S = np.zeros((dv, dk)) if init is None else np.array(init[n, h], dtype=np.float64)
            slots = {} if ckpt_cu is None else {
                int(ckpt_pos[j]): j for j in range(int(ckpt_cu[n]), int(ckpt_cu[n + 1]))}
            for t in range(cu[n + 1] - cu[n]):
                tok = cu[n] + t
                qt, kt = q[tok, h // G].copy(), k[tok, h // G].copy()
                if l2norm:
                    qt = qt / np.sqrt(np.dot(qt, qt) + eps)
                    kt = kt / np.sqrt(np.dot(kt, kt) + eps)
                S = np.exp(a[tok, h]) * S
                delta = beta[tok, h] * (v[tok, h] - S @ kt)
                S = S + np.outer(delta, kt)
                o[tok, h] = scale * (S @ qt)
                if t + 1 in slots:
                    ck[slots[t + 1], h] = S
            fin[n, h] = S
    return o, ck, fin
