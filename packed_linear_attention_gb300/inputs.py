"""Seeded synthetic workloads for packed GDN prefill and decode.

This module only draws inputs: prompt lengths, q/k/v activations, log-decays, write
strengths, initial states and checkpoint positions. It holds none of the layer's
arithmetic, so the CUDA path and the CPU oracle can both be fed from it.

Recipe (one NumPy PCG64 generator per workload, seed 0 unless given; all draws fp32, in
the order lengths, q, k, v, a_raw, b_raw, initial state):
  * q, k ~ N(0, 1), then L2-normalised per (token, key head) in fp32;
  * v ~ N(0, 1);
  * a = -c * softplus(z), z ~ N(0, 1) (c = 1, or c = 0.05 / E[softplus(z)] for the slow
    decay of the 8K-prompt pack), so g = exp(a) lies in (0, 1);
  * beta = sigmoid(z'), z' ~ N(0, 1);
  * prefix-cache initial states ~ N(0, 0.02) (0.02 is the standard deviation);
  * q, k, v are then rounded to bf16 (round to nearest even) for the bf16 workloads; the
    rounded values are the inputs both sides read.

The workload shapes follow the serving pages: a wave of 32 new 1,024-token chat prompts
prefilled in packed passes (sparkinfer v0.6.28 release notes, intro and "Measured"),
8K-token prompts (same table), prefix-cache hits that resume from a stored state
(sparkinfer v0.6.28, checkpoint bullets) and mixed steps that fill a 1,024-token prompt
budget across at most 8 waiting prompts, oldest first, beside decoding requests
(sparkinfer v0.6.4, "What changed"). No dataset is used; these draws stand in for the
prompt sets of those benchmarks.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# E[softplus(z)] for z ~ N(0, 1) (numerical quadrature), used to give the 8K-prompt pack
# a mean log-decay of -0.05 per token.
MEAN_SOFTPLUS_STD_NORMAL = 0.8060592
LONG_DECAY_SCALE = 0.05 / MEAN_SOFTPLUS_STD_NORMAL


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16, round-to-nearest-even; returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + (((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF))
    return (rounded >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Pack:
    """One packed prefill call's inputs (host arrays).

    q, k: [T, H_k, d]; v: [T, H_v, d] -- uint16 bf16 bits when io_dtype == "bf16",
    float32 when io_dtype == "f32". a, beta: [T, H_v] float32. init: [N, H_v, d, d]
    float32 or None. ckpt_cu: [N+1] int32 CSR over ckpt_pos (prompt-relative positions).
    """

    name: str
    cu_seqlens: np.ndarray
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    a: np.ndarray
    beta: np.ndarray
    init: Optional[np.ndarray]
    ckpt_cu: np.ndarray
    ckpt_pos: np.ndarray
    num_k_heads: int
    num_v_heads: int
    head_dim: int
    io_dtype: str
    scale: float
    chunk_size: int = 64
    qk_l2norm: bool = True
    meta: dict = field(default_factory=dict)
    # raw gate inputs: when set, a and beta hold the raw projections a_raw and b_raw
    a_log: Optional[np.ndarray] = None     # [H_v] float32
    dt_bias: Optional[np.ndarray] = None   # [H_v] float32

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def lengths(self) -> np.ndarray:
        return np.diff(self.cu_seqlens).astype(np.int64)

    @property
    def num_ckpts(self) -> int:
        return int(self.ckpt_cu[-1])

    def as_f32(self, name: str) -> np.ndarray:
        """q, k or v widened exactly to fp32 (the values both sides read)."""
        x = getattr(self, name)
        return bf16_bits_to_f32(x) if self.io_dtype == "bf16" else np.asarray(x, np.float32)


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def _l2norm_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x.astype(np.float32) ** 2, axis=-1, keepdims=True, dtype=np.float32))
    return (x / np.maximum(n, np.float32(1e-12))).astype(np.float32)


def _softplus(z: np.ndarray) -> np.ndarray:
    return np.logaddexp(np.float32(0), z).astype(np.float32)


def _sigmoid(z: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-z.astype(np.float64)))).astype(np.float32)


def ckpt_position_with_move_back(length: int, block: int, tail: int) -> int:
    """Last multiple of `block` <= length, moved back one block when it lies within the
    last `tail` tokens (sparkinfer v0.6.28 release notes, bullet on checkpoints in a
    prompt's last 16 tokens). 0 means no checkpoint."""
    p = (length // block) * block
    if p > length - tail:
        p -= block
    return max(p, 0)


def csr_from_lists(per_seq: list[list[int]]) -> tuple[np.ndarray, np.ndarray]:
    cu = np.zeros(len(per_seq) + 1, dtype=np.int32)
    for i, lst in enumerate(per_seq):
        cu[i + 1] = cu[i] + len(lst)
    pos = np.array([p for lst in per_seq for p in lst], dtype=np.int32)
    return cu, pos


def every_block(lengths, block: int) -> list[list[int]]:
    """Checkpoints at every multiple of `block` up to and including the prompt length."""
    return [list(range(block, int(n) + 1, block)) for n in lengths]


def make_pack(
    lengths,
    *,
    num_k_heads: int,
    num_v_heads: int,
    head_dim: int,
    io_dtype: str = "bf16",
    seed: int = 0,
    init_std: Optional[float] = None,
    decay_scale: float = 1.0,
    ckpt_lists: Optional[list[list[int]]] = None,
    scale: Optional[float] = None,
    chunk_size: int = 64,
    name: str = "custom",
    rng: Optional[np.random.Generator] = None,
) -> Pack:
    """Draw one pack with the recipe in the module docstring."""
    lengths = [int(x) for x in lengths]
    if rng is None:
        rng = np.random.default_rng(seed)
    N, T, d = len(lengths), int(sum(lengths)), head_dim
    cu = np.zeros(N + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    q = _l2norm_rows(_normal(rng, (T, num_k_heads, d)))
    k = _l2norm_rows(_normal(rng, (T, num_k_heads, d)))
    v = _normal(rng, (T, num_v_heads, d))
    a = (-np.float32(decay_scale) * _softplus(_normal(rng, (T, num_v_heads)))).astype(np.float32)
    beta = _sigmoid(_normal(rng, (T, num_v_heads)))
    init = None
    if init_std is not None:
        init = (np.float32(init_std) * _normal(rng, (N, num_v_heads, d, d))).astype(np.float32)
    if io_dtype == "bf16":
        q, k, v = f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v)
    elif io_dtype != "f32":
        raise ValueError(io_dtype)
    if ckpt_lists is None:
        ckpt_lists = [[] for _ in lengths]
    ckpt_cu, ckpt_pos = csr_from_lists(ckpt_lists)
    return Pack(
        name=name, cu_seqlens=cu, q=q, k=k, v=v, a=a, beta=beta, init=init,
        ckpt_cu=ckpt_cu, ckpt_pos=ckpt_pos, num_k_heads=num_k_heads,
        num_v_heads=num_v_heads, head_dim=d, io_dtype=io_dtype,
        scale=float(scale if scale is not None else 1.0 / np.sqrt(d)),
        chunk_size=chunk_size,
    )


# ---- the named workloads ------------------------------------------------------------------

WAVE_HEADS = dict(num_k_heads=16, num_v_heads=32, head_dim=128)


def tiny_f32(seed: int = 0) -> Pack:
    """4 prompts {17, 64, 100, 255}, H_k=2, H_v=4, d=64, fp32 io, zero initial states,
    checkpoints at every multiple of 64 (the final state is always returned as well)."""
    lengths = [17, 64, 100, 255]
    return make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=64, io_dtype="f32",
                     seed=seed, ckpt_lists=every_block(lengths, 64), name="tiny_f32")


def chat_wave(num_prompts: int = 32, length: int = 1024, seed: int = 0) -> Pack:
    """A wave of 32 new 1,024-token prompts in one pack, bf16 io, zero initial states; one
    prefix-cache checkpoint per prompt at the last multiple of 256 <= length, moved back a
    256-token block when it falls in the last 16 tokens (1024 -> 768)."""
    lengths = [length] * num_prompts
    p = ckpt_position_with_move_back(length, 256, 16)
    ck = [[p] if p > 0 else [] for _ in lengths]
    return make_pack(lengths, **WAVE_HEADS, io_dtype="bf16", seed=seed, ckpt_lists=ck,
                     name=f"chat_wave_{num_prompts}x{length}")


def ragged_prefix(seed: int = 0, num_prompts: int = 8) -> Pack:
    """8 prompts with lengths uniform in [128, 2048], each resuming from a nonzero fp32
    prefix-cache state ~ N(0, 0.02); checkpoints every 256 tokens."""
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(128, 2049, size=num_prompts)]
    return make_pack(lengths, **WAVE_HEADS, io_dtype="bf16", rng=rng, init_std=0.02,
                     ckpt_lists=every_block(lengths, 256), name="ragged_prefix")


def long_prompts(num_prompts: int = 4, length: int = 8192, seed: int = 0) -> Pack:
    """4 prompts x 8,192 tokens, slow decay (mean log-decay -0.05), checkpoints every
    1,024 tokens."""
    lengths = [length] * num_prompts
    return make_pack(lengths, **WAVE_HEADS, io_dtype="bf16", seed=seed,
                     decay_scale=LONG_DECAY_SCALE, ckpt_lists=every_block(lengths, 1024),
                     name=f"long_{num_prompts}x{length}")


def single_long_prompt(length: int = 32768, seed: int = 0) -> Pack:
    """One long-context prompt (32,768 tokens at the wave's dims, slow decay as for the 8K
    prompts, checkpoints every 8,192 tokens): the shape where N H_v = 32 units leave most
    SMs idle, for sequence splitting."""
    return make_pack([length], **WAVE_HEADS, io_dtype="bf16", seed=seed,
                     decay_scale=LONG_DECAY_SCALE, ckpt_lists=every_block([length], 8192),
                     name="single_long_prompt")


def mixed_budget(remaining, budget: int = 1024, max_prompts: int = 8) -> list[int]:
    """Oldest-first split of a prompt-token budget (sparkinfer v0.6.4, "What changed")."""
    take, left = [], budget
    for i, r in enumerate(remaining):
        if i >= max_prompts or left <= 0:
            take.append(0)
            continue
        t = min(int(r), left)
        take.append(t)
        left -= t
    return take


@dataclass
class MixedStep:
    """A mixed step: prompt slices (a prefill pack starting from zero states) plus one
    decode token for each of `decode.batch` sequences resumed from stored states."""

    prefill: Pack
    prompt_lengths: list
    take: list
    dec_q: np.ndarray
    dec_k: np.ndarray
    dec_v: np.ndarray
    dec_a: np.ndarray
    dec_beta: np.ndarray
    dec_states: np.ndarray    # [B, H_v, d, d] float32
    io_dtype: str = "bf16"


def mixed_step(seed: int = 0, num_waiting: int = 8, num_decoding: int = 32,
               budget: int = 1024) -> MixedStep:
    """8 waiting prompts with lengths uniform in [64, 256] served oldest first under a
    1,024-token prompt budget, plus 32 decoding sequences of one token each whose fp32
    states ~ N(0, 0.02)."""
    rng = np.random.default_rng(seed)
    prompt_lengths = [int(x) for x in rng.integers(64, 257, size=num_waiting)]
    take = mixed_budget(prompt_lengths, budget, 8)
    served = [t for t in take if t > 0]
    pre = make_pack(served, **WAVE_HEADS, io_dtype="bf16", rng=rng, name="mixed_prefill")
    H_k, H_v, d = WAVE_HEADS["num_k_heads"], WAVE_HEADS["num_v_heads"], WAVE_HEADS["head_dim"]
    B = num_decoding
    dq = f32_to_bf16_bits(_l2norm_rows(_normal(rng, (B, H_k, d))))
    dk = f32_to_bf16_bits(_l2norm_rows(_normal(rng, (B, H_k, d))))
    dv = f32_to_bf16_bits(_normal(rng, (B, H_v, d)))
    da = (-_softplus(_normal(rng, (B, H_v)))).astype(np.float32)
    db = _sigmoid(_normal(rng, (B, H_v)))
    ds = (np.float32(0.02) * _normal(rng, (B, H_v, d, d))).astype(np.float32)
    return MixedStep(prefill=pre, prompt_lengths=prompt_lengths, take=take, dec_q=dq,
                     dec_k=dk, dec_v=dv, dec_a=da, dec_beta=db, dec_states=ds)


def mixed_one_pack(ms: MixedStep) -> Pack:
    """The mixed step as one pack: the prompt slices (zero initial states) followed by one
    one-token prompt per decoding sequence (its stored state as initial state)."""
    pre = ms.prefill
    B = ms.dec_q.shape[0]
    lengths = list(pre.lengths) + [1] * B
    H_v, d = pre.num_v_heads, pre.head_dim
    return Pack(name="mixed_one_pack",
                cu_seqlens=np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32),
                q=np.concatenate([pre.q, ms.dec_q]), k=np.concatenate([pre.k, ms.dec_k]),
                v=np.concatenate([pre.v, ms.dec_v]), a=np.concatenate([pre.a, ms.dec_a]),
                beta=np.concatenate([pre.beta, ms.dec_beta]),
                init=np.concatenate([np.zeros((pre.num_seqs, H_v, d, d), np.float32),
                                     ms.dec_states]),
                ckpt_cu=np.zeros(len(lengths) + 1, np.int32), ckpt_pos=np.zeros(0, np.int32),
                num_k_heads=pre.num_k_heads, num_v_heads=H_v, head_dim=d, io_dtype="bf16",
                scale=pre.scale)


def with_raw_gates(p: Pack, seed: int = 0) -> Pack:
    """The same pack with raw gate projections instead of gates, drawn like a freshly
    initialised Qwen3.5/3.6-style GDN layer: a_raw, b_raw ~ N(0, 1); A = exp(A_log) ~ U(1, 16)
    per value head; dt ~ log-uniform in [1e-3, 1e-1] with dt_bias = softplus^-1(dt)."""
    rng = np.random.default_rng(seed + 7919)
    T, Hv = p.a.shape
    a_raw = _normal(rng, (T, Hv))
    b_raw = _normal(rng, (T, Hv))
    a_log = np.log(rng.uniform(1.0, 16.0, size=Hv)).astype(np.float32)
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), size=Hv))
    dt_bias = (dt + np.log(-np.expm1(-dt))).astype(np.float32)  # inverse softplus
    q = Pack(**{f: getattr(p, f) for f in p.__dataclass_fields__})
    q.a, q.beta, q.a_log, q.dt_bias = a_raw, b_raw, a_log, dt_bias
    q.name = p.name + "_raw_gates"
    return q


def sub_pack(p: Pack, seqs, v_heads=None) -> Pack:
    """The same inputs restricted to some prompts and (optionally) some value heads with
    their key heads, for sampled comparisons at full size. Value heads are taken as whole
    GQA groups' members; their key heads are remapped so head h keeps its key head."""
    seqs = [int(s) for s in seqs]
    G = p.num_v_heads // p.num_k_heads
    if v_heads is None:
        v_heads = list(range(p.num_v_heads))
    v_heads = [int(h) for h in v_heads]
    k_heads = sorted({h // G for h in v_heads})
    # one value head per key head keeps the mapping h -> h // G' with G' = 1 only when each
    # key head carries one selected value head; otherwise keep whole groups.
    groups = {kh: [h for h in v_heads if h // G == kh] for kh in k_heads}
    gsize = max(len(g) for g in groups.values())
    if any(len(g) != gsize for g in groups.values()):
        raise ValueError("select the same number of value heads from every key head")
    v_order = [h for kh in k_heads for h in groups[kh]]
    toks = np.concatenate([np.arange(p.cu_seqlens[s], p.cu_seqlens[s + 1]) for s in seqs]) \
        if seqs else np.zeros(0, dtype=np.int64)
    lengths = [int(p.cu_seqlens[s + 1] - p.cu_seqlens[s]) for s in seqs]
    cu = np.zeros(len(seqs) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    ck_lists = [list(p.ckpt_pos[p.ckpt_cu[s]:p.ckpt_cu[s + 1]]) for s in seqs]
    ckpt_cu, ckpt_pos = csr_from_lists(ck_lists)
    init = None
    if p.init is not None:
        init = np.ascontiguousarray(p.init[seqs][:, v_order])
    return Pack(
        name=p.name + "_sub", cu_seqlens=cu,
        q=np.ascontiguousarray(p.q[toks][:, k_heads]),
        k=np.ascontiguousarray(p.k[toks][:, k_heads]),
        v=np.ascontiguousarray(p.v[toks][:, v_order]),
        a=np.ascontiguousarray(p.a[toks][:, v_order]),
        beta=np.ascontiguousarray(p.beta[toks][:, v_order]),
        init=init, ckpt_cu=ckpt_cu, ckpt_pos=ckpt_pos,
        num_k_heads=len(k_heads), num_v_heads=len(v_order), head_dim=p.head_dim,
        io_dtype=p.io_dtype, scale=p.scale, chunk_size=p.chunk_size, qk_l2norm=p.qk_l2norm,
        meta=dict(parent=p.name, seqs=seqs, v_heads=v_order),
        a_log=None if p.a_log is None else np.ascontiguousarray(p.a_log[v_order]),
        dt_bias=None if p.dt_bias is None else np.ascontiguousarray(p.dt_bias[v_order]),
    )


WORKLOADS = {
    "tiny_f32": tiny_f32,
    "chat_wave": chat_wave,
    "ragged_prefix": ragged_prefix,
    "long_prompts": long_prompts,
}
