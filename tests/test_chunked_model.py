"""The chunked (UT/WY) algebra that the kernel evaluates equals the token-by-token oracle
in exact arithmetic (fp64 agreement to ~1e-12) for any chunk size and ragged tails."""
import numpy as np
import pytest

from oracle import chunked_model as cm
from oracle import ref
from packed_linear_attention_gb300 import inputs as I


def _args(p):
    return (p.cu_seqlens, p.as_f32("q"), p.as_f32("k"), p.as_f32("v"), p.a, p.beta, p.init,
            p.ckpt_cu, p.ckpt_pos)


def _rel(x, y):
    return np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300)


def test_chunked_equals_oracle_tiny():
    p = I.tiny_f32()
    o, ck, fin = ref.prefill(p)
    o2, ck2, fin2 = cm.prefill(*_args(p), scale=p.scale, chunk=64)
    assert _rel(o2, o) < 1e-12 and _rel(ck2, ck) < 1e-12 and _rel(fin2, fin) < 1e-12


@pytest.mark.parametrize("chunk", [1, 5, 16, 64])
def test_chunked_equals_oracle_any_chunk(chunk):
    lengths = [1, 2, 63, 64, 65, 130]
    p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=16, io_dtype="bf16",
                    seed=21, init_std=0.02,
                    ckpt_lists=[[n] for n in lengths])
    o, ck, fin = ref.prefill(p)
    o2, ck2, fin2 = cm.prefill(*_args(p), scale=p.scale, chunk=chunk)
    assert _rel(o2, o) < 1e-12 and _rel(ck2, ck) < 1e-12 and _rel(fin2, fin) < 1e-12


def test_chunked_equals_oracle_ragged_wave_heads():
    p = I.sub_pack(I.ragged_prefix(), [0, 1], v_heads=[0, 1])
    o, ck, fin = ref.prefill(p)
    o2, ck2, fin2 = cm.prefill(*_args(p), scale=p.scale, chunk=64)
    assert _rel(o2, o) < 1e-12 and _rel(ck2, ck) < 1e-12 and _rel(fin2, fin) < 1e-12


def test_fp16_operands_fit_the_bf16_budget():
    """Rounding every tensor-core operand once to fp16 (q, k normalised first) keeps o
    within rel-L2 2e-3 after the bf16 output cast, and states far inside it."""
    p = I.sub_pack(I.chat_wave(num_prompts=1, length=512), [0], v_heads=[0, 1])
    o, ck, fin = ref.prefill(p)

    def nf16(x):
        x32 = x.astype(np.float32)
        n = np.sqrt(np.sum(x32 * x32, axis=-1, keepdims=True) + np.float32(1e-6))
        return (x32 / n).astype(np.float16).astype(np.float64)

    H = "f16"
    prec = dict(T=(H, H), WK=(H, H), US=(H, H), QS=(H, H), PD=(H, H), DK=(H, H), inv="f32")
    o2, ck2, fin2 = cm.prefill(p.cu_seqlens, nf16(p.as_f32("q")), nf16(p.as_f32("k")),
                               p.as_f32("v").astype(np.float16), p.a, p.beta, None,
                               p.ckpt_cu, p.ckpt_pos, scale=p.scale, prec=prec, l2norm=False)
    assert _rel(cm._bf16(o2), o) < 2e-3
    assert _rel(fin2, fin) < 2e-3 and np.abs(fin2 - fin).max() < 1e-2
