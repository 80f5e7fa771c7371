"""The seeded workloads: bf16 rounding, the checkpoint move-back rule and the mixed-step
budget, each against hand-worked cases from the rules as the release notes state them."""
import numpy as np
import pytest
import torch

from packed_linear_attention_gb300 import inputs as I


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-8, 8, 100000),
                        np.array([1.0, -1.0, 0.0, 1.00390625, 1.01171875, 3.0e38], np.float32)]).astype(np.float32)
    ours = I.f32_to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, theirs)
    back = I.bf16_bits_to_f32(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("length,expect", [
    (1024, 768),    # last multiple of 256 is the length itself: inside the last 16 tokens
    (1000, 768),    # 768 <= 1000 - 16: stays
    (1030, 768),    # 1024 > 1014: moves back
    (1041, 1024),   # 1024 <= 1025: stays
    (1040, 1024),   # 1024 <= 1024: stays (exactly 16 tokens left)
    (1039, 768),    # 1024 > 1023: moves back
    (270, 0),       # 256 > 254: moves back to 0 -> no checkpoint
    (255, 0),
])
def test_move_back_rule(length, expect):
    assert I.ckpt_position_with_move_back(length, 256, 16) == expect


def test_mixed_budget_oldest_first():
    assert I.mixed_budget([300, 500, 400, 100], 1024, 8) == [300, 500, 224, 0]
    assert I.mixed_budget([100] * 10, 1024, 8) == [100] * 8 + [0, 0]
    assert I.mixed_budget([2000, 10], 1024, 8) == [1024, 0]


def test_workload_shapes():
    p = I.tiny_f32()
    assert p.lengths.tolist() == [17, 64, 100, 255]
    assert p.ckpt_pos.tolist() == [64, 64, 64, 128, 192]
    assert p.ckpt_cu.tolist() == [0, 0, 1, 2, 5]
    r = I.ragged_prefix()
    assert r.num_seqs == 8 and all(128 <= n <= 2048 for n in r.lengths)
    assert r.init is not None and abs(float(r.init.std()) - 0.02) < 1e-3
    # q, k are unit rows before the bf16 cast
    qn = np.linalg.norm(r.as_f32("q"), axis=-1)
    assert np.all(np.abs(qn - 1) < 1e-2)
    assert np.all(r.a < 0) and np.all((r.beta > 0) & (r.beta < 1))


def test_long_decay_mean():
    p = I.make_pack([4096], num_k_heads=1, num_v_heads=8, head_dim=4, io_dtype="f32",
                    decay_scale=I.LONG_DECAY_SCALE)
    assert abs(float(p.a.mean()) + 0.05) < 2e-3


def test_sub_pack_keeps_gqa_map():
    p = I.make_pack([5, 6, 7], num_k_heads=4, num_v_heads=8, head_dim=4, io_dtype="f32")
    s = I.sub_pack(p, [1], v_heads=[2, 3])
    assert s.num_k_heads == 1 and s.num_v_heads == 2
    np.testing.assert_array_equal(s.k[:, 0], p.k[5:11, 1])
    np.testing.assert_array_equal(s.v[:, 1], p.v[5:11, 3])
