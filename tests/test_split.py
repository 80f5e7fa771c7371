"""Sequence splitting (gdn_prefill_packed_split): prompts longer than a segment length run
as parallel segments whose affine state maps are composed and then re-run from their true
initial states. CPU tests cover the planner's validation and sizes; GPU tests compare the
split path with the fp64 oracle (the unsplit definition), across segment boundaries,
checkpoints on and off them, initial states, both chunked schedules and the token-serial
kernel, and check that prompts short enough to stay whole are computed exactly as by
gdn_prefill_packed."""
import numpy as np
import pytest

from packed_linear_attention_gb300 import build, gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import compare_units, handle, run, torch_cuda

CFG = dict(num_k_heads=16, num_v_heads=32, head_dim=128)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gdn.load()


def test_split_size_validation(lib):
    cfg = gdn.make_config(**CFG)
    cu = [0, 1000, 1100]
    base = gdn.gdn_prefill_split_workspace_size(cfg, cu, segment_len=256)
    assert base % 256 == 0 and base > 0
    for bad in (0, 32, 100, -64):
        with pytest.raises(gdn.GdnError) as e:
            gdn.gdn_prefill_split_workspace_size(cfg, cu, segment_len=bad)
        assert e.value.status == gdn.GDN_ERR_INVALID_ARGUMENT
    # shorter segments: more maps and split segments, so more scratch
    assert gdn.gdn_prefill_split_workspace_size(cfg, cu, segment_len=128) > base
    # nothing to split: only the work list and segment-0 states
    small = gdn.gdn_prefill_split_workspace_size(cfg, cu, segment_len=1024)
    assert small < base
    # checkpoints validated as for gdn_prefill_packed (off the chunk grid: unsupported)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill_split_workspace_size(cfg, cu, [0, 1, 1], [50], segment_len=256)
    assert e.value.status == gdn.GDN_ERR_UNSUPPORTED


def _split_run(pack, seg, pref=gdn.KERNEL_AUTO):
    torch = torch_cuda()
    h = handle()
    gdn.gdn_set_kernel_preference(h, pref)
    try:
        buf = gdn.to_device(pack)
        gdn.prefill_split(h, buf, seg)
        torch.cuda.synchronize()
        assert gdn.gdn_read_device_status(buf.split_workspace) == 0
    finally:
        gdn.gdn_set_kernel_preference(h, gdn.KERNEL_AUTO)
    return (buf.o.float().cpu().numpy().astype(np.float64),
            buf.ckpt.cpu().numpy().astype(np.float64),
            buf.final.cpu().numpy().astype(np.float64))


PREFS = [gdn.KERNEL_CHUNKED_PIPELINED, gdn.KERNEL_CHUNKED_THROUGHPUT, gdn.KERNEL_RECURRENT]


@pytest.mark.gpu
@pytest.mark.parametrize("pref", PREFS)
def test_split_vs_oracle(pref):
    """A pack mixing split and whole prompts: 4 segments (the last ragged), 2 segments,
    whole, empty; checkpoints inside segments, on segment boundaries and at the ends."""
    lengths = [1000, 300, 100, 0, 513]
    ck = [[128, 256, 512, 768, 1000], [256, 300], [64], [], [64, 512, 513]]
    p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                    seed=21, init_std=0.02, ckpt_lists=ck)
    got = _split_run(p, 256, pref)
    compare_units(p, got, list(range(len(lengths))), list(range(4)))


@pytest.mark.gpu
def test_split_fp32_d64_vs_oracle():
    """The token-serial family (fp32 io, d = 64) through the split path."""
    lengths = [700, 64]
    ck = [[192, 384, 700], [64]]
    p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=64, io_dtype="f32",
                    seed=22, init_std=0.05, ckpt_lists=ck)
    got = _split_run(p, 192)
    compare_units(p, got, [0, 1], list(range(4)))


@pytest.mark.gpu
def test_split_raw_gates_vs_oracle():
    base = I.make_pack([900], num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                       seed=23, init_std=0.02, ckpt_lists=[[448, 900]])
    p = I.with_raw_gates(base, seed=4)
    got = _split_run(p, 320)
    compare_units(p, got, [0], list(range(4)))


@pytest.mark.gpu
@pytest.mark.parametrize("pref", [gdn.KERNEL_AUTO, gdn.KERNEL_CHUNKED_PIPELINED,
                                  gdn.KERNEL_CHUNKED_THROUGHPUT])
def test_whole_prompts_match_gdn_prefill_packed_bitwise(pref):
    """Prompts no longer than the segment length are computed exactly as by
    gdn_prefill_packed (under the automatic choice too: both chunked schedules agree bit
    for bit)."""
    lengths = [300, 64, 1, 255]
    ck = [[128, 300], [64], [], [192]]
    p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                    seed=24, init_std=0.02, ckpt_lists=ck)
    a = run(p, pref)
    b = _split_run(p, 512, pref)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.gpu
def test_split_long_prompt_full_heads_sampled():
    """One 8K-token prompt at the wave's dims, cut in 3 segments (the bench's split case
    shape), sampled value heads against the oracle."""
    p = I.make_pack([8192], **CFG, io_dtype="bf16", seed=25, init_std=0.02,
                    ckpt_lists=[[4096, 8192]], decay_scale=I.LONG_DECAY_SCALE)
    got = _split_run(p, 2752)
    compare_units(p, got, [0], [0, 1, 30, 31])
