"""gdn_prefill_packed_noalloc: the prefill entry point for callers that cannot allocate
memory at call time (a serving engine whose device memory all belongs to its own pool, or
a plugin whose host framework forbids allocation on the request path). It takes no
workspace and no handle; its work list lives in a fixed per-GPU device array.

Checked through the C ABI against gdn_prefill_packed on the same inputs, twice in a row
with different packs (the shared array must be fully rewritten by each call). This file
is collected last so a stop-at-first-failure run has already run every other test."""
import numpy as np
import pytest

from packed_linear_attention_gb300 import build, gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import assert_close, run, torch_cuda


def _noalloc(pack, buf=None):
    torch = torch_cuda()
    if buf is None:
        buf = gdn.to_device(pack)
    gdn.gdn_prefill_packed_noalloc(buf.cfg, buf.cu, buf.q, buf.k, buf.v, buf.a, buf.beta,
                                   buf.init, buf.ckpt_cu, buf.ckpt_pos, buf.o,
                                   buf.ckpt if buf.ckpt.numel() else None, buf.final)
    torch.cuda.synchronize()
    assert gdn.gdn_noalloc_read_status() == 0
    return (buf.o.float().cpu().numpy().astype(np.float64),
            buf.ckpt.cpu().numpy().astype(np.float64),
            buf.final.cpu().numpy().astype(np.float64))


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    torch_cuda()
    first = I.make_pack([300, 64, 1, 129], num_k_heads=4, num_v_heads=8, head_dim=128,
                        io_dtype="bf16", seed=31, init_std=0.02,
                        ckpt_lists=[[64, 256], [64], [1], [128, 129]])
    second = I.make_pack([77, 1024, 0, 5], num_k_heads=2, num_v_heads=4, head_dim=128,
                         io_dtype="bf16", seed=32, ckpt_lists=[[77], [512, 768], [], []])
    for pack in (first, second):
        want = run(pack)
        got = _noalloc(pack)
        for g, w, what in zip(got, want, ("o", "ckpt", "final")):
            assert_close(g, w, "bf16", f"noalloc {what}")


@pytest.mark.gpu
def test_noalloc_token_serial_path_fp32():
    torch_cuda()
    p = I.tiny_f32()
    want = run(p)
    got = _noalloc(p)
    for g, w, what in zip(got, want, ("o", "ckpt", "final")):
        assert_close(g, w, "f32", f"noalloc f32 {what}")


@pytest.mark.gpu
def test_noalloc_reports_a_device_timeout_then_recovers():
    """The status word of the fixed array is readable without allocating: with the test hook
    each unit's first copy wait runs out (about a second, no fault) and the status reads
    GDN_ERR_DEVICE_TIMEOUT; the next call on the same buffers is right and reads 0."""
    torch = torch_cuda()
    p = I.make_pack([200, 64, 5], num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                    seed=33, ckpt_lists=[[64, 200], [64], []])
    buf = gdn.to_device(p)
    gdn.gdn_noalloc_set_test_hook(1)
    try:
        gdn.gdn_prefill_packed_noalloc(buf.cfg, buf.cu, buf.q, buf.k, buf.v, buf.a, buf.beta,
                                       buf.init, buf.ckpt_cu, buf.ckpt_pos, buf.o, buf.ckpt,
                                       buf.final)
        assert gdn.gdn_noalloc_read_status() == gdn.GDN_ERR_DEVICE_TIMEOUT
    finally:
        gdn.gdn_noalloc_set_test_hook(0)
    got = _noalloc(p, buf)
    want = run(p)
    for g, w, what in zip(got, want, ("o", "ckpt", "final")):
        assert_close(g, w, "bf16", f"noalloc after timeout {what}")
    torch.cuda.synchronize()


def test_noalloc_rejects_work_lists_beyond_its_array():
    """Host-side size check: nothing is enqueued, so no GPU is needed."""
    build.build()
    cfg = gdn.make_config(16, 32, 128)
    n = 2100  # 2100 prompts x 32 value heads x 16-byte units > 1 MiB
    cu = np.arange(n + 1, dtype=np.int32)
    P = lambda i: (1 << 32) * (i + 1)  # distinct fake device ranges, never touched
    st = gdn.gdn_prefill_packed_noalloc(cfg, cu, P(1), P(2), P(3), P(4), P(5), None, None,
                                        None, P(6), None, P(7), raise_on_error=False)
    assert st == gdn.GDN_ERR_UNSUPPORTED
