"""Checkpoint snapshots copied into the handle's pinned pool while the scan still runs
("the scan and the checkpoint copy run on separate streams, not one after another",
sparkinfer v0.6.28 release notes, bullet 2): gdn_prefill_packed_snapshot gives the same
bits as gdn_prefill_packed, the pool holds exactly the device checkpoints, and a consumer
stream ordered by gdn_checkpoint_copy_join (no host wait) reads the finished snapshots."""
import numpy as np
import pytest

from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import handle, run, torch_cuda

pytestmark = pytest.mark.gpu


def _pool_view(torch, h, nbytes, offset=0):
    addr, size = gdn.gdn_pool_info(h)
    assert offset + nbytes <= size
    import ctypes
    raw = (ctypes.c_uint8 * nbytes).from_address(addr + offset)
    return np.frombuffer(raw, dtype=np.uint8)


@pytest.mark.parametrize("pack_name", ["ragged", "wave"])
def test_snapshot_equals_prefill_and_pool_holds_checkpoints(pack_name):
    torch = torch_cuda()
    h = handle()
    p = I.ragged_prefix() if pack_name == "ragged" else I.chat_wave()
    want = run(p)
    buf = gdn.to_device(p)
    nbytes = buf.ckpt.numel() * 4
    offset = 4096
    pool = _pool_view(torch, h, nbytes, offset)
    pool[:] = 0xFF  # NaN bytes: a snapshot that is not written shows
    gdn.prefill_snapshot(h, buf, offset)
    gdn.gdn_checkpoint_copy_wait(h)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status(buf.workspace) == 0
    assert gdn.gdn_prefill_launch_count(h) == 1
    got = (buf.o.float().cpu().numpy().astype(np.float64), buf.ckpt.cpu().numpy(),
           buf.final.cpu().numpy())
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1].astype(np.float64), want[1])
    np.testing.assert_array_equal(got[2].astype(np.float64), want[2])
    np.testing.assert_array_equal(pool.view(np.float32).reshape(got[1].shape), got[1])


def test_consumer_stream_joined_on_the_device_sees_the_snapshots():
    torch = torch_cuda()
    h = handle()
    p = I.ragged_prefix()
    buf = gdn.to_device(p)
    nbytes = buf.ckpt.numel() * 4
    pool = _pool_view(torch, h, nbytes)
    addr, _ = gdn.gdn_pool_info(h)
    host_src = torch.from_numpy(pool.view(np.uint8))  # the pinned pool as a CPU tensor
    for rep in range(2):
        pool[:] = 0xFF
        consumer = torch.cuda.Stream()
        dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        gdn.prefill_snapshot(h, buf, 0, torch.cuda.current_stream())
        gdn.gdn_checkpoint_copy_join(h, consumer)  # device-side ordering only
        ev = gdn.gdn_checkpoint_copy_event(h)
        assert ev != 0
        with torch.cuda.stream(consumer):
            dst.copy_(host_src, non_blocking=True)  # reads the pinned pool after the join
        consumer.synchronize()  # the only host wait: on the consumer stream
        got = dst.cpu().numpy().view(np.float32)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got, buf.ckpt.cpu().numpy().reshape(-1))
    assert gdn.gdn_checkpoint_copy_query(h)


def test_snapshot_pool_bounds():
    torch = torch_cuda()
    h = handle()
    p = I.ragged_prefix()
    buf = gdn.to_device(p)
    _, size = gdn.gdn_pool_info(h)
    st = gdn.gdn_prefill_packed_snapshot(h, buf.cfg, buf.cu, buf.q, buf.k, buf.v, buf.a,
                                         buf.beta, buf.init, buf.ckpt_cu, buf.ckpt_pos, buf.o,
                                         buf.ckpt, buf.final, size - 16, buf.workspace,
                                         buf.workspace_bytes, raise_on_error=False)
    assert st == gdn.GDN_ERR_POOL_EXHAUSTED


@pytest.mark.parametrize("pref", [gdn.KERNEL_CHUNKED_PIPELINED, gdn.KERNEL_CHUNKED_THROUGHPUT])
def test_snapshot_copies_finish_after_a_device_timeout(pref):
    """With the test hook, every unit's first copy wait runs out. Each block still counts
    its prompt's arrival, so the side stream's waits end and the copies finish (polled
    here with a deadline, never waited on without one); the status word reports the
    timeout, and the next snapshot call on the same context is right."""
    import time
    torch = torch_cuda()
    h = handle()
    p = I.make_pack([200, 64, 5, 0], num_k_heads=2, num_v_heads=4, head_dim=128,
                    io_dtype="bf16", seed=43, init_std=0.02,
                    ckpt_lists=[[64, 200], [64], [5], []])
    buf = gdn.to_device(p)
    gdn.gdn_set_kernel_preference(h, pref)
    gdn.gdn_set_test_hook(h, 1)
    try:
        gdn.prefill_snapshot(h, buf, 0)
        deadline = time.monotonic() + 60.0
        while not gdn.gdn_checkpoint_copy_query(h):
            assert time.monotonic() < deadline, "the checkpoint copies never finished"
            time.sleep(0.01)
        status = gdn.gdn_read_device_status(buf.workspace)
    finally:
        gdn.gdn_set_test_hook(h, 0)
        gdn.gdn_set_kernel_preference(h, gdn.KERNEL_AUTO)
    assert status == gdn.GDN_ERR_DEVICE_TIMEOUT
    want = run(p, pref)
    nbytes = buf.ckpt.numel() * 4
    pool = _pool_view(torch, h, nbytes, 0)
    gdn.gdn_set_kernel_preference(h, pref)
    try:
        gdn.prefill_snapshot(h, buf, 0)
        gdn.gdn_checkpoint_copy_wait(h)
        torch.cuda.synchronize()
    finally:
        gdn.gdn_set_kernel_preference(h, gdn.KERNEL_AUTO)
    assert gdn.gdn_read_device_status(buf.workspace) == 0
    np.testing.assert_array_equal(buf.ckpt.cpu().numpy().astype(np.float64), want[1])
    np.testing.assert_array_equal(pool.view(np.float32).reshape(buf.ckpt.shape), want[1])
