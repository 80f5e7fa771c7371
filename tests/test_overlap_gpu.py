"""Prefill on the handle's own stream overlapping decode steps on the caller's stream.

This is the lifecycle of pegainfer PR #786 ("Changes"): at most one in-flight prefill on
an owned CUDA stream; completion events polled while decode runs; an explicit wait when
decoding stops; the stream drained on shutdown. The results must be the ones the
synchronous path gives, bit for bit."""
import numpy as np
import pytest

from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import handle, run, torch_cuda

pytestmark = pytest.mark.gpu


def _decode_setup(torch, seed=0):
    ms = I.mixed_step(seed=seed)
    up = lambda x: torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)  # noqa: E731
    B = ms.dec_q.shape[0]
    return dict(cfg=gdn.make_config(16, 32, 128), B=B, q=up(ms.dec_q), k=up(ms.dec_k),
                v=up(ms.dec_v), a=torch.from_numpy(ms.dec_a).cuda(),
                beta=torch.from_numpy(ms.dec_beta).cuda(),
                pool=torch.from_numpy(ms.dec_states).cuda(),
                slots=torch.arange(B, dtype=torch.int32, device="cuda"),
                o=torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda"))


def _decode(h, d, steps, stream=None):
    outs = []
    for _ in range(steps):
        gdn.gdn_decode_step(h, d["cfg"], d["B"], d["q"], d["k"], d["v"], d["a"], d["beta"],
                            d["pool"], d["B"], d["slots"], d["o"], stream)
        outs.append(d["o"].clone())
    return outs


def test_async_prefill_with_concurrent_decode_matches_sync():
    torch = torch_cuda()
    h = handle()
    pack = I.long_prompts(num_prompts=4, length=2048)
    want = run(pack)
    d_ref = _decode_setup(torch)
    ref_outs = _decode(h, d_ref, 6)
    torch.cuda.synchronize()

    buf = gdn.to_device(pack)
    d = _decode_setup(torch)
    stream = torch.cuda.current_stream()
    gdn.prefill_async(h, buf, stream)
    outs = _decode(h, d, 6, stream)           # decode keeps running on the caller's stream
    gdn.gdn_prefill_async_query(h)           # poll; either answer is fine here
    gdn.gdn_prefill_async_wait(h)
    assert gdn.gdn_prefill_async_query(h)
    torch.cuda.synchronize()
    for got, ref in zip(outs, ref_outs):
        assert torch.equal(got, ref)
    assert torch.equal(d["pool"], d_ref["pool"])
    np.testing.assert_array_equal(buf.o.float().cpu().numpy().astype(np.float64), want[0])
    np.testing.assert_array_equal(buf.ckpt.cpu().numpy().astype(np.float64), want[1])
    np.testing.assert_array_equal(buf.final.cpu().numpy().astype(np.float64), want[2])


def test_second_prefill_is_rejected_while_one_is_in_flight():
    torch = torch_cuda()
    h = handle()
    pack = I.long_prompts(num_prompts=4, length=8192)
    buf1, buf2 = gdn.to_device(pack), gdn.to_device(pack)
    torch.cuda.synchronize()
    gdn.prefill_async(h, buf1)
    still_running = not gdn.gdn_prefill_async_query(h)
    st = gdn.prefill_async(h, buf2, raise_on_error=False)
    if still_running:
        assert st == gdn.GDN_ERR_BUSY
    gdn.gdn_prefill_async_wait(h)
    if st == gdn.GDN_ERR_BUSY:  # nothing was enqueued: the second buffer is still untouched
        assert gdn.prefill_async(h, buf2) == gdn.GDN_OK
    gdn.gdn_prefill_async_wait(h)
    torch.cuda.synchronize()
    assert torch.equal(buf1.o, buf2.o) and torch.equal(buf1.final, buf2.final)


def test_join_orders_another_stream_after_the_prefill():
    torch = torch_cuda()
    h = handle()
    pack = I.make_pack([700, 300], num_k_heads=4, num_v_heads=8, head_dim=128, seed=9,
                       io_dtype="bf16")
    want = run(pack)
    buf = gdn.to_device(pack)
    side = torch.cuda.Stream()
    gdn.prefill_async(h, buf, torch.cuda.current_stream())
    gdn.gdn_prefill_async_join(h, side)
    with torch.cuda.stream(side):
        o_copy = buf.o.clone()            # ordered after the prefill by the join
    side.synchronize()
    np.testing.assert_array_equal(o_copy.float().cpu().numpy().astype(np.float64), want[0])
    gdn.gdn_prefill_async_wait(h)


def test_destroy_drains_the_prefill_stream():
    torch = torch_cuda()
    pack = I.make_pack([1024, 512, 64], num_k_heads=4, num_v_heads=8, head_dim=128, seed=10,
                       io_dtype="bf16", ckpt_lists=[[512], [], [64]])
    want = run(pack)
    own = gdn.gdn_handle_create(0, 0)
    buf = gdn.to_device(pack)
    torch.cuda.synchronize()
    gdn.prefill_async(own, buf)
    gdn.gdn_handle_destroy(own)               # must wait for the in-flight prefill
    np.testing.assert_array_equal(buf.o.float().cpu().numpy().astype(np.float64), want[0])
    np.testing.assert_array_equal(buf.final.cpu().numpy().astype(np.float64), want[2])
