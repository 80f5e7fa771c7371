"""The device-side timeout path of the chunked kernels, made to run without a GPU fault:
with the test hook set (gdn_set_test_hook), each unit's first q/k copy is left out, so its
first bounded wait runs out after about a second. The kernel must then record
GDN_ERR_DEVICE_TIMEOUT in the status word, let what it issued land, free its tensor memory
and return; a following call on the same context must compute the right answer."""
import time

import pytest

from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import compare_units, handle, run, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pref", [gdn.KERNEL_CHUNKED_PIPELINED, gdn.KERNEL_CHUNKED_THROUGHPUT])
def test_first_copy_wait_runs_out_then_next_call_is_correct(pref):
    torch = torch_cuda()
    p = I.make_pack([200, 64, 5, 0], num_k_heads=2, num_v_heads=4, head_dim=128,
                    io_dtype="bf16", seed=41, init_std=0.02,
                    ckpt_lists=[[64, 200], [64], [5], []])
    h = handle()
    buf = gdn.to_device(p)
    gdn.gdn_set_kernel_preference(h, pref)
    gdn.gdn_set_test_hook(h, 1)
    try:
        t0 = time.monotonic()
        gdn.prefill(h, buf)
        status = gdn.gdn_read_device_status(buf.workspace)  # synchronises the stream
        elapsed = time.monotonic() - t0
    finally:
        gdn.gdn_set_test_hook(h, 0)
        gdn.gdn_set_kernel_preference(h, gdn.KERNEL_AUTO)
    assert status == gdn.GDN_ERR_DEVICE_TIMEOUT
    assert elapsed < 30.0, elapsed  # each wait is bounded by about a second
    # same context, same buffers: a normal call succeeds and is right
    got = run(p, pref, buf=buf)
    compare_units(p, got, [0, 1, 2, 3], list(range(4)))
