"""gdn_prefill_packed_host: inputs and outputs in pinned host memory, processed in groups of
prompts whose copies overlap their neighbours' prefill. Results against gdn_prefill_packed
on the same pack (bitwise, also under the automatic choice: results do not depend on
packing, and both chunked schedules agree bit for bit) and against the oracle. Group sizes
ramp up 1, 2, 4, ... at the start and down at the end."""
import numpy as np
import pytest

from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import compare_units, handle, run, torch_cuda

pytestmark = pytest.mark.gpu


def _host_run(pack, group, pref=gdn.KERNEL_AUTO):
    torch = torch_cuda()
    h = handle()
    gdn.gdn_set_kernel_preference(h, pref)
    try:
        buf = gdn.to_device(pack)
        pin = lambda t: t.cpu().pin_memory()
        hq, hk, hv, ha, hb = (pin(getattr(buf, n)) for n in ("q", "k", "v", "a", "beta"))
        hi = pin(buf.init) if buf.init is not None else None
        ho = torch.empty(buf.o.shape, dtype=buf.o.dtype).pin_memory()
        hc = torch.full(buf.ckpt.shape, float("nan")).pin_memory()
        hf = torch.full(buf.final.shape, float("nan")).pin_memory()
        # the device copies start from garbage: every input must come from the host
        for t in (buf.q, buf.k, buf.v):
            t.zero_()
        buf.a.fill_(float("nan"))
        if buf.init is not None:
            buf.init.fill_(float("nan"))
        has_ck = buf.ckpt.numel() > 0
        host = gdn.prefill_buffers(hq, hk, hv, ha, hb, hi, ho, hc if has_ck else None, hf)
        dev = gdn.prefill_buffers(buf.q, buf.k, buf.v, buf.a, buf.beta, buf.init, buf.o,
                                  buf.ckpt if has_ck else None, buf.final)
        stream = torch.cuda.current_stream()
        nbytes = gdn.gdn_prefill_host_workspace_size(buf.cfg, buf.cu, buf.ckpt_cu, group)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        gdn.gdn_prefill_packed_host(h, buf.cfg, buf.cu, buf.ckpt_cu,
                                    buf.ckpt_pos if has_ck else None, host, dev, group,
                                    ws, nbytes, stream)
        stream.synchronize()
        assert gdn.gdn_read_device_status(ws) == 0
    finally:
        gdn.gdn_set_kernel_preference(h, gdn.KERNEL_AUTO)
    return (ho.float().numpy().astype(np.float64), hc.numpy().astype(np.float64),
            hf.numpy().astype(np.float64))


@pytest.mark.parametrize("group", [1, 3, 16])
@pytest.mark.parametrize("pref", [gdn.KERNEL_AUTO, gdn.KERNEL_CHUNKED_PIPELINED,
                                  gdn.KERNEL_CHUNKED_THROUGHPUT, gdn.KERNEL_RECURRENT])
def test_host_prefill_equals_device_prefill(group, pref):
    lengths = [300, 64, 0, 1, 700, 129, 65]
    ck = [[64, 300], [64], [], [1], [256, 512, 700], [128], []]
    p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                    seed=31, init_std=0.02, ckpt_lists=ck)
    want = run(p, pref)
    got = _host_run(p, group, pref)
    for x, y in zip(got, want):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("group", [4, 8])
def test_host_prefill_wave_vs_oracle(group):
    """The bench's e2e configuration (the wave in groups of 4 prompts, and of 8), sampled
    against the oracle: prompts in the first, a middle and the last group."""
    p = I.chat_wave()
    got = _host_run(p, group)
    compare_units(p, got, [0, 9, 31], [0, 1, 30, 31])


def test_host_prefill_no_checkpoints_no_init():
    p = I.make_pack([100, 200], num_k_heads=2, num_v_heads=4, head_dim=64, io_dtype="f32",
                    seed=32)
    want = run(p)
    got = _host_run(p, 1)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[2], want[2])

