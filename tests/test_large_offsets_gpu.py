"""Offsets past 2^31 elements. Three prompts of 262,144 tokens at the wave's head dims (H_k 16,
H_v 32, d 128) give v and o 3.2e9 elements each (6.4 GB); the last prompt's rows start at
element 2^31 of them, past the int32 range. Checkpoints mid-prompt and at every prompt end, the default
(automatic) kernel. The last prompt's first and last value heads (key heads 0 and 15) are
compared with the oracle: o over all its tokens, its checkpoints and its final state.
The inputs repeat one seeded 4,096-token block (the generator's recipe), which keeps the
host side to a few seconds; about 19 GB of device memory."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import ref
from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import assert_close, handle, torch_cuda

pytestmark = pytest.mark.gpu

LEN, N, BLOCK = 262144, 3, 4096


def _pack() -> I.Pack:
    base = I.make_pack([BLOCK], **I.WAVE_HEADS, io_dtype="bf16", seed=61)
    reps = LEN * N // BLOCK
    tile = lambda x: np.tile(x, (reps,) + (1,) * (x.ndim - 1))  # noqa: E731
    ckpt_cu, ckpt_pos = I.csr_from_lists([[LEN], [LEN], [LEN // 2, LEN]])
    return I.Pack(name="large_offsets", cu_seqlens=np.arange(N + 1, dtype=np.int32) * LEN,
                  q=tile(base.q), k=tile(base.k), v=tile(base.v), a=tile(base.a),
                  beta=tile(base.beta), init=None, ckpt_cu=ckpt_cu, ckpt_pos=ckpt_pos,
                  num_k_heads=base.num_k_heads, num_v_heads=base.num_v_heads,
                  head_dim=base.head_dim, io_dtype="bf16", scale=base.scale)


def test_rows_past_two_to_the_31_elements():
    torch = torch_cuda()
    p = _pack()
    assert (N - 1) * LEN * p.num_v_heads * p.head_dim >= 2 ** 31  # first row past int32
    heads = [0, p.num_v_heads - 1]
    buf = gdn.to_device(p)
    try:
        gdn.prefill(handle(), buf)
        torch.cuda.synchronize()
        assert gdn.gdn_read_device_status(buf.workspace) == 0
        t0 = (N - 1) * LEN
        got_o = buf.o[t0:t0 + LEN][:, heads].float().cpu().numpy().astype(np.float64)
        c0, c1 = int(p.ckpt_cu[N - 1]), int(p.ckpt_cu[N])
        got_ck = buf.ckpt[c0:c1][:, heads].cpu().numpy().astype(np.float64)
        got_fin = buf.final[N - 1:N][:, heads].cpu().numpy().astype(np.float64)
    finally:
        del buf
        torch.cuda.empty_cache()
    ro, rck, rfin = ref.prefill(I.sub_pack(p, [N - 1], heads))
    assert np.isfinite(got_o).all()
    assert_close(got_o, ro, "bf16", "o")
    for j in range(rck.shape[0]):
        for hh in range(len(heads)):
            assert_close(got_ck[j, hh], rck[j, hh], "bf16", f"ckpt[{j},{hh}]")
    for hh in range(len(heads)):
        assert_close(got_fin[0, hh], rfin[0, hh], "bf16", f"final[{hh}]")
