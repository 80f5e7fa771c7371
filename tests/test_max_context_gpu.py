"""The longest context the pages serve: one prompt of 262,144 tokens, the max model length
of the serving recipe (vllm.cpp "vLLM, online serving", the `--max-model-len 262144` flag).

Every value head (H_k 1, H_v 2, d 128, slow decay) runs through the chunked kernel whole,
in both schedules, and through sequence splitting at the automatic segment length. o,
four checkpoints (every 65,536 tokens, the last one at the end) and the final states are
compared with the oracle. The case checks token and checkpoint positions far past the
packs elsewhere, and 4,096-chunk chains."""
from __future__ import annotations

import numpy as np
import pytest

from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import compare_units, handle, run, torch_cuda

LEN = 262144
CFG = dict(num_k_heads=1, num_v_heads=2, head_dim=128)


@pytest.fixture(scope="module")
def pack():
    return I.make_pack([LEN], **CFG, io_dtype="bf16", seed=41, init_std=0.02,
                       ckpt_lists=[[65536, 131072, 196608, LEN]],
                       decay_scale=I.LONG_DECAY_SCALE)


@pytest.mark.gpu
@pytest.mark.parametrize("pref", [gdn.KERNEL_AUTO, gdn.KERNEL_CHUNKED_THROUGHPUT])
def test_max_context_whole(pack, pref):
    compare_units(pack, run(pack, pref), [0], [0, 1])


@pytest.mark.gpu
def test_max_context_split_at_the_automatic_segment(pack):
    torch = torch_cuda()
    h = handle()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    seg = gdn.gdn_split_segment_auto(pack.cu_seqlens, CFG["num_v_heads"], sms)
    assert seg > 0  # two units for the whole GPU: the model splits
    buf = gdn.to_device(pack)
    gdn.prefill_split(h, buf, seg)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status(buf.split_workspace) == 0
    got = (buf.o.float().cpu().numpy().astype(np.float64),
           buf.ckpt.cpu().numpy().astype(np.float64),
           buf.final.cpu().numpy().astype(np.float64))
    compare_units(pack, got, [0], [0, 1])
