"""GPU parity of gdn_decode_step and of a whole mixed step (prompt slices under a
1,024-token budget, oldest first, beside 32 decoding sequences; sparkinfer v0.6.4,
"What changed") against the fp64 oracle."""
import numpy as np
import pytest

from oracle import ref
from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import assert_close, handle, run, torch_cuda

pytestmark = pytest.mark.gpu


def _bf16_dev(x, torch):
    return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)


def _decode_gpu(ms, slots, pool_np, torch):
    cfg = gdn.make_config(16, 32, 128)
    B = ms.dec_q.shape[0]
    pool = torch.from_numpy(pool_np.copy()).cuda()
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    slot_t = torch.from_numpy(np.asarray(slots, np.int32)).cuda()
    gdn.gdn_decode_step(handle(), cfg, B, _bf16_dev(ms.dec_q, torch), _bf16_dev(ms.dec_k, torch),
                        _bf16_dev(ms.dec_v, torch), torch.from_numpy(ms.dec_a).cuda(),
                        torch.from_numpy(ms.dec_beta).cuda(), pool, pool_np.shape[0], slot_t, o)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), pool.cpu().numpy().astype(np.float64)


def test_decode_step_vs_oracle():
    torch = torch_cuda()
    ms = I.mixed_step()
    B = ms.dec_q.shape[0]
    rng = np.random.default_rng(3)
    S = B + 7
    pool_np = np.zeros((S, 32, 128, 128), np.float32)
    slots = rng.permutation(S)[:B].astype(np.int32)
    pool_np[slots] = ms.dec_states
    o, pool = _decode_gpu(ms, slots, pool_np, torch)
    f = I.bf16_bits_to_f32
    ro, rpool = ref.decode(f(ms.dec_q), f(ms.dec_k), f(ms.dec_v), ms.dec_a, ms.dec_beta,
                           pool_np, slots, scale=128 ** -0.5)
    assert_close(o, ro, "bf16", "decode o")
    assert_close(pool[slots], rpool[slots], "bf16", "decode states")
    untouched = np.setdiff1d(np.arange(S), slots)
    np.testing.assert_array_equal(pool[untouched], pool_np[untouched].astype(np.float64))


def test_mixed_step_prefill_plus_decode():
    """Config of a mixed step: prompt slices through gdn_prefill_packed, decode tokens
    both through gdn_decode_step and as one-token segments of the same pack."""
    torch = torch_cuda()
    ms = I.mixed_step()
    assert sum(ms.take) <= 1024 and len([t for t in ms.take if t]) <= 8
    pre = ms.prefill
    # prompt slices
    got = run(pre)
    ro, _, rfin = ref.prefill(pre)
    assert_close(got[0], ro, "bf16", "mixed prefill o")
    assert_close(got[2], rfin, "bf16", "mixed prefill states")
    # decode tokens as one-token segments with initial states, appended to the pack
    B = ms.dec_q.shape[0]
    lengths = list(pre.lengths) + [1] * B
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    init = np.concatenate([np.zeros((pre.num_seqs, 32, 128, 128), np.float32), ms.dec_states])
    rep = lambda x: x  # noqa: E731
    both = I.Pack(name="mixed_one_pack", cu_seqlens=cu,
                  q=np.concatenate([pre.q, ms.dec_q]), k=np.concatenate([pre.k, ms.dec_k]),
                  v=np.concatenate([pre.v, ms.dec_v]), a=np.concatenate([pre.a, ms.dec_a]),
                  beta=np.concatenate([pre.beta, ms.dec_beta]), init=rep(init),
                  ckpt_cu=np.zeros(len(lengths) + 1, np.int32), ckpt_pos=np.zeros(0, np.int32),
                  num_k_heads=16, num_v_heads=32, head_dim=128, io_dtype="bf16",
                  scale=128 ** -0.5)
    o1, _, f1 = run(both)
    ro1, _, rf1 = ref.prefill(both)
    assert_close(o1, ro1, "bf16", "one-pack o")
    assert_close(f1, rf1, "bf16", "one-pack states")
    # the decode kernel agrees with the one-pack path on the decode rows
    od, pool = _decode_gpu(ms, np.arange(B), ms.dec_states.copy(), torch)
    assert_close(od, ro1[pre.total_tokens:], "bf16", "decode vs oracle")
    assert_close(pool, rf1[pre.num_seqs:], "bf16", "decode states vs oracle")


def test_decode_steps_replay_from_a_cuda_graph():
    """Decode steps captured once in a CUDA graph and replayed: the call does its checks on
    the host and enqueues one kernel, so the graph holds the whole step. Three replays
    after the capture give the same o and states, bit for bit, as three direct calls."""
    torch = torch_cuda()
    ms = I.mixed_step()
    cfg = gdn.make_config(16, 32, 128)
    B = ms.dec_q.shape[0]
    rng = np.random.default_rng(5)
    S = B + 3
    pool0 = np.zeros((S, 32, 128, 128), np.float32)
    slots = rng.permutation(S)[:B].astype(np.int32)
    pool0[slots] = ms.dec_states
    q, k, v = (_bf16_dev(x, torch) for x in (ms.dec_q, ms.dec_k, ms.dec_v))
    a, b = torch.from_numpy(ms.dec_a).cuda(), torch.from_numpy(ms.dec_beta).cuda()
    slot_t = torch.from_numpy(slots).cuda()

    def steps(pool, o, n, stream=None):
        for _ in range(n):
            gdn.gdn_decode_step(handle(), cfg, B, q, k, v, a, b, pool, S, slot_t, o, stream)

    direct_pool = torch.from_numpy(pool0.copy()).cuda()
    direct_o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    steps(direct_pool, direct_o, 3)
    torch.cuda.synchronize()

    graph_pool = torch.from_numpy(pool0.copy()).cuda()
    graph_o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):  # the capture runs no step; replays do
        with torch.cuda.graph(g, stream=side):
            steps(graph_pool, graph_o, 1, side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(graph_o, direct_o)
    assert torch.equal(graph_pool, direct_pool)
