"""The mixed step in one launch with the states in a pool (sparkinfer v0.6.4 release notes,
"What changed": prompt slices under a 1,024-token budget in the same pass as the decoding
requests; vllm.cpp "vLLM, online serving", lever 2b, packed GDN decode): prompt slices and
one-token decode rows run as one pack through gdn_prefill_packed_pool, every prompt reading
its initial state from its pool slot (or starting from zeros) and writing its final state
back in place. Checked against the fp64 oracle, bit for bit against gdn_prefill_packed on
the same pack with dense initial / final arrays, and between the two chunked schedules;
slots the pack does not name stay bitwise untouched."""
import numpy as np
import pytest

from oracle import ref
from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import assert_close, handle, run, torch_cuda

pytestmark = pytest.mark.gpu


def _pool_call(pack, pool_np, slots, start_zero, pref):
    torch = torch_cuda()
    h = handle()
    buf = gdn.to_device(pack)
    pool = torch.from_numpy(pool_np.copy()).cuda()
    gdn.gdn_set_kernel_preference(h, pref)
    try:
        gdn.gdn_prefill_packed_pool(h, buf.cfg, buf.cu, buf.q, buf.k, buf.v, buf.a, buf.beta,
                                    pool, pool_np.shape[0], slots, start_zero, buf.ckpt_cu,
                                    buf.ckpt_pos if len(buf.ckpt_pos) else None, buf.o,
                                    buf.ckpt if buf.ckpt.numel() else None, buf.workspace,
                                    buf.workspace_bytes)
        launches = gdn.gdn_prefill_launch_count(h)
        torch.cuda.synchronize()
        assert gdn.gdn_read_device_status(buf.workspace) == 0
    finally:
        gdn.gdn_set_kernel_preference(h, gdn.KERNEL_AUTO)
    return (buf.o.float().cpu().numpy().astype(np.float64),
            buf.ckpt.cpu().numpy().astype(np.float64), pool.cpu().numpy(), launches)


@pytest.mark.parametrize("pref", [gdn.KERNEL_AUTO, gdn.KERNEL_CHUNKED_PIPELINED,
                                  gdn.KERNEL_CHUNKED_THROUGHPUT])
def test_mixed_step_one_launch_from_pool(pref):
    ms = I.mixed_step()
    both = I.mixed_one_pack(ms)
    N = both.num_seqs
    npre = ms.prefill.num_seqs
    rng = np.random.default_rng(11)
    S = N + 9
    slots = rng.permutation(S)[:N].astype(np.int32)
    pool_np = (0.02 * rng.standard_normal((S, 32, 128, 128))).astype(np.float32)
    pool_np[slots[npre:]] = ms.dec_states               # decoding sequences resume
    start_zero = np.array([1] * npre + [0] * (N - npre), np.int32)  # new prompts: zeros
    o, _, pool, launches = _pool_call(both, pool_np, slots, start_zero, pref)
    assert launches == 1
    ro, _, rfin = ref.prefill(both)
    assert_close(o, ro, "bf16", "mixed o")
    assert_close(pool[slots].astype(np.float64), rfin, "bf16", "mixed pool states")
    untouched = np.setdiff1d(np.arange(S), slots)
    np.testing.assert_array_equal(pool[untouched], pool_np[untouched])
    # the same pack through gdn_prefill_packed with dense initial / final arrays: same bits
    do, _, dfin = run(both, pref)
    np.testing.assert_array_equal(o, do)
    np.testing.assert_array_equal(pool[slots].astype(np.float64), dfin)


def test_pool_prefill_with_checkpoints_and_in_place_resume():
    """Prompts of several lengths (empty and one-token ones among them) with checkpoints,
    resumed from their slots: pool path == dense path bit for bit, and a second call that
    resumes every prompt from the state the first one left in its slot matches the oracle
    run over both calls' tokens."""
    lengths = [130, 1, 0, 64, 200]
    p1 = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                     seed=90, init_std=0.02, ckpt_lists=[[64, 130], [1], [], [64], [192]])
    S = 9
    slots = np.array([7, 2, 5, 0, 3], np.int32)
    pool_np = np.zeros((S, 4, 128, 128), np.float32)
    pool_np[slots] = p1.init
    marker = np.float32(123.0)
    for sl in np.setdiff1d(np.arange(S), slots):
        pool_np[sl] = marker
    o, ck, pool, launches = _pool_call(p1, pool_np, slots, None, gdn.KERNEL_AUTO)
    assert launches == 1
    do, dck, dfin = run(p1)
    np.testing.assert_array_equal(o, do)
    np.testing.assert_array_equal(ck, dck)
    np.testing.assert_array_equal(pool[slots].astype(np.float64), dfin)
    assert np.all(pool[np.setdiff1d(np.arange(S), slots)] == marker)
    # second call: new tokens for every prompt, states resumed in place from the pool
    p2 = I.make_pack([70, 1, 3, 0, 64], num_k_heads=2, num_v_heads=4, head_dim=128,
                     io_dtype="bf16", seed=91, ckpt_lists=[[64], [], [], [], [64]])
    o2, _, pool2, _ = _pool_call(p2, pool, slots, None, gdn.KERNEL_AUTO)
    p2.init = pool[slots]
    ro2, _, rfin2 = ref.prefill(p2)
    assert_close(o2, ro2, "bf16", "resumed o")
    assert_close(pool2[slots].astype(np.float64), rfin2, "bf16", "resumed states")


def test_pool_validation():
    """Slots out of range or named twice are rejected before anything is enqueued."""
    torch = torch_cuda()
    p = I.make_pack([5, 3], num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16", seed=92)
    buf = gdn.to_device(p)
    pool = torch.zeros((3, 4, 128, 128), dtype=torch.float32, device="cuda")
    for bad in ([0, 3], [1, 1], [-1, 0]):
        st = gdn.gdn_prefill_packed_pool(handle(), buf.cfg, buf.cu, buf.q, buf.k, buf.v, buf.a,
                                         buf.beta, pool, 3, bad, None, None, None, buf.o, None,
                                         buf.workspace, buf.workspace_bytes,
                                         raise_on_error=False)
        assert st == gdn.GDN_ERR_INVALID_ARGUMENT, bad
