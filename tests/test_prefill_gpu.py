"""GPU parity of gdn_prefill_packed against the fp64 oracle, through the C ABI.

Workloads follow the serving pages: the 32 x 1,024 chat wave of sparkinfer v0.6.28
(packed passes, one prefix-cache checkpoint per prompt moved back out of the last 16
tokens), ragged prefix-cache hits resuming from stored states, 8K prompts, and the tiny
fp32 pack. Packed-vs-alone identity is the pages' pack_ckpt_check, asserted bitwise.
"""
import numpy as np
import pytest

from oracle import ref
from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

from gpu_util import assert_close, compare_units, run, torch_cuda

pytestmark = pytest.mark.gpu

KERNELS = [gdn.KERNEL_AUTO, gdn.KERNEL_RECURRENT]
# the two schedules of the chunked tensor-core kernel (bf16 io, d = 128 packs)
CHUNKED = [gdn.KERNEL_CHUNKED_PIPELINED, gdn.KERNEL_CHUNKED_THROUGHPUT]


@pytest.fixture(scope="module")
def wave():
    return I.chat_wave()


@pytest.fixture(scope="module")
def ragged():
    return I.ragged_prefix()


@pytest.mark.parametrize("pref", KERNELS)
def test_tiny_f32_all_outputs(pref):
    torch_cuda()
    p = I.tiny_f32()
    o, ck, fin = run(p, pref)
    ro, rck, rfin = ref.prefill(p)
    assert_close(o, ro, "f32", "o")
    assert_close(ck, rck, "f32", "ckpt")
    assert_close(fin, rfin, "f32", "final")
    for j in range(rck.shape[0]):
        assert_close(ck[j], rck[j], "f32", f"ckpt {j}")


@pytest.mark.parametrize("pref", KERNELS)
def test_tiny_dims_bf16(pref):
    torch_cuda()
    lengths = [17, 64, 100, 255]
    p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=64, io_dtype="bf16",
                    seed=1, init_std=0.02, ckpt_lists=I.every_block(lengths, 64))
    got = run(p, pref)
    compare_units(p, got, list(range(4)), list(range(4)))


@pytest.mark.parametrize("pref", KERNELS + CHUNKED)
def test_d64_bf16_on_both_chunked_schedules(pref):
    """d = 64 bf16 heads through the tensor-core kernel (zero-padded to 128) in both
    schedules and through the token-serial kernel: every prompt and head against the
    oracle, edge lengths, initial states, checkpoints on and off the 64-token grid ends."""
    torch_cuda()
    lengths = [1, 0, 2, 63, 64, 65, 129, 200, 330]
    ck = [[q for q in range(64, n + 1, 64)] + ([n] if n % 64 and n > 0 else []) for n in lengths]
    p = I.make_pack(lengths, num_k_heads=4, num_v_heads=8, head_dim=64, io_dtype="bf16",
                    seed=12, init_std=0.02, ckpt_lists=ck)
    got = run(p, pref)
    compare_units(p, got, list(range(len(lengths))), list(range(8)))


def test_d64_bf16_schedules_bitwise_and_pack_vs_alone():
    """d = 64 bf16: the two chunked schedules agree bit for bit, and each prompt's o,
    checkpoints and final state are identical alone and in the pack."""
    torch_cuda()
    lengths = [300, 1, 77, 64, 150]
    ck = [[64, 256], [1], [77], [64], [128, 150]]
    p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=64, io_dtype="bf16",
                    seed=13, init_std=0.02, ckpt_lists=ck)
    a = run(p, gdn.KERNEL_CHUNKED_PIPELINED)
    b = run(p, gdn.KERNEL_CHUNKED_THROUGHPUT)
    c = run(p)
    for x, y, z in zip(a, b, c):
        np.testing.assert_array_equal(x, y)
        np.testing.assert_array_equal(x, z)
    for n in range(len(lengths)):
        s = I.sub_pack(p, [n])
        o1, c1, f1 = run(s)
        np.testing.assert_array_equal(c[0][p.cu_seqlens[n]:p.cu_seqlens[n + 1]], o1)
        np.testing.assert_array_equal(c[1][p.ckpt_cu[n]:p.ckpt_cu[n + 1]], c1)
        np.testing.assert_array_equal(c[2][n], f1[0])


@pytest.mark.parametrize("pref", KERNELS + CHUNKED)
def test_edge_lengths_d128(pref):
    """Empty prompts, single tokens, chunk-1/chunk/chunk+1 tails, checkpoints at ends."""
    torch_cuda()
    lengths = [1, 2, 0, 63, 64, 65, 127, 128, 129, 200, 0, 3]
    ck = [[p for p in range(64, n + 1, 64)] + ([n] if n % 64 and n > 0 else []) for n in lengths]
    p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                    seed=2, init_std=0.02, ckpt_lists=ck)
    got = run(p, pref)
    compare_units(p, got, list(range(len(lengths))), list(range(4)))
    # zero-length prompts: final state is the initial state, bit for bit
    for n in (2, 10):
        np.testing.assert_array_equal(got[2][n], p.init[n].astype(np.float64))


@pytest.mark.parametrize("pref", [gdn.KERNEL_AUTO, gdn.KERNEL_CHUNKED_PIPELINED])
def test_chat_wave_full_size_every_unit(wave, pref):
    """The 32 x 1,024 wave at full size, in the bench's launch configuration (automatic
    choice: the throughput schedule, whose last SM round is partial) and in the pipelined
    schedule: every prompt and value head against the oracle, each checkpoint and final
    state on its own as well as the whole o."""
    torch_cuda()
    got = run(wave, pref)
    compare_units(wave, got, list(range(32)), list(range(32)))


def test_chat_wave_checkpoint_is_at_768(wave):
    assert wave.ckpt_pos.tolist() == [768] * 32


@pytest.mark.parametrize("pref", CHUNKED)
def test_ragged_prefix_full(ragged, pref):
    torch_cuda()
    got = run(ragged, pref)
    compare_units(ragged, got, list(range(ragged.num_seqs)), [0, 1, 14, 15, 30, 31])


@pytest.mark.parametrize("pref", CHUNKED)
def test_ragged_resume_from_checkpoint_equals_uninterrupted(ragged, pref):
    """Prefill to a checkpoint, resume from it: equal to the uninterrupted run (bitwise
    when the cut is on the chunk grid, as every checkpoint here is)."""
    torch = torch_cuda()
    full = run(ragged, pref)
    # pick prompt 0 and its second checkpoint
    n = 0
    j0 = int(ragged.ckpt_cu[n])
    cut = int(ragged.ckpt_pos[j0 + 1])
    s, e = int(ragged.cu_seqlens[n]), int(ragged.cu_seqlens[n + 1])
    rest = I.Pack(name="rest", cu_seqlens=np.array([0, e - s - cut], np.int32),
                  q=ragged.q[s + cut:e], k=ragged.k[s + cut:e], v=ragged.v[s + cut:e],
                  a=ragged.a[s + cut:e], beta=ragged.beta[s + cut:e],
                  init=full[1][j0 + 1][None].astype(np.float32),
                  ckpt_cu=np.zeros(2, np.int32), ckpt_pos=np.zeros(0, np.int32),
                  num_k_heads=ragged.num_k_heads, num_v_heads=ragged.num_v_heads,
                  head_dim=ragged.head_dim, io_dtype="bf16", scale=ragged.scale)
    o2, _, fin2 = run(rest, pref)
    np.testing.assert_array_equal(o2, full[0][s + cut:e])
    np.testing.assert_array_equal(fin2[0], full[2][n])


@pytest.mark.parametrize("pref", CHUNKED)
def test_long_prompts_every_unit(pref):
    """4 x 8,192 tokens (slow decay, checkpoints every 1,024): every prompt and value head
    against the oracle."""
    torch_cuda()
    p = I.long_prompts()
    got = run(p, pref)
    compare_units(p, got, list(range(4)), list(range(32)))


@pytest.mark.parametrize("pref", KERNELS + CHUNKED)
def test_pack_vs_alone_bitwise(pref):
    """Each prompt alone and inside the pack: identical o, checkpoints and final state."""
    torch_cuda()
    lengths = [300, 64, 1, 1024, 0, 129, 700]
    ck = [[q for q in range(64, n + 1, 64)] for n in lengths]
    p = I.make_pack(lengths, num_k_heads=4, num_v_heads=8, head_dim=128, io_dtype="bf16",
                    seed=4, init_std=0.02, ckpt_lists=ck)
    o, c, f = run(p, pref)
    for n in range(p.num_seqs):
        s = I.sub_pack(p, [n])
        o1, c1, f1 = run(s, pref)
        np.testing.assert_array_equal(o[p.cu_seqlens[n]:p.cu_seqlens[n + 1]], o1)
        np.testing.assert_array_equal(c[p.ckpt_cu[n]:p.ckpt_cu[n + 1]], c1)
        np.testing.assert_array_equal(f[n], f1[0])


@pytest.mark.parametrize("pref", KERNELS + CHUNKED)
def test_determinism(pref):
    torch_cuda()
    p = I.make_pack([500, 77, 1024], num_k_heads=4, num_v_heads=8, head_dim=128,
                    io_dtype="bf16", seed=5, init_std=0.02, ckpt_lists=[[256], [], [512]])
    a = run(p, pref)
    b = run(p, pref)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("pref", CHUNKED)
def test_in_place_final_over_initial(pref):
    torch = torch_cuda()
    p = I.make_pack([130, 64], num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                    seed=6, init_std=0.02)
    want = run(p, pref)
    buf = gdn.to_device(p)
    buf.final = buf.init  # final_states aliases initial_state
    run(p, pref, buf=buf)
    np.testing.assert_array_equal(buf.init.cpu().numpy().astype(np.float64), want[2])


@pytest.mark.parametrize("pref", CHUNKED)
def test_guard_bands_untouched(pref):
    """Outputs are written exactly inside their buffers: canaries around each survive."""
    torch = torch_cuda()
    lengths = [65, 1, 130]
    p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                    seed=7, init_std=0.02, ckpt_lists=[[64, 65], [1], [128]])
    buf = gdn.to_device(p)
    G = 4096  # elements of guard on each side

    def guarded(t):
        big = torch.full((t.numel() + 2 * G,), float("nan"), dtype=t.dtype, device=t.device)
        return big, big[G:G + t.numel()].view(t.shape)

    o_big, buf.o = guarded(buf.o)
    c_big, buf.ckpt = guarded(buf.ckpt)
    f_big, buf.final = guarded(buf.final)
    run(p, pref, buf=buf)
    for big in (o_big, c_big, f_big):
        assert torch.isnan(big[:G].float()).all() and torch.isnan(big[-G:].float()).all()
        assert not torch.isnan(big[G:-G].float()).any()


def test_checkpoint_copy_to_pinned_pool(ragged):
    """Checkpoints reach the handle's pinned pool through the side stream."""
    torch = torch_cuda()
    from gpu_util import handle
    import ctypes
    h = handle()
    buf = gdn.to_device(ragged)
    stream = torch.cuda.current_stream()
    gdn.prefill(h, buf, stream)
    nbytes = buf.ckpt.numel() * 4
    offset = 4096
    gdn.gdn_checkpoint_copy(h, buf.ckpt, nbytes, offset, stream)
    gdn.gdn_checkpoint_copy_wait(h)
    assert gdn.gdn_checkpoint_copy_query(h)
    ptr, size = gdn.gdn_pool_info(h)
    assert size >= nbytes + offset
    host = np.ctypeslib.as_array((ctypes.c_float * (nbytes // 4)).from_address(ptr + offset))
    np.testing.assert_array_equal(host.reshape(buf.ckpt.shape), buf.ckpt.cpu().numpy())
    with pytest.raises(gdn.GdnError):
        gdn.gdn_checkpoint_copy(h, buf.ckpt, size, 16, stream)


def _assert_same(a, b):
    for x, y, what in zip(a, b, ("o", "ckpt", "final")):
        np.testing.assert_array_equal(x, y, err_msg=what)


@pytest.mark.parametrize("case", ["edges_init", "raw_gates", "ragged", "long"])
def test_chunked_schedules_agree_bitwise(case, ragged):
    """The pipelined and throughput schedules compute every value the same way (same
    operand roundings, same product accumulation order, the same gate scan), so their
    outputs, checkpoints and final states are bit-identical."""
    torch_cuda()
    if case == "edges_init":
        lengths = [1, 0, 63, 64, 65, 129, 200, 3, 1000]
        ck = [[x for x in range(64, n + 1, 64)] + ([n] if n % 64 and n > 0 else [])
              for n in lengths]
        p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                        seed=31, init_std=0.05, ckpt_lists=ck)
    elif case == "raw_gates":
        base = I.make_pack([300, 77, 128, 5], num_k_heads=2, num_v_heads=4, head_dim=128,
                           io_dtype="bf16", seed=32, init_std=0.02, ckpt_lists=[[128, 300], [], [64], [5]])
        p = I.with_raw_gates(base, seed=5)
    elif case == "ragged":
        p = ragged
    else:
        p = I.make_pack([4096, 333], num_k_heads=4, num_v_heads=8, head_dim=128, io_dtype="bf16",
                        seed=33, init_std=0.02, ckpt_lists=[[2048, 4096], [320]],
                        decay_scale=I.LONG_DECAY_SCALE)
    _assert_same(run(p, gdn.KERNEL_CHUNKED_PIPELINED), run(p, gdn.KERNEL_CHUNKED_THROUGHPUT))


def test_decay_factor_forms_straddle_threshold():
    """The A/P epilogue splits each entry's decay factor into a row and a column factor in
    chunks whose total log2-decay is at least -100 and takes one ex2 per entry in stronger
    chunks. A pack whose chunks fall on both sides of that bound (checked here from the
    gates) matches the oracle under both schedules, which agree bit for bit."""
    torch_cuda()
    lengths = [256, 200, 320, 129]
    p = I.make_pack(lengths, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                    seed=41, init_std=0.02, ckpt_lists=[[128], [], [64, 320], [129]],
                    decay_scale=1.35)
    totals = []
    for n in range(len(lengths)):
        a = p.a[p.cu_seqlens[n]:p.cu_seqlens[n + 1]].astype(np.float64)
        for c0 in range(0, lengths[n], 64):
            totals.extend(a[c0:c0 + 64].sum(axis=0) / np.log(2.0))
    totals = np.array(totals)
    assert (totals >= -100).any() and (totals < -100).any()
    pipe = run(p, gdn.KERNEL_CHUNKED_PIPELINED)
    thr = run(p, gdn.KERNEL_CHUNKED_THROUGHPUT)
    _assert_same(pipe, thr)
    compare_units(p, thr, list(range(len(lengths))), list(range(4)), per_item=False)


def test_automatic_choice_equals_forced_schedules(wave):
    """The automatic result on the wave (throughput schedule) equals either forced
    schedule bit for bit."""
    torch = torch_cuda()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert gdn.gdn_chunked_schedule(wave.cu_seqlens, 32, sms) == gdn.KERNEL_CHUNKED_THROUGHPUT
    auto = run(wave)
    _assert_same(auto, run(wave, gdn.KERNEL_CHUNKED_THROUGHPUT))
    _assert_same(auto, run(wave, gdn.KERNEL_CHUNKED_PIPELINED))


def test_auto_pack_vs_alone_bitwise_across_schedules():
    """A pack for which the automatic choice takes the throughput schedule, against each
    sampled prompt alone (for which it takes the pipelined one): identical o, checkpoints
    and final states."""
    torch = torch_cuda()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_prompts = (6 * sms + 31) // 32
    rng = np.random.default_rng(34)
    lengths = [int(x) for x in rng.integers(1000, 2000, n_prompts)]
    ck = [[q for q in range(64, n + 1, 64)] + ([n] if n % 64 else []) for n in lengths]
    p = I.make_pack(lengths, num_k_heads=16, num_v_heads=32, head_dim=128, io_dtype="bf16",
                    seed=35, init_std=0.02, ckpt_lists=ck)
    assert gdn.gdn_chunked_schedule(p.cu_seqlens, 32, sms) == gdn.KERNEL_CHUNKED_THROUGHPUT
    o, c, f = run(p)
    for n in sorted({0, 1, n_prompts // 2, n_prompts - 1}):
        s = I.sub_pack(p, [n])
        if lengths[n] > 1:  # (a one-token prompt runs the same short-unit code either way)
            assert gdn.gdn_chunked_schedule(s.cu_seqlens, 32, sms) == \
                gdn.KERNEL_CHUNKED_PIPELINED
        o1, c1, f1 = run(s)
        np.testing.assert_array_equal(o[p.cu_seqlens[n]:p.cu_seqlens[n + 1]], o1)
        np.testing.assert_array_equal(c[p.ckpt_cu[n]:p.ckpt_cu[n + 1]], c1)
        np.testing.assert_array_equal(f[n], f1[0])


@pytest.mark.parametrize("pref", KERNELS + CHUNKED)
@pytest.mark.parametrize("hk,hv", [(4, 4), (2, 4), (1, 4), (2, 8)])
def test_gqa_group_sizes(pref, hk, hv):
    """Value head h reads key head h // (H_v / H_k): groups of 1 (4/4), 2 (2/4) and 4 (1/4,
    2/8), every value head of the pack against the oracle (a wrong key-head index fails at
    once)."""
    torch_cuda()
    lengths = [130, 64, 1, 200]
    ck = [[64, 128, 130], [64], [1], [192, 200]]
    p = I.make_pack(lengths, num_k_heads=hk, num_v_heads=hv, head_dim=128, io_dtype="bf16",
                    seed=50 + hk + hv, init_std=0.02, ckpt_lists=ck)
    got = run(p, pref)
    compare_units(p, got, list(range(len(lengths))), list(range(hv)))


def test_many_short_prompts():
    """512 prompts of 0-130 tokens (8,192 units, 8 full waves of SMs): both schedules agree
    bit for bit, the automatic result equals them, and sampled prompts and heads match the
    oracle (the first, the last, empty and one-token prompts among them)."""
    torch_cuda()
    rng = np.random.default_rng(77)
    lengths = [int(x) for x in rng.integers(0, 131, 512)]
    lengths[5], lengths[6], lengths[7] = 0, 1, 64
    ck = [[q for q in range(64, n + 1, 64)] + ([n] if n % 64 and n > 0 else []) for n in lengths]
    p = I.make_pack(lengths, num_k_heads=8, num_v_heads=16, head_dim=128, io_dtype="bf16",
                    seed=78, init_std=0.02, ckpt_lists=ck)
    a = run(p, gdn.KERNEL_CHUNKED_PIPELINED)
    b = run(p, gdn.KERNEL_CHUNKED_THROUGHPUT)
    c = run(p)
    for x, y, z in zip(a, b, c):
        np.testing.assert_array_equal(x, y)
        np.testing.assert_array_equal(x, z)
    compare_units(p, b, [0, 5, 6, 7, 255, 511], [0, 1, 14, 15], per_item=False)
