"""The C ABI on the host: the library loads, exports every symbol the header declares,
and rejects malformed calls before anything is launched (no GPU needed: validation comes
before any CUDA call, and a NULL handle with well-formed arguments is itself an error)."""
import ctypes
import os
import re

import numpy as np
import pytest

from packed_linear_attention_gb300 import build, gdn
from packed_linear_attention_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gdn.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(gdn.EXPORTS)


def test_version_and_status_strings(lib):
    assert gdn.gdn_abi_version() == 1
    assert gdn.status_string(0) == "ok"
    assert gdn.status_string(3) == "workspace too small"
    assert gdn.status_string(99) == "unknown status"


@pytest.mark.parametrize("length,expect", [(1024, 768), (1000, 768), (1030, 768),
                                           (1040, 1024), (1039, 768), (270, 0), (0, 0)])
def test_ckpt_position_rule(lib, length, expect):
    assert gdn.gdn_ckpt_position(length, 256, 16) == expect
    if length > 0:
        assert I.ckpt_position_with_move_back(length, 256, 16) == expect


def test_mixed_budget(lib):
    assert gdn.gdn_mixed_budget([300, 500, 400, 100], 1024, 8) == (3, [300, 500, 224, 0])
    assert gdn.gdn_mixed_budget([100] * 10, 1024, 8) == (8, [100] * 8 + [0, 0])
    rng = np.random.default_rng(0)
    for _ in range(50):
        rem = rng.integers(1, 400, size=int(rng.integers(1, 12))).tolist()
        served, take = gdn.gdn_mixed_budget(rem, 1024, 8)
        assert take == I.mixed_budget(rem, 1024, 8)
        assert sum(take) <= 1024 and served == sum(t > 0 for t in take)


CFG = dict(num_k_heads=16, num_v_heads=32, head_dim=128)


def _call(cfg=None, cu=(0, 100, 300), ckpt_cu=None, ckpt_pos=None, ptr=1 << 20, ws=1 << 20,
          ws_bytes=None, handle=None, final=True, o=True):
    cfg = cfg or gdn.make_config(**CFG)
    if ws_bytes is None:
        ws_bytes = 1 << 20
    step = 1 << 28  # distinct, non-overlapping fake device ranges
    P = lambda i: ptr + i * step
    return gdn.gdn_prefill_packed(handle, cfg, list(cu), P(1), P(2), P(3), P(4), P(5), None,
                                  ckpt_cu, ckpt_pos, P(6) if o else None, P(7),
                                  P(8) if final else None, ws, ws_bytes, None,
                                  raise_on_error=False)


def test_prefill_validation(lib):
    E = gdn
    assert _call() == E.GDN_ERR_INVALID_ARGUMENT                        # NULL handle
    assert _call(cu=(1, 100)) == E.GDN_ERR_INVALID_ARGUMENT              # cu[0] != 0
    assert _call(cu=(0, 100, 50)) == E.GDN_ERR_INVALID_ARGUMENT          # decreasing
    assert _call(cu=(0,)) == E.GDN_ERR_INVALID_ARGUMENT                  # no prompt
    bad = gdn.make_config(**CFG)
    bad.num_v_heads = 24
    bad.num_k_heads = 16
    assert _call(cfg=bad, ws_bytes=1 << 20) == E.GDN_ERR_INVALID_ARGUMENT  # Hv % Hk
    bad = gdn.make_config(16, 32, 96)
    assert _call(cfg=bad, ws_bytes=1 << 20) == E.GDN_ERR_UNSUPPORTED     # head dim
    bad = gdn.make_config(16, 32, 128, chunk_size=32)
    assert _call(cfg=bad, ws_bytes=1 << 20) == E.GDN_ERR_UNSUPPORTED     # chunk size
    bad = gdn.make_config(16, 32, 128)
    bad.io_dtype = 7
    assert _call(cfg=bad, ws_bytes=1 << 20) == E.GDN_ERR_INVALID_ARGUMENT
    # checkpoints: out of range, not increasing, off the chunk grid
    assert _call(ckpt_cu=[0, 1, 1], ckpt_pos=[101]) == E.GDN_ERR_INVALID_ARGUMENT
    assert _call(ckpt_cu=[0, 2, 2], ckpt_pos=[64, 64]) == E.GDN_ERR_INVALID_ARGUMENT
    assert _call(ckpt_cu=[0, 1, 1], ckpt_pos=[50]) == E.GDN_ERR_UNSUPPORTED
    # well-formed checkpoints (one at a prompt's end, one on the grid): only the NULL
    # handle is left to complain about
    assert _call(ckpt_cu=[0, 1, 2], ckpt_pos=[100, 128]) == E.GDN_ERR_INVALID_ARGUMENT
    # workspace
    assert _call(ws_bytes=255) == E.GDN_ERR_WORKSPACE_TOO_SMALL
    assert _call(ws=(1 << 20) + 16) == E.GDN_ERR_INVALID_ARGUMENT          # misaligned
    # missing outputs, misaligned input
    assert _call(final=False) == E.GDN_ERR_INVALID_ARGUMENT
    assert _call(o=False) == E.GDN_ERR_INVALID_ARGUMENT
    assert _call(ptr=(1 << 20) + 8) == E.GDN_ERR_INVALID_ARGUMENT


def test_prefill_rejects_overlapping_outputs(lib):
    cfg = gdn.make_config(**CFG)
    cu = [0, 64]
    ws = gdn.gdn_prefill_workspace_size(cfg, cu)
    base = 1 << 30
    # o overlaps q
    st = gdn.gdn_prefill_packed(None, cfg, cu, base, base + (1 << 24), base + (2 << 24),
                                base + (3 << 24), base + (4 << 24), None, None, None,
                                base + 4096, None, base + (5 << 24), base + (6 << 24), ws,
                                None, raise_on_error=False)
    assert st == gdn.GDN_ERR_INVALID_ARGUMENT


def test_decode_validation(lib):
    cfg = gdn.make_config(**CFG)
    P = lambda i: (1 << 20) * (i + 1)
    args = [P(1), P(2), P(3), P(4), P(5), P(6), 4, P(7), P(8)]
    assert gdn.gdn_decode_step(None, cfg, 2, *args, raise_on_error=False) == \
        gdn.GDN_ERR_INVALID_ARGUMENT                                       # NULL handle
    assert gdn.gdn_decode_step(None, cfg, -1, *args, raise_on_error=False) == \
        gdn.GDN_ERR_INVALID_ARGUMENT
    bad = gdn.make_config(16, 32, 80)
    assert gdn.gdn_decode_step(None, bad, 2, *args, raise_on_error=False) == \
        gdn.GDN_ERR_UNSUPPORTED
    args[0] = P(1) + 4
    assert gdn.gdn_decode_step(None, cfg, 2, *args, raise_on_error=False) == \
        gdn.GDN_ERR_INVALID_ARGUMENT


def test_workspace_size_is_aligned_and_monotone(lib):
    cfg = gdn.make_config(**CFG)
    a = gdn.gdn_prefill_workspace_size(cfg, [0, 10])
    b = gdn.gdn_prefill_workspace_size(cfg, [0, 10, 20, 30], [0, 0, 0, 1])
    assert a % 256 == 0 and b % 256 == 0 and 256 <= a <= b


def test_checkpoint_copy_bounds_without_pool(lib):
    # NULL handle is an argument error; no CUDA call is made
    assert lib.gdn_checkpoint_copy(None, ctypes.c_void_p(16), 16, 0, None) == \
        gdn.GDN_ERR_INVALID_ARGUMENT


def test_gate_mode_validation(lib):
    cu = [0, 100, 300]
    ok = gdn.make_config(**CFG)
    assert gdn.gdn_prefill_workspace_size(ok, cu) > 0
    raw = gdn.make_config(**CFG)
    raw.gate_mode = gdn.GDN_GATES_RAW                     # raw gates without A_log, dt_bias
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill_workspace_size(raw, cu)
    assert e.value.status == gdn.GDN_ERR_INVALID_ARGUMENT
    raw.a_log, raw.dt_bias = 1 << 20, 2 << 20             # both given: accepted
    assert gdn.gdn_prefill_workspace_size(raw, cu) > 0
    raw.dt_bias = None
    with pytest.raises(gdn.GdnError):
        gdn.gdn_prefill_workspace_size(raw, cu)
    bad = gdn.make_config(**CFG)
    bad.gate_mode = 2
    with pytest.raises(gdn.GdnError):
        gdn.gdn_prefill_workspace_size(bad, cu)


def test_host_workspace_size(lib):
    """gdn_prefill_packed_host's workspace holds one work list per prompt group: at least
    the whole pack's, growing with the number of groups; bad group sizes are rejected."""
    cfg = gdn.make_config(**CFG)
    cu = list(range(0, 33 * 1024, 1024))
    whole = gdn.gdn_prefill_workspace_size(cfg, cu)
    sizes = [gdn.gdn_prefill_host_workspace_size(cfg, cu, group_prompts=g) for g in (32, 8, 1)]
    assert all(x % 256 == 0 for x in sizes)
    assert sizes[0] >= whole and sizes[0] <= sizes[1] <= sizes[2]
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill_host_workspace_size(cfg, cu, group_prompts=0)
    assert e.value.status == gdn.GDN_ERR_INVALID_ARGUMENT
    with pytest.raises(gdn.GdnError) as e:  # more than 64 groups
        gdn.gdn_prefill_host_workspace_size(cfg, list(range(0, 66 * 8, 8)), group_prompts=1)
    assert e.value.status == gdn.GDN_ERR_UNSUPPORTED


def _estimates(W, L, U, S, sms):
    """(pipelined, throughput) estimates in microseconds, as gdn_chunked_schedule states them:
    W chunks over U units, the longest L chunks, S one-token units."""
    import math
    has = 1.0 if U else 0.0
    mean = W / U if U else 0.0
    t_pipe = max(5.12 * L + 15.7 * has, (5.12 * W + 15.7 * U + 8.0 * S) / sms,
                 math.ceil(U / sms) * (5.12 * mean + 15.7))
    chain = 8.93 * L + 13.2 if U > sms else 6.38 * L + 17.3 * has
    full, last = divmod(U, 2 * sms)
    paired, alone = 8.93 * mean + 13.2, 6.38 * mean + 17.3
    rounds = full * paired + (paired if last > sms else alone if last else 0.0)
    t_thr = max(chain, rounds, (8.93 * W + 13.2 * U + 16.6 * S) / (2 * sms))
    return t_pipe, t_thr


def test_chunked_schedule_choice(lib):
    """The automatic choice between the chunked kernel's schedules against the cost model
    written out here, on the packs whose times were measured: pipelined for one unit per
    SM, for the ragged prefix-cache pack and for 8K prompts; throughput for two or more
    units per SM of 1,024-token prompts and for the 32 x 1,024 wave."""
    pipe, thr = gdn.KERNEL_CHUNKED_PIPELINED, gdn.KERNEL_CHUNKED_THROUGHPUT
    choose = gdn.gdn_chunked_schedule
    cu = lambda lens: np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    assert choose(cu([1024] * 19), 8, 152) == pipe      # 152 units: one per SM
    assert choose(cu([1024] * 38), 8, 152) == thr       # 304 units
    assert choose(cu([1024] * 76), 8, 152) == thr       # 608 units
    assert choose(cu([1024] * 32), 32, 152) == thr      # the wave
    assert choose(cu([4096] * 19), 8, 152) == pipe      # 152 long units
    assert choose(cu([128] * 38), 8, 152) == thr        # 304 short units
    assert choose(I.mixed_step().prefill.cu_seqlens, 32, 152) == thr
    r = I.ragged_prefix()
    assert choose(r.cu_seqlens, 32, 152) == pipe
    assert choose(cu([8192] * 4), 32, 152) == pipe
    assert choose(cu([]), 32, 152) == pipe              # empty pack
    rng = np.random.default_rng(3)
    for _ in range(200):
        lens = rng.integers(0, 5000, rng.integers(1, 40))
        lens[rng.random(len(lens)) < 0.2] = rng.integers(0, 2)  # empty and one-token prompts
        hv, sms = int(rng.choice([4, 8, 32, 64])), int(rng.choice([1, 132, 152]))
        ch = np.where(lens > 1, (lens + 63) // 64, 0)  # prompts of <= 1 token: short units
        W, L = float(ch.sum() * hv), float(ch.max())
        S, U = float((lens <= 1).sum() * hv), float((lens > 1).sum() * hv)
        t_pipe, t_thr = _estimates(W, L, U, S, sms)
        assert choose(cu(lens), hv, sms) == (thr if t_thr < t_pipe else pipe)
    for bad in ((cu([3]), 0, 152), (cu([3]), 8, 0), (np.array([1, 4], np.int32), 8, 152),
                (np.array([0, 4, 2], np.int32), 8, 152)):
        with pytest.raises(gdn.GdnError) as e:
            choose(*bad)
        assert e.value.status == gdn.GDN_ERR_INVALID_ARGUMENT


def _model_us(lens, hv, sms):
    """The chunked cost model of gdn_chunked_schedule, written out: microseconds."""
    lens = np.asarray(lens, np.int64)
    ch = np.where(lens > 1, (lens + 63) // 64, 0)
    W, L = float(ch.sum() * hv), float(ch.max()) if len(ch) else 0.0
    S, U = float((lens <= 1).sum() * hv), float((lens > 1).sum() * hv)
    return min(_estimates(W, L, U, S, sms))


def _split_choice(lens, hv, sms):
    best, best_seg = _model_us(lens, hv, sms), 0
    longest = max(lens)
    for parts in range(2, 17):
        seg = -(-longest // parts)
        seg = -(-seg // 64) * 64
        if seg < 64 or seg >= longest:
            continue
        a, a_hv, b = [], [], []
        for n in lens:
            a.append((min(n, seg), hv))
            if n <= seg:
                continue
            np_ = -(-n // seg)
            a += [(seg, 2 * hv)] * (np_ - 2)
            b += [(min(seg, n - q * seg), hv) for q in range(1, np_)]

        def us(items):
            if not items:
                return 0.0
            lens_ = np.array([x for x, _ in items])
            w = np.array([u for _, u in items], np.float64)
            ch = np.where(lens_ > 1, (lens_ + 63) // 64, 0)
            W, L, S = float((ch * w).sum()), float(ch.max()), float(((lens_ <= 1) * w).sum())
            U = float(((lens_ > 1) * w).sum())
            return min(_estimates(W, L, U, S, sms))
        t = us(a) + us(b) + 12.0
        if t < best:
            best, best_seg = t, seg
    return best_seg


def test_split_segment_choice(lib):
    """The automatic segment length for sequence splitting against the cost model written
    out here: no split for the wave or 4 x 8K (the SMs are full) nor for the ragged
    prefix-cache pack (pass 1 alone would hold more work than the unsplit chain), a split
    for one 32K prompt (its chain alone bounds it)."""
    cu = lambda lens: np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    auto = gdn.gdn_split_segment_auto
    assert auto(cu([1024] * 32), 32, 152) == 0
    assert auto(cu([8192] * 4), 32, 152) == 0
    one = auto(cu([32768]), 32, 152)
    assert one == 3328  # 10 segments (measured on GB300: 1.47 ms, against 1.48 for 5 and 2.52 whole)
    r = I.ragged_prefix()
    assert auto(r.cu_seqlens, 32, 152) == 0
    rng = np.random.default_rng(5)
    for _ in range(100):
        lens = [int(x) for x in rng.integers(0, 20000, rng.integers(1, 12))]
        hv, sms = int(rng.choice([4, 8, 32])), int(rng.choice([132, 152]))
        assert auto(cu(lens), hv, sms) == _split_choice(lens, hv, sms), (lens, hv, sms)
    with pytest.raises(gdn.GdnError):
        auto(cu([5]), 0, 152)


def test_test_hook_validation(lib):
    for hook in (0, 1):
        with pytest.raises(gdn.GdnError) as e:
            gdn.gdn_set_test_hook(None, hook)  # no handle
        assert e.value.status == gdn.GDN_ERR_INVALID_ARGUMENT
