"""The varlen scheduler: cu_seqlens and the checkpoint CSR become a work list that covers
every (prompt, value head, state row) exactly once, longest prompt first."""
import numpy as np
import pytest

from packed_linear_attention_gb300 import build, gdn


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return gdn.load()


def _check_cover(wl, cu, Hv, D):
    N = len(cu) - 1
    seen = np.zeros((N, Hv, D), dtype=np.int32)
    for seq, head, row0, nrows in wl["units"]:
        seen[seq, head, row0:row0 + nrows] += 1
    assert np.all(seen == 1)
    lens = np.diff(cu)
    unit_lens = lens[wl["units"][:, 0]]
    assert np.all(np.diff(unit_lens) <= 0), "units must be ordered longest prompt first"


@pytest.mark.parametrize("dtype,D", [(gdn.GDN_BF16, 128), (gdn.GDN_F32, 64), (gdn.GDN_BF16, 64)])
def test_cover_and_order(dtype, D):
    rng = np.random.default_rng(1)
    lens = [0, 1, 17, 64, 2048, 100, 64, 0, 255]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ck = [[p for p in range(64, n + 1, 64)] for n in lens]
    ckpt_cu = np.concatenate([[0], np.cumsum([len(c) for c in ck])]).astype(np.int32)
    ckpt_pos = np.array([p for c in ck for p in c], np.int32)
    cfg = gdn.make_config(2, 6, D, io_dtype=dtype)
    wl = gdn.gdn_prefill_worklist_host(None, cfg, cu, ckpt_cu, ckpt_pos)
    _check_cover(wl, cu, 6, D)
    assert wl["status"] == 0
    np.testing.assert_array_equal(wl["seqs"][:, 0], cu[:-1])
    np.testing.assert_array_equal(wl["seqs"][:, 1], lens)
    np.testing.assert_array_equal(wl["seqs"][:, 2], ckpt_cu[:-1])
    np.testing.assert_array_equal(wl["seqs"][:, 3], ckpt_cu[1:])
    np.testing.assert_array_equal(wl["ckpt_pos"], ckpt_pos)
    size = gdn.gdn_prefill_workspace_size(cfg, cu, ckpt_cu)
    assert wl["nbytes"] <= size


def test_stable_order_for_equal_lengths():
    cu = np.arange(0, 33 * 1024, 1024, dtype=np.int32)
    cfg = gdn.make_config(16, 32, 128)
    wl = gdn.gdn_prefill_worklist_host(None, cfg, cu)
    seqs = wl["units"][:, 0]
    assert np.all(np.diff(seqs) >= 0)  # equal lengths keep pack order


def test_recurrent_preference_changes_row_blocks():
    # no GPU: a NULL handle means automatic choice; the token-serial family splits rows
    cfg = gdn.make_config(2, 4, 64, io_dtype=gdn.GDN_F32)
    wl = gdn.gdn_prefill_worklist_host(None, cfg, np.array([0, 10, 30], np.int32))
    assert set(wl["units"][:, 3].tolist()) == {32}
    _check_cover(wl, np.array([0, 10, 30]), 4, 64)
