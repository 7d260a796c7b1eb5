"""The allocation-free grouping call (moe_permute_noalloc) against moe_permute.

moe_permute_noalloc serves callers that may not allocate device memory (for
example a plugin inside an inference engine that owns all device memory, or a
serving loop whose memory was planned at start-up): it keeps its scratch in an
array built into libmoe.so instead of a caller workspace. This file runs last
(named so that pytest collects it after the other test files) and passes both
on its own in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

from top_routing_grouped_02_gb300 import moe

pytestmark = pytest.mark.gpu

KEYS = ("offsets", "perm_token", "perm_slot", "row_of_slot", "tiles", "num_tiles")


def _routing(T, E, K, skew, seed):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** (-skew)
    g = rng.gumbel(size=(T, E)) + np.log(p / p.sum())
    return torch.from_numpy(np.argsort(-g, axis=1, kind="stable")[:, :K].astype(np.int32)).cuda()


def _same(got, ref, what):
    """Every output the grouping defines: offsets, the rows in use (up to
    offsets[E]; slots without a row leave the rest unwritten), row_of_slot and
    the tile list."""
    used = int(ref["offsets"][-1].item())
    assert torch.equal(got["offsets"], ref["offsets"]), f"offsets differ ({what})"
    for k in ("perm_token", "perm_slot"):
        assert torch.equal(got[k][:used], ref[k][:used]), f"{k} differs ({what})"
    assert torch.equal(got["row_of_slot"], ref["row_of_slot"]), f"row_of_slot differs ({what})"
    nt = int(ref["num_tiles"].item())
    assert torch.equal(got["num_tiles"], ref["num_tiles"]), f"num_tiles differs ({what})"
    assert torch.equal(got["tiles"][:nt], ref["tiles"][:nt]), f"tiles differ ({what})"


def test_noalloc_matches_workspace_call_on_two_calls_in_a_row():
    # different shapes back to back: a call must not see the previous one's scratch
    cases = [(8192, 256, 8, 1.1, 1), (4096, 8, 2, 0.0, 2), (8192, 256, 8, 1.1, 3)]
    for T, E, K, skew, seed in cases:
        idx = _routing(T, E, K, skew, seed)
        counts = torch.bincount(idx.view(-1).long(), minlength=E).to(torch.int32)
        ref = moe.moe_permute(idx, E, counts=counts)
        got = moe.moe_permute_noalloc(idx, E, counts=counts)
        torch.cuda.synchronize()
        for k in KEYS:
            assert torch.equal(got[k], ref[k]), f"{k} differs (T={T}, E={E}, K={K})"


def test_noalloc_without_counts():
    idx = _routing(3000, 16, 4, 0.7, 4)
    ref = moe.moe_permute(idx, 16)
    got = moe.moe_permute_noalloc(idx, 16)
    torch.cuda.synchronize()
    for k in KEYS:
        assert torch.equal(got[k], ref[k]), f"{k} differs"


def test_noalloc_bad_expert_then_good_call():
    # an index outside [0, E) and a repeated expert get no row (row_of_slot -1),
    # as with moe_permute; the next, valid call must match moe_permute exactly,
    # which shows that the control words the bad call left in the shared array
    # were cleared
    T, E, K = 1000, 8, 2
    idx = _routing(T, E, K, 0.0, 5)
    bad = idx.clone()
    bad[10, 1] = E + 3
    bad[20, 0] = -1
    bad[30, 1] = bad[30, 0]
    ref = moe.moe_permute(bad, E)
    got = moe.moe_permute_noalloc(bad, E)
    torch.cuda.synchronize()
    ros = got["row_of_slot"].cpu().numpy()
    assert ros[10 * K + 1] == -1 and ros[20 * K] == -1 and ros[30 * K + 1] == -1
    _same(got, ref, "bad indices")
    good = _routing(T, E, K, 0.3, 6)
    counts = torch.bincount(good.view(-1).long(), minlength=E).to(torch.int32)
    ref2 = moe.moe_permute(good, E, counts=counts)
    got2 = moe.moe_permute_noalloc(good, E, counts=counts)
    torch.cuda.synchronize()
    for k in KEYS:
        assert torch.equal(got2[k], ref2[k]), f"{k} differs after a bad call"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    T, E, K = 200000, 8, 8  # 1.6M slots: far beyond the 4 MiB scratch
    idx = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_permute_noalloc(idx, E)
    assert e.value.status == 2  # MOE_ERR_UNSUPPORTED_SHAPE, nothing enqueued
