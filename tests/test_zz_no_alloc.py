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


def test_noalloc_matches_workspace_call_on_two_calls_in_a_row():
    # two different shapes back to back: the second call must not see the first's scratch
    cases = [(8192, 256, 8, 1.1, 1), (4096, 8, 2, 0.0, 2), (8192, 256, 8, 1.1, 3)]
    for T, E, K, skew, seed in cases:
        idx = _routing(T, E, K, skew, seed)
        counts = torch.bincount(idx.view(-1).long(), minlength=E).to(torch.int32)
        ref = moe.moe_permute(idx, E, counts=counts)
        got = moe.moe_permute_noalloc(idx, E, counts=counts)
        torch.cuda.synchronize()
        for k in KEYS:
            assert torch.equal(got[k], ref[k]), f"{k} differs (T={T}, E={E}, K={K})"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    T, E, K = 200000, 8, 8  # 1.6M slots: far beyond the 4 MiB scratch
    idx = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_permute_noalloc(idx, E)
    assert e.value.status == 2  # MOE_ERR_UNSUPPORTED_SHAPE, nothing enqueued
