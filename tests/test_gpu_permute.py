"""Grouping parity on the GPU: offsets, permutation, inverse map and tile list
bit-exact against the oracle; device-side checks of bad input."""
import numpy as np
import pytest
import torch

import oracle
from top_routing_grouped_02_gb300 import moe

pytestmark = pytest.mark.gpu


def _routing(T, E, K, skew=0.0, seed=0):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** (-skew)
    p /= p.sum()
    # K distinct experts per token, drawn without replacement (Gumbel top-K)
    g = rng.gumbel(size=(T, E)) + np.log(p)
    return np.argsort(-g, axis=1, kind="stable")[:, :K].astype(np.int32)


def _check(idx: np.ndarray, E: int):
    T, K = idx.shape
    counts = oracle.expert_counts(idx, E)
    off_r, pt_r, ps_r, ros_r = oracle.permute(idx, E)
    tiles_r = oracle.tile_schedule(off_r, moe.TILE_M)
    d_idx = torch.from_numpy(idx).cuda()
    out = moe.moe_permute(d_idx, E, counts=torch.from_numpy(counts).cuda())
    ws_status = None
    torch.cuda.synchronize()
    assert np.array_equal(out["offsets"].cpu().numpy(), off_r)
    assert np.array_equal(out["perm_token"].cpu().numpy(), pt_r)
    assert np.array_equal(out["perm_slot"].cpu().numpy(), ps_r)
    assert np.array_equal(out["row_of_slot"].cpu().numpy(), ros_r)
    nt = int(out["num_tiles"].item())
    assert nt == len(tiles_r)
    assert np.array_equal(out["tiles"].cpu().numpy()[:nt], tiles_r)
    return ws_status


@pytest.mark.parametrize("T,E,K,skew", [
    (512, 8, 2, 0.0),       # tiny
    (4096, 8, 2, 0.0),      # Mixtral-shaped
    (8192, 256, 8, 1.1),    # DeepSeek-V3-shaped, Zipf-skewed loads
    (16384, 128, 4, 0.0),   # SonicMoE-shaped
    (1, 4, 4, 0.0),         # one token, every expert
    (33, 256, 8, 3.0),      # most experts empty
    (1000, 5, 1, 0.5),
    (20000, 64, 4, 0.5),    # one kernel, 10 chunks a block: warps take two chunks each
    (65536, 32, 2, 0.0),    # one kernel at its limit: 64 blocks of 32 chunks
    (65537, 32, 2, 0.0),    # one token more: the three kernels
    (70000, 16, 2, 0.0),    # many chunks (> 2048)
])
def test_permute_matches_oracle(T, E, K, skew):
    _check(_routing(T, E, K, skew, seed=T + E), E)


def test_permute_one_expert_takes_everything_and_exact_tile_multiples():
    T, E, K = 1024, 8, 1
    _check(np.full((T, K), 3, np.int32), E)            # 1024 rows = 8 full tiles
    idx = np.zeros((256, 2), np.int32)
    idx[:, 0] = 2
    idx[:, 1] = 5                                        # two experts, 256 rows each
    _check(idx, E)


def test_permute_flags_bad_expert_and_count_mismatch():
    T, E, K = 64, 8, 2
    idx = _routing(T, E, K, seed=3)
    counts = oracle.expert_counts(idx, E)
    bad = idx.copy()
    bad[5, 1] = 11                                       # out of range
    ws = moe.workspace(T, 0, E, K, 0)
    out = moe.moe_permute(torch.from_numpy(bad).cuda(), E, counts=torch.from_numpy(counts).cuda(),
                          ws=ws)
    status, word = moe.moe_sync_check(ws)
    assert status == 7 and (word & 0x2) and (word & 0x4)
    ros = out["row_of_slot"].cpu().numpy()
    assert ros[5 * K + 1] == -1
    good = np.delete(np.arange(T * K), 5 * K + 1)
    assert np.all(ros[good] >= 0)
    assert int(out["offsets"][-1]) == T * K - 1
    status, word = moe.moe_sync_check(ws)                # cleared by the previous read
    assert status == 0 and word == 0


def test_permute_skips_and_flags_a_repeated_expert():
    # Each top-K row names K distinct experts. A row that repeats an expert
    # would give both slots one rank (one bit per token and expert), so the
    # repeat is skipped (row_of_slot -1) and flagged. The rest must equal the
    # oracle's grouping with the repeated slot sent to an extra last expert,
    # which takes no row before offsets[E].
    T, E, K = 200, 8, 3
    idx = _routing(T, E, K, seed=11)
    idx[7] = [3, 3, 5]                                   # slot 7*K+1 repeats expert 3
    idx[40] = [6, 1, 6]                                  # slot 40*K+2 repeats expert 6
    rep = [7 * K + 1, 40 * K + 2]
    ws = moe.workspace(T, 0, E, K, 0)
    out = moe.moe_permute(torch.from_numpy(idx).cuda(), E, ws=ws)
    status, word = moe.moe_sync_check(ws)
    assert status == 7 and (word & 0x8) and not (word & 0x2), word
    ref_idx = idx.copy().reshape(-1)
    ref_idx[rep] = E
    off_r, pt_r, ps_r, ros_r = oracle.permute(ref_idx.reshape(T, K), E + 1)
    used = int(off_r[E])
    assert used == T * K - len(rep)
    assert np.array_equal(out["offsets"].cpu().numpy(), off_r[:E + 1])
    assert np.array_equal(out["perm_token"].cpu().numpy()[:used], pt_r[:used])
    assert np.array_equal(out["perm_slot"].cpu().numpy()[:used], ps_r[:used])
    ros = out["row_of_slot"].cpu().numpy()
    assert np.all(ros[rep] == -1)
    keep = np.setdiff1d(np.arange(T * K), rep)
    assert np.array_equal(ros[keep], ros_r[keep])
    tiles_r = oracle.tile_schedule(off_r[:E + 1], moe.TILE_M)
    nt = int(out["num_tiles"].item())
    assert nt == len(tiles_r)
    assert np.array_equal(out["tiles"].cpu().numpy()[:nt], tiles_r)
