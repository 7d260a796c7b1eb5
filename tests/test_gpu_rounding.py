"""Token Rounding parity on the GPU (through the C-ABI) against the oracle.

The rounded counts, offsets, perm_token, row_map and tile list are compared bit
for bit; row weights within 1e-6; combine and whole-layer outputs within the Y
tolerances. Logits are seeded synthetic inputs made on the host, so the GPU's
top-K choice (itself checked bit-exact against the oracle) feeds the rounding
kernel and the oracle rounds its own top-K choice.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import W_ABS, bits, check_y, layer_np
from top_routing_grouped_02_gb300 import moe, synth

pytestmark = pytest.mark.gpu


def _logits(T, E, seed, ties=False, skew=0.0):
    L = synth.normal("L", (T, E), 1.0, seed=seed)
    if ties:
        # integer grid: many exactly equal scores within an expert's column
        L = torch.round(L * 2.0)
    if skew:
        L = L - skew * torch.log(torch.arange(1, E + 1, dtype=torch.float32))
    return L.float().contiguous()


def _round_both(L, K, M, renorm):
    T, E = L.shape
    idx_r, _ = oracle.topk_softmax(L.numpy(), K, renorm)
    ref = oracle.token_rounding(L.numpy(), idx_r, M, renorm)
    Ld = L.cuda()
    idx, _, counts = moe.moe_route_logits(Ld, K, renorm)
    got = moe.moe_round_routing(Ld, idx, counts, M, renorm)
    st, word = moe.moe_sync_check(got["ws"])
    assert st == 0, (st, word)
    assert np.array_equal(idx.cpu().numpy(), idx_r)
    return ref, got


def _check_rounding(ref, got):
    R = int(ref["offsets"][-1])
    assert np.array_equal(got["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(got["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(got["perm_token"].cpu().numpy()[:R], ref["perm_token"])
    assert np.array_equal(got["row_map"].cpu().numpy(), ref["row_map"])
    w = got["row_w"].cpu().numpy()[:R].astype(np.float64)
    assert float(np.abs(w - ref["row_w"]).max(initial=0.0)) <= W_ABS
    tiles_r = oracle.tile_schedule(ref["offsets"], moe.TILE_M)
    assert int(got["num_tiles"].item()) == len(tiles_r)
    assert np.array_equal(got["tiles"].cpu().numpy()[:len(tiles_r)], tiles_r)


@pytest.mark.parametrize("T,E,K,M", [(512, 8, 2, 128), (16384, 128, 4, 128), (8192, 256, 8, 128),
                                     (3000, 16, 2, 64), (777, 32, 3, 7), (2048, 64, 6, 1)])
@pytest.mark.parametrize("renorm", [True, False])
def test_rounding_matches_oracle(T, E, K, M, renorm):
    ref, got = _round_both(_logits(T, E, seed=T + E), K, M, renorm)
    _check_rounding(ref, got)


@pytest.mark.parametrize("T,E,K,M", [(1000, 8, 2, 32), (4000, 64, 4, 128), (333, 5, 2, 16)])
def test_rounding_exact_ties(T, E, K, M):
    # many equal logits: the second sort's tie rule (lower token first) decides
    ref, got = _round_both(_logits(T, E, seed=7, ties=True), K, M, True)
    _check_rounding(ref, got)


def test_rounding_skewed_load_and_column_scratch():
    # T above the on-chip column size: the per-expert columns go through the
    # workspace scratch; Zipf-like skew makes some experts round to zero
    T, E, K, M = 40000, 16, 2, 128
    ref, got = _round_both(_logits(T, E, seed=3, skew=1.1), K, M, True)
    assert int(moe.lib().moe_round_workspace_bytes(T, E)) > 256
    _check_rounding(ref, got)


@pytest.mark.parametrize("T,E,K,M", [(1, 4, 1, 128), (3, 2, 1, 4), (100, 8, 2, 128),
                                     (130, 2, 2, 128), (64, 256, 8, 2)])
def test_rounding_edge_cases(T, E, K, M):
    # T < M (experts round to 0 or are capped at T), K == E, E = 256
    ref, got = _round_both(_logits(T, E, seed=11), K, M, True)
    _check_rounding(ref, got)


def test_rounding_half_tile_rounds_up():
    # expert 0 is chosen by M/2 tokens and expert 1 by 3M/2: both counts lie
    # halfway between multiples of M and both round up (expert 1 to T itself)
    T, E, M = 256, 2, 128
    L = torch.zeros(T, E)
    L[:64, 0] = 1.0
    L[64:, 1] = 1.0
    L[:, 0] += torch.linspace(0, 0.5, T)
    ref, got = _round_both(L.float().contiguous(), 1, M, True)
    assert ref["counts"].tolist() == [128, 256]
    _check_rounding(ref, got)


def test_rounding_flags_counts_that_disagree_with_idx():
    T, E, K, M = 512, 8, 2, 128
    Ld = _logits(T, E, seed=5).cuda()
    idx, _, counts = moe.moe_route_logits(Ld, K, True)
    bad = counts.clone()
    bad[0] += 1
    bad[1] -= 1
    got = moe.moe_round_routing(Ld, idx, bad, M, True)
    st, word = moe.moe_sync_check(got["ws"])
    assert st == 7 and (word & 0x4)
    # no row was written outside the capacity, and the stream is still usable
    cap = moe.moe_round_capacity(T, E, K, M)
    rm = got["row_map"].cpu().numpy()
    assert rm.max() < cap
    torch.cuda.synchronize()


@pytest.mark.parametrize("T,E,d", [(512, 8, 256), (1000, 64, 1536), (3, 256, 8)])
def test_combine_rows_matches_oracle(T, E, d):
    rng = np.random.default_rng(T + E)
    kept = rng.random((T, E)) < min(1.0, 6.0 / E)
    kept[0] = False  # a token no expert kept
    R = int(kept.sum())
    rm = np.full((T, E), -1, np.int32)
    rm[kept] = rng.permutation(R).astype(np.int32)
    Zb = synth.normal("Z", (max(R, 1), d), 0.5, torch.bfloat16, "cuda")
    Y_ref = oracle.combine_rows_bf16(bits(Zb)[:R], rm)
    Y = moe.moe_combine_rows(Zb, torch.from_numpy(rm).cuda())
    torch.cuda.synchronize()
    got = bits(Y)
    diff = np.abs(got.astype(np.int32) - Y_ref.astype(np.int32))
    assert np.mean(diff == 0) > 0.999
    assert np.all(got[0] == 0)
    check_y(got, Y_ref, "Y")


def _forward_rounded(inp, K):
    T, d = inp["X"].shape
    E, _, n = inp["W1"].shape
    ws = moe.workspace_rounded(T, d, E, K, n)
    rm = torch.empty((T, E), dtype=torch.int32, device="cuda")
    Y = moe.moe_forward_rounded(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K,
                                inp["bias"], ws=ws, row_map=rm)
    st, word = moe.moe_sync_check(ws)
    assert st == 0, (st, word)
    return Y, rm


@pytest.mark.parametrize("cfg", [dict(T=512, d=256, E=8, K=2, n=512, zipf=False),
                                 dict(T=1500, d=512, E=16, K=4, n=256, zipf=True),
                                 dict(T=2048, d=256, E=4, K=1, n=384, zipf=False)])
@pytest.mark.parametrize("pair", ["0", "1"])
def test_forward_rounded_matches_oracle(cfg, pair, monkeypatch):
    monkeypatch.setenv("MOE_GEMM_CTA_PAIR", pair)
    inp = synth.layer_inputs(device="cuda", **cfg)
    Y, rm = _forward_rounded(inp, cfg["K"])
    torch.cuda.synchronize()
    X, Wr, bias, W1, W3, W2 = layer_np(inp)
    ref = oracle.forward_rounded(X, Wr, bias, W1, W3, W2, cfg["K"])
    assert np.array_equal(rm.cpu().numpy(), ref["row_map"])
    assert np.all(ref["counts"] % moe.TILE_M == 0)
    check_y(bits(Y), ref["Y"], "Y")


def _many_experts_inputs(device):
    # router coordinate 0 adds 2*X[t,0] to every logit of token t; token 0 has
    # X[0,0] = 8, so it outranks every other token for every expert, while its
    # MLP input stays ordinary
    cfg = dict(T=4096, d=256, E=64, K=2, n=256, zipf=False)
    inp = synth.layer_inputs(device=device, **cfg)
    inp["Wr"][0, :] = 2.0
    inp["X"][0, 0] = 8.0
    return cfg, inp


def test_forward_rounded_token_with_many_experts():
    # every expert that rounds up adds token 0: it ends with more rows than the
    # compact per-token list holds, and the combine reads its row_map entries
    cfg, inp = _many_experts_inputs("cuda")
    Y, rm = _forward_rounded(inp, cfg["K"])
    torch.cuda.synchronize()
    X, Wr, bias, W1, W3, W2 = layer_np(inp)
    ref = oracle.forward_rounded(X, Wr, bias, W1, W3, W2, cfg["K"])
    assert (ref["row_map"][0] >= 0).sum() > 16
    assert np.array_equal(rm.cpu().numpy(), ref["row_map"])
    check_y(bits(Y), ref["Y"], "Y")


def test_forward_rounded_sonic_shape_sampled():
    # the SonicMoE-shaped layer (T=16384 d=1536 E=128 K=4 n=256) at full size:
    # routing in full, Y on sampled tokens from the token-by-token definition
    cfg = synth.WORKLOADS["sonic"]
    K = cfg["K"]
    inp = synth.layer_inputs(device="cuda", **cfg)
    Y, rm = _forward_rounded(inp, K)
    torch.cuda.synchronize()
    X, Wr, bias, W1, W3, W2 = layer_np(inp)
    L = oracle.router_logits(X, Wr, bias)
    idx_r, _ = oracle.topk_softmax(L, K, True)
    ref = oracle.token_rounding(L, idx_r, moe.TILE_M, True)
    assert np.array_equal(rm.cpu().numpy(), ref["row_map"])
    rng = np.random.default_rng(99)
    toks = np.sort(rng.choice(cfg["T"], size=48, replace=False))
    Y_rows = oracle.forward_assigned(X, W1, W3, W2, ref["row_map"], ref["row_w"], toks)
    check_y(bits(Y)[toks], Y_rows, "Y (sampled tokens)")


def test_forward_rounded_traced_events():
    cfg = dict(synth.WORKLOADS["tiny"])
    inp = synth.layer_inputs(device="cuda", **cfg)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    moe.moe_forward_rounded(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], cfg["K"],
                            inp["bias"], events=ev)
    torch.cuda.synchronize()
    assert all(ev[i].elapsed_time(ev[i + 1]) >= 0 for i in range(5))
