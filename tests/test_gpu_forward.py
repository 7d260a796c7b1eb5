"""Whole-layer parity on the GPU for every workload, through the C-ABI.

The step-by-step entry points are checked against the oracle at full size:
routing and grouping bit-exact on every workload; H, Z and Y in full on the
tiny, SonicMoE- and Mixtral-shaped layers (the Mixtral shape is the benchmarked
one); on the DeepSeek-V3-shaped layer H and Z on rows of every 128-row tile of
every expert (its first and last row and two more) and Y on at least 1024
tokens chosen so that every tile holds a checked row. moe_forward, in the
configuration the benchmark times, must reproduce the step-by-step result bit
for bit. Y[t] depends only on X[t] and the weights, and H and Z rows only on
their token and expert, so checking a subset against the oracle's definition
on that subset is exact.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import W_ABS, bits, check_hz, check_y, layer_np
from top_routing_grouped_02_gb300 import moe, synth

pytestmark = pytest.mark.gpu

# DeepSeek-V3 shape: rows checked per 128-row tile and the least number of
# tokens whose Y is checked
ROWS_PER_TILE = 4
MIN_TOKENS = 1024


def _steps(inp, K):
    """The layer through the individual entry points; returns every output."""
    T, d = inp["X"].shape
    E, _, n = inp["W1"].shape
    ws = moe.workspace(T, d, E, K, n)
    idx, w, counts = moe.moe_route(inp["X"], inp["Wr"], K, inp["bias"])
    g = moe.moe_permute(idx, E, counts=counts, ws=ws)
    H, Z = moe.moe_expert_mlp(inp["X"], inp["W1"], inp["W3"], inp["W2"], w, g["perm_token"],
                              g["perm_slot"], g["offsets"], K, ws=ws)
    Y = moe.moe_combine(Z, g["row_of_slot"], K)
    st, word = moe.moe_sync_check(ws)
    assert st == 0, (st, word)
    return dict(idx=idx, w=w, counts=counts, H=H, Z=Z, Y=Y, **g)


def _forward(inp, K):
    T, d = inp["X"].shape
    E, _, n = inp["W1"].shape
    ws = moe.workspace(T, d, E, K, n)
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    Y = moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K, inp["bias"],
                        ws=ws, topk_idx=idx, topk_w=w)
    st, word = moe.moe_sync_check(ws)
    assert st == 0, (st, word)
    return Y, idx, w


def _check_grouping(s, idx_r, E):
    off_r, pt_r, ps_r, ros_r = oracle.permute(idx_r, E)
    assert np.array_equal(s["offsets"].cpu().numpy(), off_r)
    assert np.array_equal(s["perm_token"].cpu().numpy(), pt_r)
    assert np.array_equal(s["perm_slot"].cpu().numpy(), ps_r)
    assert np.array_equal(s["row_of_slot"].cpu().numpy(), ros_r)
    assert np.array_equal(s["counts"].cpu().numpy(), oracle.expert_counts(idx_r, E))
    tiles_r = oracle.tile_schedule(off_r, moe.TILE_M)
    assert int(s["num_tiles"].item()) == len(tiles_r)
    assert np.array_equal(s["tiles"].cpu().numpy()[:len(tiles_r)], tiles_r)
    return off_r, pt_r, ps_r, ros_r


def tile_rows(off, per_tile, rng):
    """Sorted grouped rows with, from every 128-row tile of every expert, its
    first and last row and per_tile - 2 more drawn at random."""
    rows = []
    M = moe.TILE_M
    for e in range(len(off) - 1):
        for r0 in range(int(off[e]), int(off[e + 1]), M):
            r1 = min(r0 + M, int(off[e + 1]))
            pick = {r0, r1 - 1}
            inner = np.arange(r0 + 1, r1 - 1)
            if inner.size:
                pick.update(rng.choice(inner, size=min(per_tile - 2, inner.size),
                                       replace=False).tolist())
            rows.extend(pick)
    return np.array(sorted(rows), np.int64)


def oracle_rows(X, W1, W3, W2, w_r, pt, ps, off, P):
    """Oracle H (bf16 bits) and Z (float64) of the grouped rows P (sorted):
    the same definition run on a grouping that holds only those rows."""
    E = len(off) - 1
    e_of = np.searchsorted(off, P, side="right") - 1
    off_sub = np.zeros(E + 1, np.int32)
    off_sub[1:] = np.cumsum(np.bincount(e_of, minlength=E))
    H = oracle.gate_up(X, W1, W3, pt[P], off_sub)
    Z = oracle.down(H, W2, w_r, ps[P], off_sub)
    return H, Z


def _run_workload(name, full_oracle: bool):
    cfg = synth.WORKLOADS[name]
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    inp = synth.layer_inputs(device="cuda", **cfg)
    s = _steps(inp, K)
    Yf, idx_f, w_f = _forward(inp, K)
    torch.cuda.synchronize()
    # moe_forward (the benchmarked call) reproduces the step-by-step result exactly
    assert torch.equal(Yf.view(torch.int16), s["Y"].view(torch.int16))
    assert torch.equal(idx_f, s["idx"]) and torch.equal(w_f, s["w"])

    X, Wr, bias, W1, W3, W2 = layer_np(inp)
    L = oracle.router_logits(X, Wr, bias)
    idx_r, w_r = oracle.topk_softmax(L, K, True)
    assert np.array_equal(s["idx"].cpu().numpy(), idx_r)
    assert float(np.abs(s["w"].cpu().numpy().astype(np.float64) - w_r).max()) <= W_ABS
    off_r, pt_r, ps_r, ros_r = _check_grouping(s, idx_r, E)

    if full_oracle:
        H_ref = oracle.gate_up(X, W1, W3, pt_r, off_r)
        check_hz(bits(s["H"]), H_ref, "H")
        Z_ref = oracle.down(H_ref, W2, w_r, ps_r, off_r)
        check_hz(bits(s["Z"]), Z_ref, "Z")
        Y_ref = oracle.combine(Z_ref, ros_r, K)
        check_y(bits(s["Y"]), Y_ref, "Y")
        return
    rng = np.random.default_rng(12345)
    # H and Z on rows of every tile
    P = tile_rows(off_r, ROWS_PER_TILE, rng)
    H_ref, Z_ref = oracle_rows(X, W1, W3, W2, w_r, pt_r, ps_r, off_r, P)
    Pt = torch.from_numpy(P).cuda()
    check_hz(bits(s["H"][Pt]), H_ref, "H (rows of every tile)")
    check_hz(bits(s["Z"][Pt]), Z_ref, "Z (rows of every tile)")
    # Y on the token of one row of every tile, topped up to MIN_TOKENS tokens
    mid = [int(pt_r[(r0 + min(r0 + moe.TILE_M, int(off_r[e + 1]))) // 2])
           for e in range(E) for r0 in range(int(off_r[e]), int(off_r[e + 1]), moe.TILE_M)]
    toks = set(mid) | {0, T - 1}
    rest = np.setdiff1d(np.arange(T), np.fromiter(toks, np.int64))
    extra = max(0, MIN_TOKENS - len(toks))
    toks.update(rng.choice(rest, size=min(extra, rest.size), replace=False).tolist())
    toks = np.array(sorted(toks), np.int64)
    assert len(toks) >= min(MIN_TOKENS, T)
    covered = np.isin(pt_r, toks)
    for e in range(E):
        for r0 in range(int(off_r[e]), int(off_r[e + 1]), moe.TILE_M):
            assert covered[r0:min(r0 + moe.TILE_M, int(off_r[e + 1]))].any()
    Y_rows, idx_rows, w_rows = oracle.forward_tokens(X, Wr, bias, W1, W3, W2, K, toks)
    assert np.array_equal(idx_rows, idx_r[toks])
    check_y(bits(s["Y"])[toks], Y_rows, "Y (tokens covering every tile)")


def test_tiny_workload():
    _run_workload("tiny", full_oracle=True)


def test_sonic_workload():
    _run_workload("sonic", full_oracle=True)


def test_mixtral_workload():
    # the benchmarked configuration: H, Z and Y of all 8192 rows / 4096 tokens
    _run_workload("mixtral", full_oracle=True)


def test_dsv3_workload():
    _run_workload("dsv3", full_oracle=False)


def test_forward_host_roundtrip_matches_device_call():
    cfg = dict(synth.WORKLOADS["tiny"])
    inp = synth.layer_inputs(device="cuda", **cfg)
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    Y_dev_ref, _, _ = _forward(inp, K)
    Xh = inp["X"].cpu().pin_memory()
    Yh = torch.empty_like(Xh).pin_memory()
    Xd = torch.empty_like(inp["X"])
    Yd = torch.empty_like(inp["X"])
    moe.moe_forward_host(Xh, Yh, Xd, Yd, inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K, inp["bias"])
    assert torch.equal(Yh.view(torch.int16), Y_dev_ref.cpu().view(torch.int16))


def test_forward_host_stream_matches_device_calls():
    # three different batches through the overlapped host path, each against a
    # plain device call on the same batch
    cfg = dict(synth.WORKLOADS["tiny"])
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    inp = synth.layer_inputs(device="cuda", **cfg)
    Xs = torch.stack([synth.normal("X", (T, d), 1.0, torch.bfloat16, "cpu", seed=s)
                      for s in (1, 2, 3)]).pin_memory()
    Ys = torch.empty_like(Xs).pin_memory()
    Xd2 = torch.empty((2, T, d), dtype=torch.bfloat16, device="cuda")
    Yd2 = torch.empty_like(Xd2)
    stream = torch.cuda.Stream()
    moe.moe_forward_host_stream(Xs, Ys, Xd2, Yd2, inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K,
                                inp["bias"], stream=stream)
    for i in range(3):
        one = dict(inp, X=Xs[i].cuda())
        Y_ref, _, _ = _forward(one, K)
        assert torch.equal(Ys[i].view(torch.int16), Y_ref.cpu().view(torch.int16))


def test_forward_host_stream_rejects_shared_streams():
    cfg = dict(synth.WORKLOADS["tiny"])
    T, d, K = cfg["T"], cfg["d"], cfg["K"]
    inp = synth.layer_inputs(device="cuda", **cfg)
    Xs = torch.zeros((1, T, d), dtype=torch.bfloat16).pin_memory()
    Ys = torch.empty_like(Xs).pin_memory()
    Xd2 = torch.empty((2, T, d), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward_host_stream(Xs, Ys, Xd2, torch.empty_like(Xd2), inp["Wr"], inp["W1"],
                                    inp["W3"], inp["W2"], K, stream=s, h2d_stream=s)
    assert e.value.status == 1


def test_forward_traced_records_stage_events():
    cfg = dict(synth.WORKLOADS["tiny"])
    inp = synth.layer_inputs(device="cuda", **cfg)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], cfg["K"], inp["bias"],
                    events=ev)
    torch.cuda.synchronize()
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(5)]
    assert all(t >= 0 for t in times)


def test_forward_rejects_small_workspace():
    cfg = dict(synth.WORKLOADS["tiny"])
    inp = synth.layer_inputs(device="cuda", **cfg)
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], cfg["K"], ws=ws)
    assert e.value.status == 3
