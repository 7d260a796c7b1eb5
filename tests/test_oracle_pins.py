"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not compute itself: values
worked out by hand from the pages' definitions (tests/golden/), library routines
(numpy stable sort, bincount, cumsum, scipy softmax, torch float64 matmul and
bf16 conversion), closed forms and invariants. Together they are chosen so that
a plausible slip anywhere in the oracle (a dropped term, a wrong sign or index,
a swapped operand, a wrong summation order, an unstable sort) fails one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from top_routing_grouped_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(a):
    return oracle.bf16_bits_to_f64(a)


def torch_bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_of_f64_via_torch(a: np.ndarray) -> np.ndarray:
    # float64 -> bf16 by torch (may round twice through fp32; compared within 1 ulp)
    t = torch.from_numpy(np.ascontiguousarray(a, np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 steps between two arrays of bf16 bits (same-sign finite)."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return np.abs(key(a) - key(b))


# ----------------------------------------------------------------- bf16 --

@pytest.mark.parametrize("value,bits", [
    (1.0 + 2.0**-8, 0x3F80),            # halfway, ties to even (down)
    (1.0 + 3 * 2.0**-8, 0x3F82),        # halfway, ties to even (up)
    (1.0 + 2.0**-8 + 2.0**-30, 0x3F81), # just above halfway
    (-(1.0 + 2.0**-8), 0xBF80),
    ((2 - 2.0**-7) * 2.0**127, 0x7F7F), # largest finite
    ((2 - 2.0**-8) * 2.0**127, 0x7F80), # halfway to 2^128 -> even -> overflow
    (2.0**-133, 0x0001),                # smallest subnormal
    (2.0**-134, 0x0000),                # halfway to zero, ties to even
    (1.5 * 2.0**-134, 0x0001),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (3.0, 0x4040),
])
def test_bf16_rounding_hand_cases(oracle_lib, value, bits):
    assert oracle.bf16_from_double(value) == bits


def test_bf16_rounding_matches_torch_on_fp32_values(oracle_lib):
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = raw.view(np.float32)
    f = f[np.isfinite(f)]
    ours = np.array([oracle.bf16_from_double(float(v)) for v in f[:20000]], np.uint16)
    assert np.array_equal(ours, torch_bf16_bits_from_f32(f[:20000]))


def test_bf16_to_double_roundtrip(oracle_lib):
    for b in (0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4040, 0x8000):
        assert oracle.bf16_from_double(oracle.bf16_to_double(b)) == b


# --------------------------------------------------------------- logits --

def _read_logit_cases():
    cases = []
    for line in open(os.path.join(GOLDEN, "logits_cases.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        xs, ws, b, exp = [p.strip() for p in line.split("|")]
        cases.append((_hex_list(xs), _hex_list(ws), None if b == "-" else float.fromhex(b),
                       float.fromhex(exp)))
    return cases


def _hex_list(text):
    # hex floats; "a*n" stands for n copies of a
    out = []
    for tok in text.split():
        v, _, n = tok.partition("*")
        out.extend([float.fromhex(v)] * (int(n) if n else 1))
    return out


@pytest.mark.parametrize("case", _read_logit_cases())
def test_logits_golden_order_and_fusion(oracle_lib, case):
    xs, ws, b, exp = case
    X = torch_bf16_bits_from_f32(np.array([xs], np.float32))
    assert np.array_equal(f64(X)[0], np.array(xs))  # fixture x values are bf16-exact
    Wr = np.array(ws, np.float32).reshape(-1, 1)
    bias = None if b is None else np.array([b], np.float32)
    L = oracle.router_logits(X, Wr, bias)
    assert L[0, 0] == np.float32(exp), (L[0, 0].hex() if hasattr(L[0, 0], "hex") else L[0, 0])


def test_logits_blocks_only_with_few_experts(oracle_lib):
    # the block case of the golden file (a 2^24 weight in block 0, two 1-weights
    # in block 1, x = 1): blocks give 2^24 + 2, one chain over all j gives 2^24.
    # With E <= 32 every column is blocked, with E = 33 none is.
    d = 2048
    w = np.zeros(d, np.float32)
    w[0], w[1024], w[1025] = 2.0 ** 24, 1.0, 1.0
    X = torch_bf16_bits_from_f32(np.ones((1, d), np.float32))
    for E, expect in ((32, 2.0 ** 24 + 2), (33, 2.0 ** 24)):
        L = oracle.router_logits(X, np.ascontiguousarray(np.repeat(w[:, None], E, axis=1)))
        assert np.all(L == np.float32(expect)), (E, L[0, :3])


def test_logits_exact_integer_dot(oracle_lib):
    # small integers: every partial sum is exact in fp32, so L equals the exact dot
    rng = np.random.default_rng(2)
    T, d, E = 7, 96, 5
    xi = rng.integers(-8, 9, size=(T, d))
    wi = rng.integers(-64, 65, size=(d, E))
    bias = rng.integers(-3, 4, size=E).astype(np.float32)
    L = oracle.router_logits(torch_bf16_bits_from_f32(xi.astype(np.float32)),
                             wi.astype(np.float32), bias)
    assert np.array_equal(L, (xi @ wi + bias).astype(np.float32))


def test_logits_close_to_float64_dot_and_column_permutation(oracle_lib):
    inp = synth.layer_inputs(T=16, d=512, E=12, n=8)
    X = synth.bf16_bits(inp["X"])
    Wr = inp["Wr"].numpy()
    L = oracle.router_logits(X, Wr)
    ref = f64(X) @ Wr.astype(np.float64)
    assert np.max(np.abs(L - ref)) < 1e-5
    perm = np.random.default_rng(3).permutation(12)
    assert np.array_equal(oracle.router_logits(X, np.ascontiguousarray(Wr[:, perm]))[:, :], L[:, perm])


# ----------------------------------------------------------- top-k/softmax --

def _read_router_cases():
    cases = []
    for line in open(os.path.join(GOLDEN, "router_cases.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, lg, idx, w = [p.strip() for p in line.split("|")]
        E, K, renorm = (int(v) for v in head.split())
        cases.append((E, K, renorm, [float(v) for v in lg.split()], [int(v) for v in idx.split()],
                      [float(v) for v in w.split()]))
    return cases


@pytest.mark.parametrize("case", _read_router_cases())
def test_route_golden(oracle_lib, case):
    E, K, renorm, lg, idx, w = case
    L = np.array([lg], np.float32)
    got_idx, got_w = oracle.topk_softmax(L, K, bool(renorm))
    assert got_idx[0].tolist() == idx
    assert np.max(np.abs(got_w[0].astype(np.float64) - np.array(w))) <= 1e-7


def _rank_select(L, K):
    # independent selection: rank_e = #{strictly larger} + #{equal with lower index}
    T, E = L.shape
    out = np.empty((T, K), np.int64)
    for t in range(T):
        row = L[t]
        ranks = [(row > row[e]).sum() + (row[:e] == row[e]).sum() for e in range(E)]
        for e, r in enumerate(ranks):
            if r < K:
                out[t, r] = e
    return out


@pytest.mark.parametrize("E,K", [(8, 2), (16, 4), (64, 8), (5, 5), (7, 1)])
def test_topk_matches_rank_count_and_stable_sort(oracle_lib, E, K):
    rng = np.random.default_rng(E * 10 + K)
    T = 64
    L = rng.standard_normal((T, E)).astype(np.float32)
    L[::3] = rng.integers(-2, 3, size=(len(L[::3]), E)).astype(np.float32)  # many exact ties
    L[1] = 0.0
    idx, w = oracle.topk_softmax(L, K)
    assert np.array_equal(idx, _rank_select(L, K))
    assert np.array_equal(idx, np.argsort(-L, axis=1, kind="stable")[:, :K])
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 1e-6)
    assert np.all(w > 0) and np.all(np.diff(w, axis=1) <= 0)


def test_softmax_values_against_scipy(oracle_lib):
    from scipy.special import softmax
    rng = np.random.default_rng(5)
    L = (rng.standard_normal((32, 8)) * 3).astype(np.float32)
    p = softmax(L.astype(np.float64), axis=1)
    idx, w = oracle.topk_softmax(L, 8, renorm=True)          # K = E: full softmax
    assert np.max(np.abs(w - np.take_along_axis(p, idx, 1))) <= 1e-7
    idx2, w2 = oracle.topk_softmax(L, 2, renorm=False)       # raw top-K probabilities
    assert np.max(np.abs(w2 - np.take_along_axis(p, idx2, 1))) <= 1e-7
    idx3, w3 = oracle.topk_softmax(L, 2, renorm=True)        # renormalised
    pk = np.take_along_axis(p, idx3, 1)
    assert np.max(np.abs(w3 - pk / pk.sum(1, keepdims=True))) <= 1e-7


def test_zero_input_and_k1_and_extremes(oracle_lib):
    X = np.zeros((4, 64), np.uint16)
    Wr = np.random.default_rng(6).standard_normal((64, 8)).astype(np.float32)
    L = oracle.router_logits(X, Wr)
    assert np.all(L == 0)
    idx, w = oracle.topk_softmax(L, 3)
    assert np.array_equal(idx, np.tile([0, 1, 2], (4, 1)))
    assert np.all(w == np.float32(1 / 3))
    idx1, w1 = oracle.topk_softmax(Wr[:4] * 10, 1)
    assert np.all(w1 == 1.0)
    big = np.array([[80, -80, 79.5, -80, 0, 0, 0, 0]], np.float32)
    idx, w = oracle.topk_softmax(big, 2, renorm=False)
    assert np.all(np.isfinite(w)) and idx[0].tolist() == [0, 2]


# ------------------------------------------------------ counts / permute --

def _read_permute_case():
    vals = {}
    for line in open(os.path.join(GOLDEN, "permute_case.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, *v = line.split()
        vals[k] = [int(x) for x in v]
    return vals


def test_permute_golden(oracle_lib):
    g = _read_permute_case()
    T, K, E, M = g["T"][0], g["K"][0], g["E"][0], g["M"][0]
    idx = np.array(g["idx"], np.int32).reshape(T, K)
    assert oracle.expert_counts(idx, E).tolist() == g["counts"]
    offsets, pt, ps, ros = oracle.permute(idx, E)
    assert offsets.tolist() == g["offsets"]
    assert pt.tolist() == g["perm_token"]
    assert ps.tolist() == g["perm_slot"]
    assert ros.tolist() == g["row_of_slot"]
    assert oracle.tile_schedule(offsets, M).ravel().tolist() == g["tiles"]


@pytest.mark.parametrize("T,E,K,skew", [(300, 8, 2, False), (257, 64, 8, True), (1, 4, 4, False),
                                        (33, 256, 8, True)])
def test_permute_against_library_sort(oracle_lib, T, E, K, skew):
    rng = np.random.default_rng(T + E)
    p = np.arange(1, E + 1, dtype=np.float64) ** (-3.0 if skew else 0.0)
    idx = np.stack([rng.choice(E, size=K, replace=False, p=p / p.sum()) for _ in range(T)]).astype(np.int32)
    counts = oracle.expert_counts(idx, E)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert counts.sum() == T * K
    offsets, pt, ps, ros = oracle.permute(idx, E)
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    order = np.argsort(idx.ravel(), kind="stable")
    assert np.array_equal(ps, order)
    assert np.array_equal(pt, order // K)
    assert np.array_equal(ros[ps], np.arange(T * K))
    for e in range(E):
        rows = pt[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(rows) > 0)
    for M in (1, 3, 128):
        tiles = oracle.tile_schedule(offsets, M)
        assert len(tiles) == sum(-(-int(c) // M) for c in counts)
        cover = np.zeros(T * K, np.int64)
        for e, r0, nr, _ in tiles:
            assert 1 <= nr <= M and offsets[e] <= r0 and r0 + nr <= offsets[e + 1]
            cover[r0:r0 + nr] += 1
        assert np.all(cover == 1)


# ------------------------------------------------------------ expert MLP --

def _dense_swiglu_torch(x, W1, W3, W2):
    """Dense SwiGLU MLP in float64 with torch: h rounded to bf16, y in float64."""
    x = torch.from_numpy(f64(x))
    a1 = x @ torch.from_numpy(f64(W1))
    a3 = x @ torch.from_numpy(f64(W3))
    h = (torch.nn.functional.silu(a1) * a3)
    hb = h.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    return h, hb, hb @ torch.from_numpy(f64(W2))


def _small_layer(T, d, E, n, seed=0, zipf=False):
    inp = synth.layer_inputs(T=T, d=d, E=E, n=n, zipf=zipf, seed=seed)
    return (synth.bf16_bits(inp["X"]), inp["Wr"].numpy(),
            None if inp["bias"] is None else inp["bias"].numpy(),
            synth.bf16_bits(inp["W1"]), synth.bf16_bits(inp["W3"]), synth.bf16_bits(inp["W2"]))


def test_single_expert_equals_dense_swiglu(oracle_lib):
    # K = E = 1: the layer is one dense SwiGLU MLP with weight 1
    X, Wr, _, W1, W3, W2 = _small_layer(T=40, d=64, E=1, n=96, seed=11)
    out = oracle.forward(X, Wr, None, W1, W3, W2, K=1)
    assert np.all(out["w"] == 1.0) and np.all(out["idx"] == 0)
    h, hb, y = _dense_swiglu_torch(X, W1[0], W3[0], W2[0])
    H = out["H"][out["row_of_slot"]]  # back to token order (identity here)
    assert np.array_equal(out["perm_token"], np.arange(40))
    assert np.mean(H == bf16_bits_of_f64_via_torch(h.numpy())) > 0.999
    assert ulp_diff(H, bf16_bits_of_f64_via_torch(h.numpy())).max() <= 1
    assert np.max(np.abs(out["Z"] - y.numpy())) < 1e-12
    assert ulp_diff(out["Y"], bf16_bits_of_f64_via_torch(y.numpy())).max() <= 1


def test_pre_activations_are_the_grouped_rows_times_w1_and_w3(oracle_lib):
    # A1 = x W1[e], A3 = x W3[e] of each grouped row, against torch float64
    # matmuls of the gathered rows expert by expert; and SiLU(A1) * A3 rounded
    # to bf16 gives the oracle's H
    X, Wr, _, W1, W3, W2 = _small_layer(T=50, d=64, E=4, n=48, seed=21)
    out = oracle.forward(X, Wr, None, W1, W3, W2, K=2)
    A1, A3 = oracle.gate_up_pre(X, W1, W3, out["perm_token"], out["offsets"])
    off = out["offsets"]
    xs = torch.from_numpy(f64(X))
    for e in range(4):
        rows = xs[torch.from_numpy(out["perm_token"][off[e]:off[e + 1]].astype(np.int64))]
        r1 = (rows @ torch.from_numpy(f64(W1[e]))).numpy()
        r3 = (rows @ torch.from_numpy(f64(W3[e]))).numpy()
        assert np.max(np.abs(A1[off[e]:off[e + 1]] - r1)) < 1e-12
        assert np.max(np.abs(A3[off[e]:off[e + 1]] - r3)) < 1e-12
    h = torch.nn.functional.silu(torch.from_numpy(A1)) * torch.from_numpy(A3)
    assert ulp_diff(out["H"], bf16_bits_of_f64_via_torch(h.numpy())).max() <= 1


def test_silu_gate_is_w1_not_w3(oracle_lib):
    X, Wr, _, W1, W3, W2 = _small_layer(T=8, d=64, E=1, n=64, seed=12)
    a = oracle.forward(X, Wr, None, W1, W3, W2, K=1)["Y"]
    b = oracle.forward(X, Wr, None, W3, W1, W2, K=1)["Y"]
    _, _, y = _dense_swiglu_torch(X, W1[0], W3[0], W2[0])
    assert ulp_diff(a, bf16_bits_of_f64_via_torch(y.numpy())).max() <= 1
    assert not np.array_equal(a, b)


def test_identical_experts_give_single_mlp(oracle_lib):
    X, Wr, _, W1, W3, W2 = _small_layer(T=24, d=64, E=6, n=32, seed=13)
    W1 = np.repeat(W1[:1], 6, 0)
    W3 = np.repeat(W3[:1], 6, 0)
    W2 = np.repeat(W2[:1], 6, 0)
    out = oracle.forward(X, Wr, None, W1, W3, W2, K=3)
    _, _, y = _dense_swiglu_torch(X, W1[0], W3[0], W2[0])
    # sum_k w_k = 1 up to fp32 rounding of each weight
    assert np.max(np.abs(f64(out["Y"]) - y.numpy())) <= 2 ** -7 * np.abs(y.numpy()).max()
    assert ulp_diff(out["Y"], bf16_bits_of_f64_via_torch(y.numpy())).max() <= 1


def test_zero_up_projection_gives_zero(oracle_lib):
    X, Wr, _, W1, W3, W2 = _small_layer(T=16, d=64, E=4, n=32, seed=14)
    out = oracle.forward(X, Wr, None, W1, np.zeros_like(W3), W2, K=2)
    assert np.all((out["Y"] & 0x7FFF) == 0)


def test_one_hot_routing_picks_that_expert(oracle_lib):
    X, Wr, _, W1, W3, W2 = _small_layer(T=20, d=64, E=4, n=32, seed=15)
    out = oracle.forward(X, Wr, None, W1, W3, W2, K=1)
    for t in range(20):
        e = out["idx"][t, 0]
        _, _, y = _dense_swiglu_torch(X[t:t + 1], W1[e], W3[e], W2[e])
        assert ulp_diff(out["Y"][t:t + 1], bf16_bits_of_f64_via_torch(y.numpy())).max() <= 1


def test_grouped_path_equals_token_by_token_definition(oracle_lib):
    X, Wr, bias, W1, W3, W2 = _small_layer(T=48, d=128, E=16, n=64, seed=16, zipf=True)
    out = oracle.forward(X, Wr, bias, W1, W3, W2, K=4)
    toks = np.arange(48)
    Y, idx, w = oracle.forward_tokens(X, Wr, bias, W1, W3, W2, K=4, tokens=toks)
    assert np.array_equal(idx, out["idx"])
    assert np.array_equal(w, out["w"])
    assert np.array_equal(Y, out["Y"])


def test_combine_matches_library_gather_sum(oracle_lib):
    rng = np.random.default_rng(17)
    T, K, d = 9, 3, 40
    Zb = torch.randn(T * K, d).to(torch.bfloat16)
    ros = rng.permutation(T * K).astype(np.int32)
    Y = oracle.combine_bf16(Zb.view(torch.int16).numpy().view(np.uint16), ros, K)
    ref = Zb.double()[torch.from_numpy(ros.astype(np.int64))].view(T, K, d).sum(1)
    assert ulp_diff(Y, bf16_bits_of_f64_via_torch(ref.numpy())).max() <= 1
    Yd = oracle.combine(Zb.double().numpy(), ros, K)
    assert np.array_equal(Yd, Y)


def test_bias_enters_selection(oracle_lib):
    X, Wr, _, W1, W3, W2 = _small_layer(T=32, d=64, E=8, n=32, seed=18)
    bias = np.zeros(8, np.float32)
    bias[5] = 100.0
    L = oracle.router_logits(X, Wr, bias)
    idx, _ = oracle.topk_softmax(L, 2)
    assert np.all(idx[:, 0] == 5)
