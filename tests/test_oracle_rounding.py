"""Pins of the Token Rounding oracle to facts outside itself (CPU only).

Token Rounding ("混合专家模型(MoE)架构优化与SonicMoE实践" §3) rounds each expert's
top-K row count to a multiple of the tile size M and picks, by a second sort,
which tokens the expert drops or gains. The oracle is checked against:
hand-worked cases with closed-form weights (tests/golden/token_rounding_cases.txt);
the special case M = 1, where nothing is rounded and the result must be the plain
grouping of the already pinned top-K routing; order invariants that hold at any
size (every kept token outranks every passed-over one); numpy/scipy softmax for
the weights; and the token-by-token layer definition for the grouped path.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from top_routing_grouped_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_cases():
    cases, cur = {}, None
    for line in open(os.path.join(GOLDEN, "token_rounding_cases.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = cases.setdefault(rest.strip(), {})
        elif key in ("w1", "w0"):
            cur[key] = [s.strip() for s in rest.split(";") if s.strip()]
        else:
            cur[key] = [float(v) if key == "L" else int(v) for v in rest.split()]
    return cases


CASES = _read_cases()


def _closed_form(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"exp": math.exp}))


@pytest.mark.parametrize("name", sorted(CASES))
def test_rounding_golden(oracle_lib, name):
    g = CASES[name]
    T, E, K, M = g["T"][0], g["E"][0], g["K"][0], g["M"][0]
    L = np.array(g["L"], np.float32).reshape(T, E)
    idx, _ = oracle.topk_softmax(L, K)
    for renorm, key in ((True, "w1"), (False, "w0")):
        tr = oracle.token_rounding(L, idx, M, renorm)
        assert tr["counts"].tolist() == g["counts"]
        assert tr["offsets"].tolist() == g["offsets"]
        assert tr["perm_token"].tolist() == g.get("perm_token", [])
        assert tr["row_map"].ravel().tolist() == g["row_map"]
        want = np.array([_closed_form(x) for x in g[key]], np.float64)
        assert tr["row_w"].shape == want.shape
        assert np.max(np.abs(tr["row_w"] - want), initial=0.0) <= 1e-7


def _logits(T, E, seed, skew=0.0):
    L = synth.normal("L", (T, E), 1.0, seed=seed).numpy().astype(np.float32)
    if skew:
        L = L + (skew * np.log(np.arange(1, E + 1, dtype=np.float64)) * -1.0).astype(np.float32)
    return L


@pytest.mark.parametrize("T,E,K", [(200, 8, 2), (97, 16, 4), (64, 256, 8)])
def test_unit_tile_is_plain_grouping(oracle_lib, T, E, K):
    # M = 1: every count is already a multiple, so nothing moves and the result
    # is the plain expert-grouped layout of the top-K routing
    L = _logits(T, E, seed=T + E)
    for renorm in (True, False):
        idx, w = oracle.topk_softmax(L, K, renorm)
        offsets, pt, ps, ros = oracle.permute(idx, E)
        tr = oracle.token_rounding(L, idx, 1, renorm)
        assert np.array_equal(tr["counts"], np.bincount(idx.ravel(), minlength=E))
        assert np.array_equal(tr["offsets"], offsets)
        assert np.array_equal(tr["perm_token"], pt)
        rm = tr["row_map"]
        assert np.count_nonzero(rm >= 0) == T * K
        t_of_slot = np.repeat(np.arange(T), K)
        assert np.array_equal(rm[t_of_slot, idx.ravel()], ros)
        assert np.array_equal(tr["row_w"][ros], w.ravel())


def test_counts_already_multiples_leave_routing_unchanged(oracle_lib):
    # 64 tokens, 4 experts, top-1, each expert the favourite of exactly 16 tokens
    T, E, M = 64, 4, 16
    rng = np.random.default_rng(5)
    L = rng.normal(size=(T, E)).astype(np.float32)
    fav = np.repeat(np.arange(E), T // E)
    rng.shuffle(fav)
    L[np.arange(T), fav] += 10.0
    idx, w = oracle.topk_softmax(L, 1)
    for m in (4, 8, 16):
        tr = oracle.token_rounding(L, idx, m)
        assert tr["counts"].tolist() == [16] * 4
        assert np.array_equal(tr["row_map"][np.arange(T), fav], oracle.permute(idx, E)[3])
        assert np.all(tr["row_w"] == 1.0)


def _key(L, e, t):
    # rank key of token t for expert e: higher logit first, then lower index
    return (float(L[t, e]), -int(t))


@pytest.mark.parametrize("T,E,K,M,skew", [(300, 8, 2, 16, 0.0), (257, 16, 4, 8, 0.0),
                                          (400, 32, 2, 32, 1.1), (130, 8, 8, 128, 0.0),
                                          (50, 4, 1, 7, 0.5)])
def test_rounding_invariants(oracle_lib, T, E, K, M, skew):
    L = _logits(T, E, seed=7 * T + E, skew=skew)
    idx, _ = oracle.topk_softmax(L, K)
    f = np.bincount(idx.ravel(), minlength=E)
    member = np.zeros((T, E), bool)
    member[np.repeat(np.arange(T), K), idx.ravel()] = True
    for renorm in (True, False):
        tr = oracle.token_rounding(L, idx, M, renorm)
        c, rm, pt, off, rw = tr["counts"], tr["row_map"], tr["perm_token"], tr["offsets"], tr["row_w"]
        assert np.all(c % M == 0) and np.all(c <= T)
        for e in range(E):
            lo, hi = f[e] // M * M, -(-f[e] // M) * M
            assert c[e] in (lo, hi)
            if hi <= T:
                # the nearer multiple; halves go up
                assert abs(c[e] - f[e]) <= abs(lo + hi - c[e] - f[e])
                if f[e] - lo == hi - f[e] and hi != lo:
                    assert c[e] == hi
            else:
                assert c[e] == lo
        kept = rm >= 0
        assert np.array_equal(kept.sum(axis=0), c)
        for e in range(E):
            k_e, m_e = kept[:, e], member[:, e]
            if c[e] <= f[e]:
                assert not np.any(k_e & ~m_e)
                pool_in, pool_out = np.flatnonzero(k_e), np.flatnonzero(m_e & ~k_e)
            else:
                assert not np.any(m_e & ~k_e)
                pool_in, pool_out = np.flatnonzero(k_e & ~m_e), np.flatnonzero(~m_e & ~k_e)
            if len(pool_in) and len(pool_out):
                assert min(_key(L, e, t) for t in pool_in) > max(_key(L, e, t) for t in pool_out)
        # grouped rows: expert-major, ascending t, consistent with row_map
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(c)]))
        for e in range(E):
            assert np.array_equal(pt[off[e]:off[e + 1]], np.flatnonzero(kept[:, e]))
        tt, ee = np.nonzero(kept)
        assert np.array_equal(pt[rm[tt, ee]], tt)
        assert sorted(rm[kept].tolist()) == list(range(int(off[-1])))
        # weights against scipy's softmax of the logit row
        P = softmax(L.astype(np.float64), axis=1)
        for t in range(T):
            es = np.flatnonzero(kept[t])
            if len(es) == 0:
                continue
            want = P[t, es] / P[t, es].sum() if renorm else P[t, es]
            assert np.max(np.abs(rw[rm[t, es]] - want)) <= 2e-7


def test_capacity_bound_is_reached_and_respected(oracle_lib):
    # every expert 1 row past half a tile: all round up, by M/2 - 1 each
    T, E, M = 1024, 8, 16
    L = np.zeros((T, E), np.float32)
    fav = np.concatenate([np.repeat(np.arange(E), 9), np.zeros(T - 9 * E, np.int64)])
    L[np.arange(T), fav] = 1.0
    idx, _ = oracle.topk_softmax(L, 1)
    tr = oracle.token_rounding(L, idx, M)
    f = np.bincount(idx.ravel(), minlength=E)
    assert np.all(tr["counts"] - f <= M // 2)
    assert tr["offsets"][-1] <= oracle.rounding_capacity(T, E, 1, M)


def test_combine_rows_against_numpy(oracle_lib):
    rng = np.random.default_rng(3)
    T, E, d = 37, 6, 24
    rm = np.full((T, E), -1, np.int32)
    kept = rng.random((T, E)) < 0.4
    rm[kept] = rng.permutation(int(kept.sum()))
    Z = rng.normal(size=(int(kept.sum()), d))
    Y = oracle.combine_rows(Z, rm)
    want = np.zeros((T, d))
    for t in range(T):
        for e in range(E):
            if rm[t, e] >= 0:
                want[t] += Z[rm[t, e]]
    got = oracle.bf16_bits_to_f64(Y)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-300)
    assert np.all(got[~kept.any(axis=1)] == 0.0)
    # with one row per (t, k) slot the map form and the slot form agree
    idx = np.stack([rng.choice(E, 2, replace=False) for _ in range(T)]).astype(np.int32)
    _, _, _, ros = oracle.permute(idx, E)
    rm2 = np.full((T, E), -1, np.int32)
    rm2[np.repeat(np.arange(T), 2), idx.ravel()] = ros
    Z2 = rng.normal(size=(2 * T, d))
    # the slot form sums in rank order, the map form in expert order: equal up to
    # the order of two addends, which the bf16 rounding hides except at halfway
    a, b = oracle.combine_rows(Z2, rm2), oracle.combine(Z2, ros, 2)
    assert np.mean(a == b) > 0.999


def test_rounded_layer_grouped_equals_token_by_token(oracle_lib):
    inp = synth.layer_inputs(T=96, d=64, E=4, n=64, zipf=False, seed=21)
    X, Wr = synth.bf16_bits(inp["X"]), inp["Wr"].numpy()
    W1, W3, W2 = synth.bf16_bits(inp["W1"]), synth.bf16_bits(inp["W3"]), synth.bf16_bits(inp["W2"])
    for M in (16, 32):
        out = oracle.forward_rounded(X, Wr, None, W1, W3, W2, K=2, M=M)
        assert np.all(out["counts"] % M == 0)
        Yt = oracle.forward_assigned(X, W1, W3, W2, out["row_map"], out["row_w"], np.arange(96))
        assert np.array_equal(out["Y"], Yt)
        dropped = ~(out["row_map"] >= 0).any(axis=1)
        assert np.all(out["Y"][dropped] == 0)
    # M = 1 reduces to the plain layer
    a = oracle.forward_rounded(X, Wr, None, W1, W3, W2, K=2, M=1)["Y"]
    b = oracle.forward(X, Wr, None, W1, W3, W2, K=2)["Y"]
    assert np.mean(a == b) > 0.999
