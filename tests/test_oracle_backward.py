"""Pins of the oracle's backward pass (CPU only).

The backward is the gradient of sum(Y * dY) for the layer with the top-K choice
held fixed, in double, without the forward pass's bf16 roundings (they pass
gradients through unchanged). It is checked against things other than itself:
central finite differences of the oracle's fixed-choice forward for every
element of every input, a dense SwiGLU MLP differentiated by torch autograd
(K = E = 1), and closed forms of the router's softmax gradient.
"""
import numpy as np
import pytest
import torch

import oracle


def _tiny(T=3, d=6, E=4, K=2, n=5, seed=0):
    rng = np.random.default_rng(seed)
    inp = {
        "X": rng.normal(0, 1, (T, d)),
        "Wr": rng.normal(0, 0.7, (d, E)),
        "bias": rng.normal(0, 0.3, E),
        "W1": rng.normal(0, 0.5, (E, d, n)),
        "W3": rng.normal(0, 0.5, (E, d, n)),
        "W2": rng.normal(0, 0.5, (E, n, d)),
    }
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    dY = rng.normal(0, 1, (T, d))
    return inp, idx, dY


def _loss(inp, idx, dY, renorm):
    Y = oracle.forward_fixed(inp["X"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"],
                             idx, renorm)
    return float(np.sum(Y * dY))


@pytest.mark.parametrize("renorm", [True, False])
def test_backward_matches_central_differences(oracle_lib, renorm):
    inp, idx, dY = _tiny()
    g = oracle.backward(inp["X"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], idx,
                        dY, renorm)
    h = 1e-6
    for name in ("X", "Wr", "bias", "W1", "W3", "W2"):
        num = np.zeros_like(inp[name])
        it = np.nditer(inp[name], flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            v = inp[name][i]
            inp[name][i] = v + h
            up = _loss(inp, idx, dY, renorm)
            inp[name][i] = v - h
            dn = _loss(inp, idx, dY, renorm)
            inp[name][i] = v
            num[i] = (up - dn) / (2 * h)
        ana = g["d" + name]
        scale = max(1.0, float(np.max(np.abs(num))))
        assert np.max(np.abs(ana - num)) <= 1e-6 * scale, (name, np.max(np.abs(ana - num)))


def test_backward_single_expert_matches_autograd(oracle_lib):
    # K = E = 1 with renormalisation: the weight is exactly 1 and the layer is a
    # dense SwiGLU MLP, so torch autograd (float64) gives the reference gradients;
    # the router gets none
    inp, _, dY = _tiny(T=5, d=7, E=1, K=1, n=6, seed=4)
    idx = np.zeros((5, 1), np.int32)
    g = oracle.backward(inp["X"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], idx,
                        dY, True)
    X = torch.tensor(inp["X"], requires_grad=True)
    W1 = torch.tensor(inp["W1"][0], requires_grad=True)
    W3 = torch.tensor(inp["W3"][0], requires_grad=True)
    W2 = torch.tensor(inp["W2"][0], requires_grad=True)
    Y = (torch.nn.functional.silu(X @ W1) * (X @ W3)) @ W2
    (Y * torch.tensor(dY)).sum().backward()
    for ours, ref in ((g["dX"], X.grad), (g["dW1"][0], W1.grad), (g["dW3"][0], W3.grad),
                      (g["dW2"][0], W2.grad)):
        assert np.allclose(ours, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(g["dWr"] == 0.0) and np.all(g["dbias"] == 0.0)


@pytest.mark.parametrize("renorm", [True, False])
def test_router_gradient_sums_to_zero_over_experts(oracle_lib, renorm):
    # dL = p * (dp - sum_e p_e dp_e) sums to zero over the experts of every token,
    # so dbias sums to zero and so does every row of dWr
    inp, idx, dY = _tiny(T=6, d=5, E=6, K=3, n=4, seed=2)
    g = oracle.backward(inp["X"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], idx,
                        dY, renorm)
    assert abs(g["dbias"].sum()) <= 1e-12 * max(1.0, np.abs(g["dbias"]).max())
    assert np.max(np.abs(g["dWr"].sum(axis=1))) <= 1e-12 * max(1.0, np.abs(g["dWr"]).max())
    assert np.abs(g["dbias"]).max() > 1e-6  # and is not zero itself


def test_identical_experts_give_the_router_no_gradient(oracle_lib):
    # with every expert the same and renormalised weights, Y = MLP(x) whatever the
    # weights are, so the router parameters get zero gradient
    inp, idx, dY = _tiny(T=4, d=6, E=5, K=3, n=4, seed=6)
    for w in ("W1", "W3", "W2"):
        inp[w][:] = inp[w][0]
    g = oracle.backward(inp["X"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], idx,
                        dY, True)
    assert np.max(np.abs(g["dWr"])) <= 1e-12 and np.max(np.abs(g["dbias"])) <= 1e-12
    assert np.max(np.abs(g["dX"])) > 1e-3


@pytest.mark.parametrize("renorm", [True, False])
def test_backward_rows_sum_to_the_backward(oracle_lib, renorm):
    # the per-row quantities, summed per token and per expert as their definition
    # says, give the token-by-token backward (itself pinned by finite differences)
    inp, idx, dY = _tiny(T=7, d=6, E=4, K=3, n=5, seed=3)
    T, d = inp["X"].shape
    E, _, n = inp["W1"].shape
    K = idx.shape[1]
    off, pt, ps, ros = oracle.permute(idx, E)
    r = oracle.backward_rows(inp["X"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"],
                             idx, ps, dY, renorm)
    g = oracle.backward(inp["X"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], idx,
                        dY, renorm)
    dX = r["dL"] @ inp["Wr"].T
    dW1 = np.zeros_like(g["dW1"])
    dW3 = np.zeros_like(g["dW3"])
    for p in range(T * K):
        t, e = pt[p], idx.ravel()[ps[p]]
        assert ps[p] // K == t
        dX[t] += r["dXg"][p]
        dW1[e] += np.outer(inp["X"][t], r["dA1"][p])
        dW3[e] += np.outer(inp["X"][t], r["dA3"][p])
    # rows of one expert are contiguous in the grouped order
    for e in range(E):
        assert np.all(idx.ravel()[ps[off[e]:off[e + 1]]] == e)
    for name, got in (("dX", dX), ("dW1", dW1), ("dW3", dW3), ("dWr", inp["X"].T @ r["dL"]),
                      ("dbias", r["dL"].sum(axis=0))):
        want = g[name]
        assert np.max(np.abs(got - want)) <= 1e-12 * max(1.0, np.max(np.abs(want))), name


def test_backward_rows_weight_gradient_is_output_dot_dy(oracle_lib):
    # dS of row (t, k) is dY[t] . o with o = (silu(x W1) * (x W3)) W2 of expert
    # idx[t, k], the routed output before its weight
    inp, idx, dY = _tiny(T=5, d=6, E=4, K=2, n=5, seed=7)
    T, _ = inp["X"].shape
    E = inp["W1"].shape[0]
    K = idx.shape[1]
    _, pt, ps, _ = oracle.permute(idx, E)
    r = oracle.backward_rows(inp["X"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"],
                             idx, ps, dY, True)
    x_t = torch.tensor(inp["X"], dtype=torch.float64)
    for p in range(T * K):
        t, e = int(pt[p]), int(idx.ravel()[ps[p]])
        a1 = x_t[t] @ torch.tensor(inp["W1"][e])
        a3 = x_t[t] @ torch.tensor(inp["W3"][e])
        o = (torch.nn.functional.silu(a1) * a3) @ torch.tensor(inp["W2"][e])
        assert abs(float(o @ torch.tensor(dY[t])) - r["dS"][p]) <= 1e-12 * max(1.0, abs(r["dS"][p]))
