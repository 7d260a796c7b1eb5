"""Near-tie report of the routing decisions (CPU).

The router's logits are fp32 sums in a fixed order (router_logits). A token
whose K-th and (K+1)-th best exact logits lie closer than the fp32 rounding
of those sums can change its top-K set with the summation order. This file
counts, for every workload, the tokens within 1e-5 of such a tie (float64
logits from one library matrix product) and the tokens whose top-K set under
the fp32 definition differs from the float64 one. The counts are reported, not
judged; the one check is the textbook bound on fp32 summation error: where the
two sets differ, the exact gap must be within twice the worst-case rounding
error of the logits involved (gamma_n * sum |x_j w_j| with n the chain length
plus the block and bias additions).
"""
import math

import numpy as np
import pytest

import oracle
from top_routing_grouped_02_gb300 import synth

U = 2.0 ** -24  # unit roundoff of fp32


def _router_inputs(name):
    c = synth.WORKLOADS[name]
    T, d, E = c["T"], c["d"], c["E"]
    X = synth.bf16_bits(synth.normal("X", (T, d), 1.0, synth.torch.bfloat16, "cpu", 0))
    Wr = synth.normal("Wr", (d, E), 1.0 / math.sqrt(d), synth.torch.float32, "cpu", 0).numpy()
    bias = synth.zipf_bias(E, seed=0).numpy() if c["zipf"] else None
    return X, Wr, bias, c["K"]


def _check_bound(X, Wr, bias, K, L32, rep):
    """Where the fp32 top-K set differs from the float64 one, the float64 gap
    at the K-th place is within the worst-case fp32 error of two logits."""
    if rep["fp32_topk_differs_from_f64"] == 0:
        return
    Xf = oracle.bf16_bits_to_f64(X)
    Wf = Wr.astype(np.float64)
    L64 = Xf @ Wf + (0.0 if bias is None else bias.astype(np.float64))
    idx32, _ = oracle.topk_softmax(L32, K, True)
    T, E = L64.shape
    d = X.shape[1]
    n = d + 2 + (d + 1023) // 1024  # chain steps, block additions, bias
    gamma = n * U / (1 - n * U)
    mag = np.abs(Xf) @ np.abs(Wf)  # sum_j |x_j w_je| per (t, e)
    srt = -np.sort(-L64, axis=1)
    for t in range(T):
        order = np.lexsort((np.arange(E), -L64[t]))
        if set(order[:K]) == set(idx32[t]):
            continue
        gap = srt[t, K - 1] - srt[t, K]
        bound = 2 * gamma * (mag[t].max() + (0.0 if bias is None else np.abs(bias).max()))
        assert gap <= bound, (t, gap, bound)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "sonic", "dsv3"])
def test_near_tie_report_layer_workloads(name, oracle_lib):
    X, Wr, bias, K = _router_inputs(name)
    L32 = oracle.router_logits(X, Wr, bias)
    rep = oracle.near_ties(X, Wr, bias, K, tol=1e-5, L32=L32)
    print(f"\n{name}: {rep}")
    assert rep["tokens"] == X.shape[0]
    _check_bound(X, Wr, bias, K, L32, rep)


def test_near_tie_report_router_only(oracle_lib):
    # given fp32 logits: no summation order is involved, only the gaps
    for T in synth.ROUTER_T:
        L = synth.router_logits_input(T).numpy()
        srt = -np.sort(-L.astype(np.float64), axis=1)
        gap = srt[:, synth.ROUTER_K - 1] - srt[:, synth.ROUTER_K]
        print(f"\nrouter-only T={T}: near ties (gap < 1e-5): {int(np.sum(gap < 1e-5))}, "
              f"exact ties: {int(np.sum(gap == 0))}, min gap {gap.min():.3e}")


def test_near_tie_report_counts_a_planted_tie(oracle_lib):
    # d = 8, E = 4, K = 2: token 0's second and third logits differ by 2^-20
    # (a near-tie), token 1's by 0.5; the report must count exactly one
    X = np.full((2, 8), 0x3F80, np.uint16)  # x = 1.0 everywhere, except
    X[0, 1] = 0x0000                        # token 0: x_1 = 0
    X[1, 0] = 0x0000                        # token 1: x_0 = 0
    Wr = np.zeros((8, 4), np.float32)
    Wr[0] = [1.0, 0.5, 0.5 + 2.0 ** -20, 0.0]
    Wr[1] = [2.0, 1.0, 0.5, 0.0]
    rep = oracle.near_ties(X, Wr, None, 2, tol=1e-5)
    # token 0 logits: [1, 0.5, 0.5 + 2^-20, 0]; token 1: [2, 1, 0.5, 0]
    assert rep["near_ties"] == 1
    assert rep["fp32_topk_differs_from_f64"] == 0
    assert rep["min_gap"] == pytest.approx(2.0 ** -20)
