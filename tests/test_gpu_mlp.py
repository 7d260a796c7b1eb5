"""Expert GEMM and combine parity on the GPU against the oracle, each step fed
the oracle's own inputs (routing, grouping, H) so a mismatch points at one kernel."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_common import bits, check_hz, check_y, layer_np
from top_routing_grouped_02_gb300 import moe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["single", "pair"], autouse=True)
def gemm_variant(request, monkeypatch):
    # run every GEMM case on both kernels: one CTA per tile, and CTA pairs
    # (cta_group::2) that the library otherwise picks only for large experts
    monkeypatch.setenv("MOE_GEMM_CTA_PAIR", "1" if request.param == "pair" else "0")
    return request.param

MLP_CASES = [
    # (T, d, E, K, n, zipf)
    (512, 256, 8, 2, 512, False),   # tiny workload
    (300, 512, 6, 3, 384, False),   # ragged tiles, several 128-row tiles per expert
    (97, 256, 16, 4, 128, True),    # many small / empty experts
    (1, 256, 4, 1, 128, False),     # one token
    (700, 256, 1, 1, 256, False),   # K = E = 1: one dense SwiGLU MLP
    (1024, 768, 8, 2, 256, False),  # rows per expert around exact tile multiples
    # Zipf-skewed loads: experts with at most two tiles (one pair) and experts with
    # more, so the GEMM's unit order interleaves both streams
    (2000, 256, 8, 1, 256, True),   # 6 light and 2 heavy experts
    (3000, 256, 32, 4, 128, True),  # 22 light and 10 heavy experts
]


def _setup(T, d, E, K, n, zipf, seed=0):
    inp = synth.layer_inputs(T=T, d=d, E=E, n=n, zipf=zipf, device="cuda", seed=seed)
    X, Wr, bias, W1, W3, W2 = layer_np(inp)
    L = oracle.router_logits(X, Wr, bias)
    idx, w = oracle.topk_softmax(L, K, True)
    off, pt, ps, ros = oracle.permute(idx, E)
    return inp, (X, W1, W3, W2), idx, w, off, pt, ps, ros


@pytest.mark.parametrize("T,d,E,K,n,zipf", MLP_CASES)
def test_gate_up_swiglu_matches_oracle(T, d, E, K, n, zipf):
    inp, (X, W1, W3, W2), idx, w, off, pt, ps, ros = _setup(T, d, E, K, n, zipf)
    H_ref = oracle.gate_up(X, W1, W3, pt, off)
    H = moe.moe_gemm_gate_up(inp["X"], inp["W1"], inp["W3"], torch.from_numpy(pt).cuda(),
                             torch.from_numpy(off).cuda(), K)
    torch.cuda.synchronize()
    check_hz(bits(H), H_ref, "H")


@pytest.mark.parametrize("T,d,E,K,n,zipf", MLP_CASES)
def test_down_weighted_matches_oracle(T, d, E, K, n, zipf):
    inp, (X, W1, W3, W2), idx, w, off, pt, ps, ros = _setup(T, d, E, K, n, zipf)
    H_ref = oracle.gate_up(X, W1, W3, pt, off)
    Z_ref = oracle.down(H_ref, W2, w, ps, off)
    Z = moe.moe_gemm_down(synth.bf16_from_bits(H_ref, "cuda"), inp["W2"],
                          torch.from_numpy(w).cuda(), torch.from_numpy(ps).cuda(),
                          torch.from_numpy(off).cuda(), T, K)
    torch.cuda.synchronize()
    check_hz(bits(Z), Z_ref, "Z")


@pytest.mark.parametrize("T,K,d", [(512, 2, 256), (333, 8, 7168), (1, 1, 8), (4096, 4, 1536)])
def test_combine_matches_oracle(T, K, d):
    Zb = synth.normal("Z", (T * K, d), 0.5, torch.bfloat16, "cuda")
    ros = np.random.default_rng(T + K).permutation(T * K).astype(np.int32)
    Y_ref = oracle.combine_bf16(bits(Zb), ros, K)
    Y = moe.moe_combine(Zb, torch.from_numpy(ros).cuda(), K)
    torch.cuda.synchronize()
    got = bits(Y)
    # one rounding of an fp32 sum vs of a float64 sum: equal or one bf16 step apart
    diff = np.abs(got.astype(np.int32) - Y_ref.astype(np.int32))
    assert np.mean(diff == 0) > 0.999
    check_y(got, Y_ref, "Y")


def test_gemm_rejects_unsupported_shapes():
    X = torch.zeros(8, 200, dtype=torch.bfloat16, device="cuda")  # d % 256 != 0
    W = torch.zeros(2, 200, 128, dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros(8, dtype=torch.int32, device="cuda")
    off = torch.tensor([0, 8, 8], dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_gemm_gate_up(X, W, W, pt, off, 1)
    assert e.value.status == 2
