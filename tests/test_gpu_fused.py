"""The fused expert MLP: both expert GEMMs in one persistent launch (small n),
with each down unit waiting on counter words for the gate/up units of its row
tile. Checked against the oracle, and bit for bit against the two separate
single-CTA launches: every unit issues the same tensor-core instructions over
the same k-blocks, so only the order in which units run differs."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import bits, check_hz, layer_np
from top_routing_grouped_02_gb300 import moe, synth

pytestmark = pytest.mark.gpu

CASES = [
    # (T, d, E, K, n, zipf)
    (512, 256, 8, 2, 512, False),     # tiny workload
    (300, 512, 6, 3, 384, False),     # ragged tiles, several tiles per expert
    (97, 256, 16, 4, 128, True),      # many small and empty experts
    (1, 256, 4, 1, 128, False),       # one token: one tile, one expert
    (700, 256, 1, 1, 256, False),     # K = E = 1: one dense SwiGLU MLP
    (3000, 256, 32, 4, 128, True),    # Zipf-skewed loads
    (4096, 1536, 128, 4, 256, False), # SonicMoE-shaped experts, a quarter of its tokens
    (2048, 512, 8, 2, 1024, False),   # n above the default choice (forced on)
]


def _setup(T, d, E, K, n, zipf, seed=0):
    inp = synth.layer_inputs(T=T, d=d, E=E, n=n, zipf=zipf, device="cuda", seed=seed)
    X, Wr, bias, W1, W3, W2 = layer_np(inp)
    L = oracle.router_logits(X, Wr, bias)
    idx, w = oracle.topk_softmax(L, K, True)
    off, pt, ps, ros = oracle.permute(idx, E)
    dev = dict(w=torch.from_numpy(w).cuda(), pt=torch.from_numpy(pt).cuda(),
               ps=torch.from_numpy(ps).cuda(), off=torch.from_numpy(off).cuda())
    return inp, (X, W1, W3, W2), (w, off, pt, ps), dev


def _mlp(inp, dev, K, ws):
    H, Z = moe.moe_expert_mlp(inp["X"], inp["W1"], inp["W3"], inp["W2"], dev["w"], dev["pt"],
                              dev["ps"], dev["off"], K, ws=ws)
    st, word = moe.moe_sync_check(ws)
    assert st == 0, (st, hex(word))
    return H, Z


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.fixture
def single_cta(monkeypatch):
    monkeypatch.setenv("MOE_GEMM_CTA_PAIR", "0")
    return monkeypatch


@pytest.mark.parametrize("T,d,E,K,n,zipf", CASES)
def test_fused_matches_oracle_and_separate_launches(T, d, E, K, n, zipf, single_cta):
    inp, (X, W1, W3, W2), (w, off, pt, ps), dev = _setup(T, d, E, K, n, zipf)
    ws = moe.workspace(T, d, E, K, n)
    single_cta.setenv("MOE_GEMM_FUSED", "1")
    assert moe.forward_launches(T, d, E, K, n, part="expert_mlp") == 1
    H, Z = _mlp(inp, dev, K, ws)
    H_ref = oracle.gate_up(X, W1, W3, pt, off)
    check_hz(bits(H), H_ref, "H")
    check_hz(bits(Z), oracle.down(H_ref, W2, w, ps, off), "Z")
    single_cta.setenv("MOE_GEMM_FUSED", "0")
    assert moe.forward_launches(T, d, E, K, n, part="expert_mlp") == 2
    H2, Z2 = _mlp(inp, dev, K, ws)
    assert _same(H, H2) and _same(Z, Z2)


@pytest.mark.parametrize("gap", ["0", "1", "1000"])
def test_fused_unit_spacing(gap, single_cta):
    # 0: a down round may follow the gate/up round it reads right away, so many
    # units wait; 1000: every gate/up round before every down round
    T, d, E, K, n = 4096, 1536, 128, 4, 256
    inp, _, _, dev = _setup(T, d, E, K, n, False, seed=3)
    ws = moe.workspace(T, d, E, K, n)
    single_cta.setenv("MOE_GEMM_FUSED", "0")
    H0, Z0 = _mlp(inp, dev, K, ws)
    single_cta.setenv("MOE_GEMM_FUSED", "1")
    single_cta.setenv("MOE_FUSED_GAP_ROUNDS", gap)
    for _ in range(3):
        H, Z = _mlp(inp, dev, K, ws)
        assert _same(H, H0) and _same(Z, Z0)


def test_fused_workspace_reused_across_shapes(single_cta):
    # one workspace, filled with random bytes past its control words, serves
    # calls of three shapes in turn: counter words from other shapes and earlier
    # calls carry other epochs (or garbage) and must never complete a tile early
    shapes = [(512, 256, 8, 2, 512, False), (97, 256, 16, 4, 128, True),
              (1024, 768, 8, 2, 256, False)]
    nbytes = max(moe.moe_workspace_bytes(T, d, E, K, n) for T, d, E, K, n, _ in shapes)
    g = torch.Generator(device="cuda").manual_seed(7)
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)
    moe.moe_workspace_init(ws)
    runs = [_setup(*s, seed=i) for i, s in enumerate(shapes)]
    want = []
    single_cta.setenv("MOE_GEMM_FUSED", "0")
    for (T, d, E, K, n, _), (inp, _, _, dev) in zip(shapes, runs):
        want.append(_mlp(inp, dev, K, moe.workspace(T, d, E, K, n)))
    single_cta.setenv("MOE_GEMM_FUSED", "1")
    for _ in range(3):
        for (T, d, E, K, n, _), (inp, _, _, dev), (H0, Z0) in zip(shapes, runs, want):
            H, Z = _mlp(inp, dev, K, ws)
            assert _same(H, H0) and _same(Z, Z0)


def test_fused_forward_matches_unfused_forward(single_cta):
    cfg = dict(synth.WORKLOADS["tiny"])
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    inp = synth.layer_inputs(device="cuda", **cfg)
    out = {}
    for f in ("0", "1"):
        single_cta.setenv("MOE_GEMM_FUSED", f)
        ws = moe.workspace(T, d, E, K, n)
        out[f] = [moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K,
                                  inp["bias"], ws=ws) for _ in range(2)]
        st, word = moe.moe_sync_check(ws)
        assert st == 0, (st, hex(word))
    assert all(_same(y, out["0"][0]) for y in out["0"] + out["1"])
