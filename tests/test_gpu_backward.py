"""The backward's dH step on the GPU against the oracle (through the C-ABI).

moe_gemm_gate_up_train must give H bit for bit as moe_gemm_gate_up does and
the pre-activations A1 = x W1[e], A3 = x W3[e] (fp32) within the tolerance
below of the oracle's unrounded products. moe_backward_dh, fed with those, must give
dA1, dA3 and the routing-weight gradient dS of every grouped row within the
tolerance the forward's H and Z are held to, against oracle.backward_rows
(the gradient of sum(Y * dY) with the top-K choice fixed, in double), and
moe_backward_dx, fed with dA1 and dA3, each row's share of dX within that
tolerance and their sum per token within the Y tolerance; moe_backward_dw the
weight gradients dW1, dW3, dW2 within the fp32 bound below (an expert that no
token chose gets exact zeros); moe_backward_router
the logits' gradient dL, dbias and dWr within the fp32 bound below and the full
input gradient dX (experts' rows plus the router's share) within the Y
tolerance, against oracle.backward.

A row's quantities depend only on its token, its expert and the weights, so
on the SonicMoE and Mixtral shapes the oracle runs on sampled tokens alone
(their own grouping) and its rows are matched to the full grouping's through
the slots.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_common import bits, check_hz, check_y, f64_of_bits, layer_np
from top_routing_grouped_02_gb300 import moe, synth

pytestmark = pytest.mark.gpu

REL = 2.0 ** -6
FRO = 5e-3


def check_f32(got: np.ndarray, ref: np.ndarray, what: str):
    """fp32 values against float64 ones: |d| / max(1, |ref|) and relative Frobenius."""
    got = got.astype(np.float64)
    worst = float((np.abs(got - ref) / np.maximum(1.0, np.abs(ref))).max())
    fro = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    assert worst <= REL, f"{what}: max |d|/max(1,|ref|) {worst:.3e} > {REL}"
    assert fro <= FRO, f"{what}: rel-Frobenius {fro:.3e} > {FRO}"


def _gpu_steps(inp, dY, K):
    T, d = inp["X"].shape
    E, _, n = inp["W1"].shape
    ws = moe.workspace(T, d, E, K, n)
    E_ = inp["Wr"].shape[1]
    logits = torch.empty((T, E_), dtype=torch.float32, device="cuda")
    idx, w, counts = moe.moe_route(inp["X"], inp["Wr"], K, inp["bias"], logits=logits)
    g = moe.moe_permute(idx, E, counts=counts, ws=ws)
    H0 = moe.moe_gemm_gate_up(inp["X"], inp["W1"], inp["W3"], g["perm_token"], g["offsets"], K, ws=ws)
    H, A1, A3 = moe.moe_gemm_gate_up_train(inp["X"], inp["W1"], inp["W3"], g["perm_token"],
                                           g["offsets"], K, ws=ws)
    dA1, dA3, dS = moe.moe_backward_dh(dY, inp["W2"], A1, A3, w.view(-1), g["perm_token"],
                                       g["perm_slot"], g["offsets"], K, ws=ws)
    dXg, dX = moe.moe_backward_dx(dA1, dA3, inp["W1"], inp["W3"], g["offsets"], g["row_of_slot"],
                                  K, ws=ws)
    rb = moe.moe_backward_router(inp["X"], inp["Wr"], logits, idx, dS, g["row_of_slot"], dXg, ws=ws)
    torch.cuda.synchronize()
    st, word = moe.moe_sync_check(ws)
    assert st == 0, (st, word)
    R = int(g["offsets"][-1].item())
    # the training gate/up GEMM stores H exactly as the forward one does
    assert torch.equal(H[:R].view(torch.int16), H0[:R].view(torch.int16))
    return dict(idx=idx, H=H, A1=A1, A3=A3, dA1=dA1, dA3=dA3, dS=dS, dXg=dXg, dX_experts=dX,
                dX=rb["dX"], dL=rb["dL"], dWr=rb["dWr"], dbias=rb["dbias"], **g)


def _f64(a):
    # fp32 router weights and bias widen to float64 exactly
    return None if a is None else np.asarray(a, np.float64)


def _dY(T, d):
    return synth.normal("dY", (T, d), 1.0, torch.bfloat16, "cuda", seed=7)


@pytest.mark.parametrize("pair", ["0", "1"])
def test_backward_dh_matches_oracle_in_full(pair, monkeypatch):
    # the tiny layer, with the training gate/up GEMM on single CTAs and on CTA
    # pairs (the dH GEMM runs single CTAs either way)
    monkeypatch.setenv("MOE_GEMM_CTA_PAIR", pair)
    cfg = synth.WORKLOADS["tiny"]
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    inp = synth.layer_inputs(device="cuda", **cfg)
    dY = _dY(T, d)
    s = _gpu_steps(inp, dY, K)
    X, Wr, bias, W1, W3, W2 = layer_np(inp)
    idx_r, _ = oracle.topk_softmax(oracle.router_logits(X, Wr, bias), K, True)
    assert np.array_equal(s["idx"].cpu().numpy(), idx_r)
    off_r, pt_r, ps_r, _ = oracle.permute(idx_r, E)
    A1r, A3r = oracle.gate_up_pre(X, W1, W3, pt_r, off_r)
    check_f32(s["A1"].cpu().numpy(), A1r, "A1")
    check_f32(s["A3"].cpu().numpy(), A3r, "A3")
    ref = oracle.backward_rows(X, _f64(Wr), _f64(bias), W1, W3, W2, idx_r, ps_r,
                               f64_of_bits(bits(dY)))
    check_hz(bits(s["dA1"]), ref["dA1"], "dA1")
    check_hz(bits(s["dA3"]), ref["dA3"], "dA3")
    check_f32(s["dS"].cpu().numpy(), ref["dS"], "dS")
    # dX step: each row's share, then the sum over a token's rows
    check_hz(bits(s["dXg"]), ref["dXg"], "dXg")
    _, _, _, ros_r = oracle.permute(idx_r, E)
    check_y(bits(s["dX_experts"]), oracle.combine(ref["dXg"], ros_r, K), "dX (experts' share)")
    # the router's backward and the full input gradient
    check_f32(s["dL"].cpu().numpy(), ref["dL"], "dL")
    full = oracle.backward(X, _f64(Wr), _f64(bias), W1, W3, W2, idx_r, f64_of_bits(bits(dY)))
    check_f32(s["dbias"].cpu().numpy(), full["dbias"], "dbias")
    check_f32(s["dWr"].cpu().numpy(), full["dWr"], "dWr")
    check_y(bits(s["dX"]), full["dX"], "dX")


@pytest.mark.parametrize("T,E,K,d", [
    (300, 20, 2, 256),    # E <= 32 with a partly used 32-expert block; 10 token chunks
    (300, 40, 3, 256),    # E > 32: two expert blocks; 5 chunks
    (300, 256, 8, 256),   # E = 256: T too short for chunks, dWr written directly
    (4100, 8, 2, 256),    # 129 chunks of 32 tokens, the last one ragged
    (2048, 128, 4, 256),  # dWr on the tensor cores: 2 chunks of 1024 tokens
    (2048, 128, 1, 256),  # the same with K = 1: no second scratch, dL Wr^T in the combine
    (1024, 256, 8, 768),  # the same with E = 256 (two 256-column blocks) and 6 row tiles
])
def test_router_backward_matches_oracle(T, E, K, d):
    n = 256
    inp = synth.layer_inputs(T=T, d=d, E=E, n=n, device="cuda", seed=3)
    dY = _dY(T, d)
    s = _gpu_steps(inp, dY, K)
    X, Wr, bias, W1, W3, W2 = layer_np(inp)
    idx_r, _ = oracle.topk_softmax(oracle.router_logits(X, Wr, bias), K, True)
    assert np.array_equal(s["idx"].cpu().numpy(), idx_r)
    _, _, ps_r, _ = oracle.permute(idx_r, E)
    ref = oracle.backward_rows(X, _f64(Wr), _f64(bias), W1, W3, W2, idx_r, ps_r,
                               f64_of_bits(bits(dY)))
    check_f32(s["dL"].cpu().numpy(), ref["dL"], "dL")
    full = oracle.backward(X, _f64(Wr), _f64(bias), W1, W3, W2, idx_r, f64_of_bits(bits(dY)))
    check_f32(s["dbias"].cpu().numpy(), full["dbias"], "dbias")
    check_f32(s["dWr"].cpu().numpy(), full["dWr"], "dWr")
    check_y(bits(s["dX"]), full["dX"], "dX")


@pytest.mark.parametrize("workload,ntok", [("sonic", 192), ("mixtral", 48)])
def test_backward_full_shape_sampled_tokens(workload, ntok):
    # The full layer on the GPU (Mixtral: CTA-pair training gate/up at the full
    # reduction depth); the oracle on the sampled tokens alone, with their own
    # grouping. (The DeepSeek-V3 shape is left out: the oracle would widen its
    # 22.5 GB of expert weights to double.)
    cfg = synth.WORKLOADS[workload]
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    inp = synth.layer_inputs(device="cuda", **cfg)
    dY = _dY(T, d)
    s = _gpu_steps(inp, dY, K)
    X, Wr, bias, W1, W3, W2 = layer_np(inp)
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(T, size=ntok, replace=False))
    toks[0], toks[-1] = 0, T - 1
    idx_full = s["idx"].cpu().numpy()
    # the oracle's routing of those tokens is the GPU's (checked bit for bit in
    # the router tests); the sub-problem keeps it fixed
    L = oracle.router_logits(X[toks], Wr, bias)
    idx_sub, _ = oracle.topk_softmax(L, K, True)
    assert np.array_equal(idx_sub, idx_full[toks])
    _, _, ps_sub, _ = oracle.permute(idx_sub, E)
    ref = oracle.backward_rows(X[toks], _f64(Wr), _f64(bias), W1, W3, W2, idx_sub, ps_sub,
                               f64_of_bits(bits(dY))[toks])
    # sub-problem row p holds slot ps_sub[p] = t' * K + k of token toks[t']; its
    # row in the full grouping is row_of_slot[toks[t'] * K + k]
    ros = s["row_of_slot"].cpu().numpy()
    full_rows = ros[toks[ps_sub // K] * K + ps_sub % K]
    P = torch.from_numpy(full_rows.astype(np.int64)).cuda()
    check_hz(bits(s["dA1"][P]), ref["dA1"], "dA1 (sampled tokens)")
    check_hz(bits(s["dA3"][P]), ref["dA3"], "dA3 (sampled tokens)")
    check_f32(s["dS"][P].cpu().numpy(), ref["dS"], "dS (sampled tokens)")
    check_hz(bits(s["dXg"][P]), ref["dXg"], "dXg (sampled tokens)")
    # the sampled tokens' dX: the oracle's combine over the sub-problem's rows
    _, _, _, ros_sub = oracle.permute(idx_sub, E)
    Tt = torch.from_numpy(toks.astype(np.int64)).cuda()
    dx_experts = oracle.combine(ref["dXg"], ros_sub, K)
    check_y(bits(s["dX_experts"][Tt]), dx_experts, "dX, experts' share (sampled tokens)")
    # per-token quantities of the router's backward on the same sub-problem
    check_f32(s["dL"][Tt].cpu().numpy(), ref["dL"], "dL (sampled tokens)")
    # the full input gradient: each token's rows of dXg (double, unrounded) plus
    # the router's share dL Wr^T, from the oracle's per-row quantities (its
    # whole-layer backward would also form every expert's weight gradient)
    rows_of = ros_sub.reshape(len(toks), K)
    dx_rows = np.stack([ref["dXg"][r[r >= 0]].sum(axis=0) for r in rows_of])
    check_y(bits(s["dX"][Tt]), dx_rows + ref["dL"] @ _f64(Wr).T, "dX (sampled tokens)")


def test_backward_dh_rejects_n_not_a_multiple_of_256():
    T, d, E, K, n = 64, 256, 4, 2, 384
    z = torch.zeros
    with pytest.raises(moe.MoeError) as e:
        moe.moe_backward_dh(z((T, d), dtype=torch.bfloat16, device="cuda"),
                            z((E, n, d), dtype=torch.bfloat16, device="cuda"),
                            z((T * K, n), dtype=torch.float32, device="cuda"),
                            z((T * K, n), dtype=torch.float32, device="cuda"),
                            z(T * K, dtype=torch.float32, device="cuda"),
                            z(T * K, dtype=torch.int32, device="cuda"),
                            z(T * K, dtype=torch.int32, device="cuda"),
                            z(E + 1, dtype=torch.int32, device="cuda"), K)
    assert e.value.status == 2


@pytest.mark.parametrize("T,d,E,K,n,empty", [
    (512, 256, 8, 2, 512, None),   # the tiny layer
    (300, 256, 16, 2, 256, 5),     # expert 5 chosen by no token: its gradients are zero
    (700, 512, 4, 3, 768, None),   # several 64-row k-blocks and 128-row output tiles per expert
])
@pytest.mark.parametrize("pair", ["0", "1"])
def test_weight_gradients_match_oracle(T, d, E, K, n, empty, pair, monkeypatch):
    # single CTAs, and CTA pairs (two 128-row output tiles a unit)
    monkeypatch.setenv("MOE_GEMM_CTA_PAIR", pair)
    inp = synth.layer_inputs(T=T, d=d, E=E, n=n, device="cuda", seed=T)
    if empty is not None:
        bias = torch.zeros(E, dtype=torch.float32)
        bias[empty] = -100.0
        inp["bias"] = bias.cuda()
    dY = _dY(T, d)
    ws = moe.workspace(T, d, E, K, n)
    idx, w, counts = moe.moe_route(inp["X"], inp["Wr"], K, inp["bias"])
    g = moe.moe_permute(idx, E, counts=counts, ws=ws)
    H, A1, A3 = moe.moe_gemm_gate_up_train(inp["X"], inp["W1"], inp["W3"], g["perm_token"],
                                           g["offsets"], K, ws=ws)
    dA1, dA3, dS = moe.moe_backward_dh(dY, inp["W2"], A1, A3, w.view(-1), g["perm_token"],
                                       g["perm_slot"], g["offsets"], K, ws=ws)
    out = moe.moe_backward_dw(inp["X"], dY, H, dA1, dA3, w.view(-1), g["perm_token"],
                              g["perm_slot"], g["offsets"], K)
    torch.cuda.synchronize()
    for buf in (ws, out["scratch"]):
        st, word = moe.moe_sync_check(buf)
        assert st == 0, (st, word)
    X, Wr, bias, W1, W3, W2 = layer_np(inp)
    idx_r, _ = oracle.topk_softmax(oracle.router_logits(X, Wr, bias), K, True)
    assert np.array_equal(idx.cpu().numpy(), idx_r)
    if empty is not None:
        assert int(counts[empty].item()) == 0
        for k in ("dW1", "dW3", "dW2"):
            assert torch.count_nonzero(out[k][empty]).item() == 0
    full = oracle.backward(X, _f64(Wr), _f64(bias), W1, W3, W2, idx_r, f64_of_bits(bits(dY)))
    # Each gradient entry is a sum over the expert's rows of products whose GPU
    # operands are bf16 (dA1, dA3; H and w dY), each within 2^-8 of the exact
    # value. So |error| <= 2^-8 * sum_p |a_p b_p| plus the fp32 accumulation's
    # share; the check allows twice that, with the sums of absolute products
    # taken from the oracle's own operands, and the relative Frobenius bound.
    off_r, pt_r, ps_r, _ = oracle.permute(idx_r, E)
    rows = oracle.backward_rows(X, _f64(Wr), _f64(bias), W1, W3, W2, idx_r, ps_r,
                                f64_of_bits(bits(dY)))
    A1r, A3r = oracle.gate_up_pre(X, W1, W3, pt_r, off_r)
    h_r = np.abs(A1r / (1.0 + np.exp(-A1r)) * A3r)
    _, w_r = oracle.topk_softmax(oracle.router_logits(X, Wr, bias), K, True)
    wdy = np.abs(w_r.reshape(-1)[ps_r].astype(np.float64)[:, None]
                 * f64_of_bits(bits(dY))[pt_r])
    xg = np.abs(oracle.bf16_bits_to_f64(X)[pt_r])
    for k, a, b in (("dW1", xg, np.abs(rows["dA1"])), ("dW3", xg, np.abs(rows["dA3"])),
                    ("dW2", h_r, wdy)):
        got = out[k].cpu().numpy().astype(np.float64)
        ref = full[k]
        for e in range(E):
            r0, r1 = int(off_r[e]), int(off_r[e + 1])
            bound = 2.0 ** -7 * (a[r0:r1].T @ b[r0:r1]) + 1e-6
            err = np.abs(got[e] - ref[e])
            assert np.all(err <= bound), (k, e, float((err / bound).max()))
        fro = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
        assert fro <= FRO, f"{k}: rel-Frobenius {fro:.3e} > {FRO}"
