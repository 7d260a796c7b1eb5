"""Failure detection on the GPU without a GPU fault.

Every pipeline wait in the kernels is bounded (about one second): a wait that
gives up sets MOE_DEVERR_TIMEOUT in the workspace's error word and the kernel
returns, so the host learns of it from moe_sync_check and the context stays
usable. Bad data the kernels can detect (offsets that are not a split of the
rows, token indices out of range) is flagged in the same word and skipped, with
nothing read or written out of bounds.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import bits, check_hz
from top_routing_grouped_02_gb300 import moe, synth

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_TIMEOUT = 6
MOE_ERR_DEVICE_CHECK = 7
DEVERR_TIMEOUT = 0x1
DEVERR_BAD_EXPERT = 0x2


def _tiny():
    cfg = dict(synth.WORKLOADS["tiny"])
    return cfg, synth.layer_inputs(device="cuda", **cfg)


def test_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    cfg, inp = _tiny()
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    ws = moe.workspace(T, d, E, K, n)
    moe.moe_selftest_wait_timeout(ws)
    status, word = moe.moe_sync_check(ws)
    assert status == MOE_ERR_DEVICE_TIMEOUT and (word & DEVERR_TIMEOUT)
    # the word was cleared and the device still runs the layer
    Y = moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K, inp["bias"],
                        ws=ws)
    status, word = moe.moe_sync_check(ws)
    assert status == 0 and word == 0
    assert torch.isfinite(Y.float()).all()


@pytest.mark.parametrize("pair", ["0", "1"])
def test_gemm_does_no_work_on_offsets_that_are_not_a_split(pair, monkeypatch):
    monkeypatch.setenv("MOE_GEMM_CTA_PAIR", pair)
    cfg, inp = _tiny()
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    R = T * K
    ws = moe.workspace(T, d, E, K, n)
    perm_token = torch.arange(R, dtype=torch.int32, device="cuda") // K
    bad = torch.tensor([0, 300, 200, 500, 600, 700, 800, 900, R], dtype=torch.int32,
                       device="cuda")  # decreasing at expert 1
    H = torch.full((R, n), 7.0, dtype=torch.bfloat16, device="cuda")
    status = moe.lib().moe_gemm_gate_up(
        moe._ptr(inp["X"]), moe._ptr(inp["W1"]), moe._ptr(inp["W3"]), moe._ptr(perm_token),
        moe._ptr(bad), T, d, E, K, n, moe._ptr(H), moe._ptr(ws), ws.numel(), moe._stream(None))
    assert status == 0
    status, word = moe.moe_sync_check(ws)
    assert status == MOE_ERR_DEVICE_CHECK and (word & DEVERR_BAD_EXPERT)
    assert bool((H.float() == 7.0).all())  # nothing was written


@pytest.mark.parametrize("pair", ["0", "1"])
def test_gemm_skips_token_indices_out_of_range(pair, monkeypatch):
    monkeypatch.setenv("MOE_GEMM_CTA_PAIR", pair)
    cfg, inp = _tiny()
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    idx, w, counts = moe.moe_route(inp["X"], inp["Wr"], K, inp["bias"])
    ws = moe.workspace(T, d, E, K, n)
    g = moe.moe_permute(idx, E, counts=counts, ws=ws)
    offsets = g["offsets"].cpu().numpy()
    pt = g["perm_token"].clone()
    # corrupt two rows of expert 0 (below 0, beyond T)
    r0 = int(offsets[0])
    pt[r0] = -3
    pt[r0 + 1] = T + 5
    H = moe.moe_gemm_gate_up(inp["X"], inp["W1"], inp["W3"], pt, g["offsets"], K, ws=ws)
    status, word = moe.moe_sync_check(ws)
    assert status == MOE_ERR_DEVICE_CHECK and (word & DEVERR_BAD_EXPERT)
    # every other expert's rows are still exact
    X, W1, W3 = bits(inp["X"]), bits(inp["W1"]), bits(inp["W3"])
    H_ref = oracle.gate_up(X, W1, W3, g["perm_token"].cpu().numpy(), offsets)
    lo = int(offsets[1])
    check_hz(bits(H)[lo:], H_ref[lo:], "H (experts 1..E-1)")
