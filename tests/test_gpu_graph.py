"""moe_forward inside a CUDA graph: the layer issues only stream-ordered work
(kernel launches, one memset) and never synchronises with the host, so after one
warm-up call (which caches per-device set-up) a caller can capture it once and
replay it; every replay must match the oracle (routing bit-exact, Y within the
bf16 tolerance) and reproduce a direct call bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import W_ABS, bits, check_y, layer_np
from top_routing_grouped_02_gb300 import moe, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,pair", [("tiny", "0"), ("tiny", "1"), ("sonic", None)])
def test_forward_captured_in_cuda_graph_matches_direct_call(name, pair, monkeypatch):
    if pair is not None:
        monkeypatch.setenv("MOE_GEMM_CTA_PAIR", pair)
    cfg = synth.WORKLOADS[name]
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    inp = synth.layer_inputs(device="cuda", **cfg)
    ws = moe.workspace(T, d, E, K, n)
    Y_direct = moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K,
                               inp["bias"], ws=ws)
    torch.cuda.synchronize()
    Y = torch.empty_like(Y_direct)
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K,
                            inp["bias"], ws=ws, Y=Y, stream=side, topk_idx=idx, topk_w=w)
    ref = oracle.forward(*layer_np(inp), K)
    for _ in range(3):
        Y.zero_()
        idx.fill_(-1)
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), ref["idx"])
        assert float(np.abs(w.cpu().numpy().astype(np.float64) - ref["w"]).max()) <= W_ABS
        check_y(bits(Y), ref["Y"], "Y (graph replay)")
        assert torch.equal(Y.view(torch.int16), Y_direct.view(torch.int16))
    status, word = moe.moe_sync_check(ws)
    assert status == 0, word


def test_traced_forward_events_time_inside_a_captured_graph():
    # the stage events of moe_forward_traced become external event nodes when
    # the stream is capturing, so each replay records them and they can be timed
    cfg = synth.WORKLOADS["tiny"]
    T, d, E, K, n = cfg["T"], cfg["d"], cfg["E"], cfg["K"], cfg["n"]
    inp = synth.layer_inputs(device="cuda", **cfg)
    ws = moe.workspace(T, d, E, K, n)
    Y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record(side)
    with torch.cuda.stream(side):
        moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K, inp["bias"],
                        ws=ws, Y=Y, stream=side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K, inp["bias"],
                        ws=ws, Y=Y, stream=side, events=ev)
    with torch.cuda.stream(side):
        graph.replay()
    torch.cuda.synchronize()
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(5)]
    assert all(t > 0 for t in times), times
