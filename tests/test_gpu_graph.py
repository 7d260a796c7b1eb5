"""moe_forward inside a CUDA graph: the layer issues only stream-ordered work
(kernel launches, one memset) and never synchronises with the host, so after one
warm-up call (which caches per-device set-up) a caller can capture it once and
replay it; the replay must reproduce a direct call bit for bit."""
import pytest
import torch

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
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            moe.moe_forward(inp["X"], inp["Wr"], inp["W1"], inp["W3"], inp["W2"], K,
                            inp["bias"], ws=ws, Y=Y, stream=side)
    for _ in range(3):
        Y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), Y_direct.view(torch.int16))
    status, word = moe.moe_sync_check(ws)
    assert status == 0, word
