"""Router parity on the GPU (through the C-ABI) against the oracle.

Top-K indices and per-expert counts bit-exact; weights within 1e-6.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_common import W_ABS, bits
from top_routing_grouped_02_gb300 import moe, synth

pytestmark = pytest.mark.gpu


def _check_routing(idx_g, w_g, counts_g, idx_r, w_r, E):
    assert np.array_equal(idx_g.cpu().numpy(), idx_r)
    assert float(np.abs(w_g.cpu().numpy().astype(np.float64) - w_r).max()) <= W_ABS
    assert np.array_equal(counts_g.cpu().numpy(), np.bincount(idx_r.ravel(), minlength=E))


def test_generator_gives_same_bits_on_cpu_and_gpu(monkeypatch):
    monkeypatch.setattr(synth, "_CHUNK", 1000)
    for dtype, std in ((torch.bfloat16, 1.0), (torch.float32, 0.03)):
        a = synth.normal("W1", (7, 531), std, dtype, "cpu")
        b = synth.normal("W1", (7, 531), std, dtype, "cuda").cpu()
        assert torch.equal(a.view(torch.int16) if dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if dtype == torch.bfloat16 else b.view(torch.int32))


@pytest.mark.parametrize("T", synth.ROUTER_T)
@pytest.mark.parametrize("renorm", [True, False])
def test_route_logits_router_only_workload(T, renorm):
    logits = synth.router_logits_input(T)
    idx_r, w_r = oracle.topk_softmax(logits.numpy(), synth.ROUTER_K, renorm)
    idx, w, counts = moe.moe_route_logits(logits.cuda(), synth.ROUTER_K, renorm)
    torch.cuda.synchronize()
    _check_routing(idx, w, counts, idx_r, w_r, synth.ROUTER_E)


@pytest.mark.parametrize("T,E,K", [(2049, 8, 2), (70000, 8, 2), (400000, 8, 2), (5000, 16, 4), (3001, 5, 3),
                                   (1 << 20, 8, 2)])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_logits_many_blocks_thread_per_token(T, E, K, renorm):
    # E <= 16 above 2048 tokens: one thread per token over many blocks, with ties
    # and signed zeros mixed in
    logits = synth.router_logits_input(T, E=E, seed=T)
    logits[::5] = torch.round(logits[::5])   # exact ties
    logits[1::97] = 0.0
    logits[2::97] = -0.0
    idx_r, w_r = oracle.topk_softmax(logits.numpy(), K, renorm)
    idx, w, counts = moe.moe_route_logits(logits.cuda(), K, renorm)
    torch.cuda.synchronize()
    _check_routing(idx, w, counts, idx_r, w_r, E)


@pytest.mark.parametrize("E,K", [(8, 1), (8, 8), (5, 2), (64, 6), (128, 4), (256, 8), (200, 3)])
def test_route_logits_ties_and_extremes(E, K):
    g = torch.Generator().manual_seed(E * 31 + K)
    T = 333
    L = torch.randn(T, E, generator=g)
    L[::4] = torch.randint(-2, 3, (len(L[::4]), E), generator=g).float()  # exact ties
    L[1] = 0.0
    L[2] = -0.0
    L[3, : E // 2] = 80.0
    L[3, E // 2:] = -80.0
    L = L.float().contiguous()
    for renorm in (True, False):
        idx_r, w_r = oracle.topk_softmax(L.numpy(), K, renorm)
        idx, w, counts = moe.moe_route_logits(L.cuda(), K, renorm)
        torch.cuda.synchronize()
        _check_routing(idx, w, counts, idx_r, w_r, E)


ROUTE_CASES = [
    # (T, d, E, K, zipf)
    (512, 256, 8, 2, False),      # tiny workload
    (4096, 4096, 8, 2, False),    # Mixtral-shaped router
    (8192, 7168, 256, 8, True),   # DeepSeek-V3-shaped router with Zipf bias
    (16384, 1536, 128, 4, False), # SonicMoE-shaped router
    (77, 40, 5, 2, False),        # ragged: d not a multiple of 32, odd E, partial block
    (1, 8, 3, 3, True),           # single token, E == K
    (300, 96, 64, 6, False),
    (129, 200, 16, 1, True),
    (65, 64, 200, 8, False),
    (100, 256, 100, 4, True),     # E not a multiple of 64: partial expert tile
    (40, 1024, 33, 2, False),     # smallest tiled E, scalar weight loads
    (1000, 512, 32, 4, False),    # largest per-thread-chain E
    (3000, 1000, 12, 3, False),   # E <= 32 kernel, d not a multiple of its stage
    # E <= 32: logits in 1024-step blocks and selection in one kernel, a warp per
    # (token group, block) item
    (600, 3000, 32, 4, True),     # 3 blocks: 3 warps per CTA, partial last block
    (200, 9216, 8, 2, False),     # 9 blocks: warps take 3, 2, 2, 2 items
    (64, 16392, 8, 2, False),     # 17 blocks
    (130, 2056, 20, 3, True),     # E padded to 32, a last block of 8 steps
    (37, 32776, 8, 2, False),     # 33 blocks: beyond the one-kernel router, the small kernel
    (5000, 2048, 16, 4, False),   # 2 blocks: 2 token groups per CTA
    (4100, 1024, 8, 2, True),     # 1 block: up to 4 token groups per CTA, partial last group
    (9, 520, 4, 4, False),        # E = K = 4 padded to 8, one partial group
    (333, 4096, 24, 8, True),     # E padded to 32, K = 8
]


def _route_case(T, d, E, K, zipf, renorm):
    X = synth.normal("X", (T, d), 1.0, torch.bfloat16, "cuda")
    Wr = synth.normal("Wr", (d, E), 1.0 / math.sqrt(d), torch.float32, "cuda")
    bias = synth.zipf_bias(E).cuda() if zipf else None
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    idx, w, counts = moe.moe_route(X, Wr, K, bias, renorm=renorm, logits=logits)
    torch.cuda.synchronize()
    Xn, Wn = bits(X), Wr.cpu().numpy()
    bn = None if bias is None else bias.cpu().numpy()
    L = oracle.router_logits(Xn, Wn, bn)
    # the logits themselves are the sequential fp32 chain: identical bits
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), L.view(np.uint32))
    idx_r, w_r = oracle.topk_softmax(L, K, renorm)
    _check_routing(idx, w, counts, idx_r, w_r, E)


@pytest.mark.parametrize("T,d,E,K,zipf", ROUTE_CASES)
def test_route_from_activations(T, d, E, K, zipf):
    _route_case(T, d, E, K, zipf, True)


@pytest.mark.parametrize("T,d,E,K,zipf", [(4096, 4096, 8, 2, False), (600, 3000, 32, 4, True),
                                          (9, 520, 4, 4, False), (1000, 512, 32, 4, False),
                                          (300, 96, 64, 6, False)])
def test_route_from_activations_without_renormalisation(T, d, E, K, zipf):
    _route_case(T, d, E, K, zipf, False)


def test_route_exact_ties_from_activations():
    # X = 0 gives all-zero logits: the first K experts win, each with weight 1/K
    T, d, E, K = 100, 2048, 8, 3
    X = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    Wr = synth.normal("Wr", (d, E), 1.0 / math.sqrt(d), torch.float32, "cuda")
    idx, w, counts = moe.moe_route(X, Wr, K)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), np.tile(np.arange(K, dtype=np.int32), (T, 1)))
    assert np.array_equal(w.cpu().numpy(), np.full((T, K), 1.0 / K, np.float32))
    assert np.array_equal(counts.cpu().numpy(), np.array([T] * K + [0] * (E - K), np.int32))


@pytest.mark.parametrize("pairs", ["4", "5", "6", "7", "8", None])
@pytest.mark.parametrize("T,d,E,K,zipf", [
    (9000, 200, 132, 4, True),   # second expert block holds 4 experts; d ends mid-stage
    (700, 72, 256, 8, False),    # two full expert blocks, partial token block
    (300, 96, 64, 6, False),     # fewer experts than a block
])
def test_router_logits_one_block_per_sm_kernel(T, d, E, K, zipf, pairs, monkeypatch):
    # the 2P-token x 8-expert register tile, for every P (None: the host's choice)
    if pairs is not None:
        monkeypatch.setenv("MOE_ROUTER_PAIRS", pairs)
    X = synth.normal("X", (T, d), 1.0, torch.bfloat16, "cuda")
    Wr = synth.normal("Wr", (d, E), 1.0 / math.sqrt(d), torch.float32, "cuda")
    bias = synth.zipf_bias(E).cuda() if zipf else None
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    idx, w, counts = moe.moe_route(X, Wr, K, bias, logits=logits)
    torch.cuda.synchronize()
    L = oracle.router_logits(bits(X), Wr.cpu().numpy(), None if bias is None else bias.cpu().numpy())
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), L.view(np.uint32))
    idx_r, w_r = oracle.topk_softmax(L, K, True)
    _check_routing(idx, w, counts, idx_r, w_r, E)


def test_route_zero_activations_and_exact_ties():
    T, d, E, K = 100, 64, 8, 3
    X = torch.zeros(T, d, dtype=torch.bfloat16, device="cuda")
    Wr = synth.normal("Wr", (d, E), 0.1, torch.float32, "cuda")
    idx, w, counts = moe.moe_route(X, Wr, K)
    torch.cuda.synchronize()
    assert torch.equal(idx.cpu(), torch.tensor([[0, 1, 2]] * T, dtype=torch.int32))
    assert torch.all(w.cpu() == np.float32(1 / 3))
    # integer-valued activations and weights: exact logits with many ties
    g = torch.Generator().manual_seed(7)
    Xi = torch.randint(-3, 4, (T, d), generator=g).to(torch.bfloat16)
    Wi = torch.randint(-2, 3, (d, E), generator=g).float()
    idx, w, counts = moe.moe_route(Xi.cuda(), Wi.cuda(), K)
    torch.cuda.synchronize()
    L = oracle.router_logits(bits(Xi), Wi.numpy())
    idx_r, w_r = oracle.topk_softmax(L, K, True)
    _check_routing(idx, w, counts, idx_r, w_r, E)


def test_route_unaligned_router_weights():
    # Wr starting 4 bytes into an allocation: the kernels must not use 16-byte loads
    for T, d, E, K in ((64, 128, 64, 4), (50, 256, 8, 2)):
        X = synth.normal("X", (T, d), 1.0, torch.bfloat16, "cuda")
        big = synth.normal("Wr", (d * E + 1,), 0.1, torch.float32, "cuda")
        Wr = big[1:].view(d, E)
        assert Wr.data_ptr() % 16 == 4
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        moe.moe_route(X, Wr, K, logits=logits)
        torch.cuda.synchronize()
        L = oracle.router_logits(bits(X), Wr.cpu().numpy())
        assert np.array_equal(logits.cpu().numpy().view(np.uint32), L.view(np.uint32))


def test_route_rejects_bad_arguments():
    X = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    Wr = torch.zeros(64, 8, dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route(X, Wr, 9)
    assert e.value.status in (1, 2)
    with pytest.raises(moe.MoeError):
        moe.moe_route(X[:, :60].contiguous(), Wr[:60].contiguous(), 2)  # d % 8 != 0
