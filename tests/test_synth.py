"""The seeded input generator (CPU only): determinism, counter independence,
distribution moments, the Zipf bias profile."""
import math

import numpy as np
import torch

from top_routing_grouped_02_gb300 import synth


def test_hash32_reference_values_and_tensor_agreement():
    xs = [0, 1, 2, 0xDEADBEEF, 0xFFFFFFFF, 12345678]
    t = synth.hash32_t(torch.tensor(xs, dtype=torch.int64)).tolist()
    assert t == [synth.hash32(x) for x in xs]
    # lowbias32 is a bijection on 32-bit words: no collisions on a block of inputs
    block = synth.hash32_t(torch.arange(1 << 16, dtype=torch.int64))
    assert torch.unique(block).numel() == 1 << 16
    assert int(block.min()) >= 0 and int(block.max()) <= 0xFFFFFFFF


def test_normal_is_counter_based_and_chunk_independent(monkeypatch):
    a = synth.normal("W1", (3, 1000), 0.5, torch.float32)
    b = synth.normal("W1", (3000,), 0.5, torch.float32).view(3, 1000)
    assert torch.equal(a, b)
    monkeypatch.setattr(synth, "_CHUNK", 777)
    c = synth.normal("W1", (3, 1000), 0.5, torch.float32)
    assert torch.equal(a, c)
    assert not torch.equal(a, synth.normal("W3", (3, 1000), 0.5, torch.float32))
    assert not torch.equal(a, synth.normal("W1", (3, 1000), 0.5, torch.float32, seed=1))


def test_normal_moments():
    v = synth.normal("X", (400000,), 2.0, torch.float32).double()
    assert abs(v.mean().item()) < 0.02
    assert abs(v.std().item() - 2.0) < 0.02
    assert v.abs().max().item() <= 2.0 * 2 * math.sqrt(3) + 1e-6
    # Irwin-Hall(4) kurtosis is 3 - 1.2/4 = 2.7
    k = ((v - v.mean()) ** 4).mean() / v.var() ** 2
    assert abs(k.item() - 2.7) < 0.05


def test_bf16_bits_roundtrip():
    x = synth.normal("X", (64, 32), 1.0, torch.bfloat16)
    assert torch.equal(synth.bf16_from_bits(synth.bf16_bits(x)), x)


def test_zipf_bias_profile():
    b = synth.zipf_bias(256).double()
    ranks = torch.round(torch.exp(-b / synth.ZIPF_S)).long()
    assert sorted(ranks.tolist()) == list(range(1, 257))
    assert b.max().item() == 0.0
    assert torch.equal(synth.zipf_bias(256), synth.zipf_bias(256))


def test_layer_shapes_and_scales():
    inp = synth.layer_inputs(T=64, d=256, E=4, n=128)
    assert inp["X"].dtype == torch.bfloat16 and inp["X"].shape == (64, 256)
    assert inp["Wr"].dtype == torch.float32 and inp["Wr"].shape == (256, 4)
    assert inp["W1"].shape == (4, 256, 128) and inp["W2"].shape == (4, 128, 256)
    assert inp["bias"] is None
    assert abs(inp["W2"].double().std().item() - 1 / math.sqrt(128)) < 0.005
    assert abs(inp["Wr"].double().std().item() - 1 / math.sqrt(256)) < 0.005
