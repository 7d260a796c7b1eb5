"""Seeded synthetic inputs for the MoE-layer workloads.

This module holds none of the layer's arithmetic: it only draws inputs. Both the
CUDA path (tests, benchmark) and the CPU oracle take their inputs from here, so
the two sides see identical bytes.

Generator. Counter-based: element i of tensor ``name`` depends only on
(seed, name, i). Each element takes two 32-bit words from the "lowbias32"
integer hash (C. Wellons, hash-prospector, 2018) keyed by (seed, name, lane,
high bits of i), splits them into four 16-bit uniforms and standardises their
sum (the Irwin-Hall construction of an approximate normal: mean 0, variance 1,
support |z| <= 2*sqrt(3)). Every step up to the final scaling is integer
arithmetic kept below 2**63, then one float64 multiply and IEEE round-to-nearest
conversions to fp32 / bf16. Those steps are exact or correctly rounded on any
device, so the CPU and the GPU produce the same bits, and large tensors can be
drawn on the GPU in chunks.

Workloads (the shapes the layer is measured and checked on):
  tiny     T=512   d=256  E=8   K=2 n=512
  router   logits [T,8] fp32 ~N(0,1), T in {256,512,1024,2048}, K=2
  mixtral  T=4096  d=4096 E=8   K=2 n=14336
  dsv3     T=8192  d=7168 E=256 K=8 n=2048, router bias from a Zipf(1.1) profile
  sonic    T=16384 d=1536 E=128 K=4 n=256
X ~ N(0,1) bf16; Wr ~ N(0,1/d) fp32; W1, W3 ~ N(0,1/d) bf16 [E,d,n];
W2 ~ N(0,1/n) bf16 [E,n,d].
"""
from __future__ import annotations

import math
import zlib

import torch

MASK32 = 0xFFFFFFFF
_CHUNK = 1 << 25

WORKLOADS = {
    "tiny": dict(T=512, d=256, E=8, K=2, n=512, zipf=False),
    "mixtral": dict(T=4096, d=4096, E=8, K=2, n=14336, zipf=False),
    "dsv3": dict(T=8192, d=7168, E=256, K=8, n=2048, zipf=True),
    "sonic": dict(T=16384, d=1536, E=128, K=4, n=256, zipf=False),
}
ROUTER_T = (256, 512, 1024, 2048)
ROUTER_E = 8
ROUTER_K = 2
ZIPF_S = 1.1


def _mul32_int(x: int, c: int) -> int:
    return (x * c) & MASK32


def hash32(x: int) -> int:
    """lowbias32 on a Python int in [0, 2**32)."""
    x &= MASK32
    x ^= x >> 16
    x = _mul32_int(x, 0x7FEB352D)
    x ^= x >> 15
    x = _mul32_int(x, 0x846CA68B)
    x ^= x >> 16
    return x


def _mul32_t(x: torch.Tensor, c: int) -> torch.Tensor:
    # (x * c) mod 2**32 for int64 x in [0, 2**32), split so no product passes 2**49
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & MASK32


def hash32_t(x: torch.Tensor) -> torch.Tensor:
    """lowbias32 on an int64 tensor with values in [0, 2**32)."""
    x = x ^ (x >> 16)
    x = _mul32_t(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32_t(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _key(seed: int, name: str, lane: int, hi: int) -> int:
    k = hash32((seed & MASK32) ^ zlib.crc32(name.encode()))
    k = hash32((k + lane * 0x9E3779B9) & MASK32)
    return hash32(k ^ hash32((hi + 0x85EBCA6B) & MASK32))


def normal(name: str, shape, std: float, dtype=torch.float32, device="cpu", seed: int = 0,
           out: torch.Tensor | None = None) -> torch.Tensor:
    """Approximate N(0, std**2) values, counter-based on (seed, name, flat index)."""
    numel = math.prod(shape)
    if out is None:
        out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    scale = std * math.sqrt(3.0) / 65536.0
    start = 0
    while start < numel:
        hi = start >> 32
        end = min(numel, start + _CHUNK, (hi + 1) << 32)
        k0, k1 = _key(seed, name, 0, hi), _key(seed, name, 1, hi)
        lo = torch.arange(start - (hi << 32), end - (hi << 32), dtype=torch.int64,
                          device=out.device)
        h0 = hash32_t(lo ^ k0)
        h1 = hash32_t(lo ^ k1)
        s = (h0 & 0xFFFF) + (h0 >> 16) + (h1 & 0xFFFF) + (h1 >> 16) - 131070
        v = s.to(torch.float64) * scale
        flat[start:end] = v.to(torch.float32).to(out.dtype)
        start = end
    return out


def zipf_bias(E: int, s: float = ZIPF_S, seed: int = 0) -> torch.Tensor:
    """Per-expert router bias -s*ln(r_e), r a seeded permutation of 1..E, so the
    prior routing odds of expert e fall off as r_e**-s (fp32, on the CPU)."""
    order = sorted(range(E), key=lambda e: hash32(e ^ _key(seed, "zipf", 0, 0)))
    rank = [0] * E
    for pos, e in enumerate(order):
        rank[e] = pos + 1
    return torch.tensor([-s * math.log(r) for r in rank], dtype=torch.float64).to(torch.float32)


def layer_inputs(T: int, d: int, E: int, n: int, zipf: bool = False, device="cpu",
                 seed: int = 0, **_ignored) -> dict:
    """X [T,d] bf16, Wr [d,E] fp32, bias [E] fp32 or None, W1/W3 [E,d,n] bf16,
    W2 [E,n,d] bf16."""
    X = normal("X", (T, d), 1.0, torch.bfloat16, device, seed)
    Wr = normal("Wr", (d, E), 1.0 / math.sqrt(d), torch.float32, device, seed)
    W1 = normal("W1", (E, d, n), 1.0 / math.sqrt(d), torch.bfloat16, device, seed)
    W3 = normal("W3", (E, d, n), 1.0 / math.sqrt(d), torch.bfloat16, device, seed)
    W2 = normal("W2", (E, n, d), 1.0 / math.sqrt(n), torch.bfloat16, device, seed)
    bias = zipf_bias(E, seed=seed).to(device) if zipf else None
    return dict(X=X, Wr=Wr, bias=bias, W1=W1, W3=W3, W2=W2)


def router_logits_input(T: int, E: int = ROUTER_E, device="cpu", seed: int = 0) -> torch.Tensor:
    """Given router logits [T,E] fp32 ~ N(0,1) (the router-only workload)."""
    return normal("logits", (T, E), 1.0, torch.float32, device, seed)


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a bf16 tensor's bits (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def bf16_from_bits(a, device="cpu") -> torch.Tensor:
    """bf16 tensor from a numpy uint16 array of bit patterns."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
