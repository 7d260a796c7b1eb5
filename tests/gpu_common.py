"""Shared helpers of the GPU parity tests: tolerances, comparisons, input setup."""
import numpy as np
import torch

import oracle
from top_routing_grouped_02_gb300 import synth

# Tolerances for bf16 outputs with fp32 accumulation (Y, checked against the
# oracle's float64 values): max-abs <= 2e-2 and relative Frobenius <= 5e-3;
# routing weights within 1e-6 absolute. Intermediates H and Z are bf16 values
# of magnitude up to ~10, where one bf16 step is 2^-4; they are checked
# relative to max(1, |ref|) within 2^-6 (two bf16 steps of a value in [1,2))
# and with the same Frobenius bound.
Y_MAX_ABS = 2e-2
Y_REL_FRO = 5e-3
W_ABS = 1e-6
HZ_REL = 2.0 ** -6


def bits(t: torch.Tensor) -> np.ndarray:
    """numpy uint16 bits of a bf16 tensor (any device)."""
    return synth.bf16_bits(t)


def f64_of_bits(a: np.ndarray) -> np.ndarray:
    return oracle.bf16_bits_to_f64(a)


def check_y(got_bits: np.ndarray, ref, what="Y"):
    """got: bf16 bits; ref: float64 values or bf16 bits."""
    g = f64_of_bits(got_bits)
    r = ref if ref.dtype == np.float64 else f64_of_bits(ref)
    err = np.abs(g - r)
    max_abs = float(err.max()) if err.size else 0.0
    fro = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    assert max_abs <= Y_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {Y_MAX_ABS}"
    assert fro <= Y_REL_FRO, f"{what}: rel-Frobenius {fro:.3e} > {Y_REL_FRO}"
    return max_abs, fro


def check_hz(got_bits: np.ndarray, ref, what="H"):
    g = f64_of_bits(got_bits)
    r = ref if ref.dtype == np.float64 else f64_of_bits(ref)
    rel = np.abs(g - r) / np.maximum(1.0, np.abs(r))
    worst = float(rel.max()) if rel.size else 0.0
    fro = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    assert worst <= HZ_REL, f"{what}: max |d|/max(1,|ref|) {worst:.3e} > {HZ_REL}"
    assert fro <= Y_REL_FRO, f"{what}: rel-Frobenius {fro:.3e} > {Y_REL_FRO}"
    return worst, fro


def layer_np(inp: dict):
    """numpy views for the oracle from a dict of (CPU or GPU) input tensors."""
    bias = inp["bias"]
    return (bits(inp["X"]), inp["Wr"].detach().cpu().numpy(),
            None if bias is None else bias.detach().cpu().numpy(),
            bits(inp["W1"]), bits(inp["W3"]), bits(inp["W2"]))


def to_dev(inp: dict, device="cuda") -> dict:
    return {k: (None if v is None else v.to(device).contiguous()) for k, v in inp.items()}
