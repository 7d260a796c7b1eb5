"""Thin ctypes binding over libmoe.so (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Tensors must be contiguous CUDA tensors of the dtype each call names;
their ``data_ptr()`` and the current torch stream are passed straight through.
There is no fallback: if libmoe.so is missing or a call fails, a ``MoeError``
is raised.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "moe.h")

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
          3: "MOE_ERR_WORKSPACE_TOO_SMALL", 4: "MOE_ERR_ARCH", 5: "MOE_ERR_CUDA",
          6: "MOE_ERR_DEVICE_TIMEOUT", 7: "MOE_ERR_DEVICE_CHECK"}
# Kernels each call enqueues; the gate/up GEMM launches one more (a row gather)
# when it runs on CTA pairs, the router's backward one fewer when T is too
# short to split into chunks, moe_permute one kernel instead of three for
# T <= 65536, and the whole-layer calls depend on the shape
# (forward_launches).
LAUNCHES = {"moe_route": 2, "moe_route_logits": 1, "moe_permute": 3, "moe_gemm_gate_up": 1,
            "moe_gemm_gate_up_train": 1, "moe_backward_dh": 2, "moe_backward_dx": 2,
            "moe_backward_router": 5, "moe_backward_dw": 5,
            "moe_gemm_down": 1, "moe_combine": 1, "moe_round_routing": 3, "moe_combine_rows": 1}
TILE_M = 128


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_abi_version": (_I, []),
    "moe_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_forward_launches": (_I, [_I, _I, _I, _I, _I, _I]),
    "moe_expert_mlp_launches": (_I, [_I, _I, _I, _I, _I, _I]),
    "moe_workspace_init": (_I, [_P, _SZ, _P]),
    "moe_route": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_route_logits": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "moe_permute": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_noalloc": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "moe_gemm_gate_up": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_gemm_down": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_gemm_gate_up_train": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _SZ,
                                    _P]),
    "moe_backward_dh": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                             _SZ, _P]),
    "moe_backward_dx": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "moe_backward_router": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                                 _P, _SZ, _P]),
    "moe_backward_dw_scratch_bytes": (_SZ, [_I, _I, _I, _I]),
    "moe_backward_dw": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P,
                             _P, _SZ, _P]),
    "moe_expert_mlp": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _SZ,
                            _P]),
    "moe_combine": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "moe_forward": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _SZ,
                         _P]),
    "moe_forward_traced": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                _SZ, _P, ctypes.POINTER(_P), _I]),
    "moe_forward_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ,
                              _P]),
    "moe_sync_check": (_I, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_selftest_wait_timeout": (_I, [_P, _SZ, _P]),
    "moe_forward_host_stream": (_I, [_P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                     _I, _P, _SZ, _P, _P, _P]),
    "moe_round_capacity": (ctypes.c_int64, [_I, _I, _I, _I]),
    "moe_round_workspace_bytes": (_SZ, [_I, _I]),
    "moe_round_routing": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                               _P]),
    "moe_combine_rows": (_I, [_P, _P, _I, _I, _I, ctypes.c_int64, _P, _P]),
    "moe_workspace_bytes_rounded": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_forward_rounded": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _SZ,
                                 _P]),
    "moe_forward_rounded_traced": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P,
                                        _SZ, _P, ctypes.POINTER(_P), _I]),
}


def header_symbols() -> list[str]:
    """Entry points declared in include/moe.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(moe_\w+)\s*\(", text, re.M)))


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def moe_workspace_bytes(T: int, d: int, E: int, K: int, n: int) -> int:
    return int(lib().moe_workspace_bytes(T, d, E, K, n))


def forward_launches(T: int, d: int, E: int, K: int, n: int, rounded: bool = False,
                     part: str = "forward") -> int:
    """Kernels moe_forward (or moe_forward_rounded) enqueues for this shape on the
    current device under the current environment (host only); part="expert_mlp":
    the expert GEMMs' share (1 when fused)."""
    fn = lib().moe_forward_launches if part == "forward" else lib().moe_expert_mlp_launches
    v = int(fn(T, d, E, K, n, int(rounded)))
    if v < 0:
        raise ValueError("invalid layer shape")
    return v


def workspace(T: int, d: int, E: int, K: int, n: int, device=None) -> torch.Tensor:
    """A zeroed workspace tensor (uint8) for this layer shape."""
    nbytes = moe_workspace_bytes(T, d, E, K, n)
    if nbytes == 0:
        raise ValueError("invalid layer shape")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check("moe_workspace_init", lib().moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)))


def moe_route(X, Wr, K: int, bias=None, renorm: bool = True, stream=None, logits=None):
    """(topk_idx [T,K] int32, topk_w [T,K] fp32, counts [E] int32); the router
    logits [T,E] fp32 land in `logits` (allocated when not given)."""
    T, d = X.shape
    E = Wr.shape[1]
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=X.device)
    idx = torch.empty((T, K), dtype=torch.int32, device=X.device)
    w = torch.empty((T, K), dtype=torch.float32, device=X.device)
    counts = torch.empty(E, dtype=torch.int32, device=X.device)
    _check("moe_route", lib().moe_route(
        _ptr(X, torch.bfloat16, "X"), _ptr(Wr, torch.float32, "Wr"), _ptr(bias, torch.float32, "bias"),
        T, d, E, K, int(bool(renorm)), _ptr(logits, torch.float32, "logits"), _ptr(idx), _ptr(w),
        _ptr(counts), _stream(stream)))
    return idx, w, counts


def moe_route_logits(logits, K: int, renorm: bool = True, stream=None):
    T, E = logits.shape
    idx = torch.empty((T, K), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, K), dtype=torch.float32, device=logits.device)
    counts = torch.empty(E, dtype=torch.int32, device=logits.device)
    _check("moe_route_logits", lib().moe_route_logits(
        _ptr(logits, torch.float32, "logits"), T, E, K, int(bool(renorm)), _ptr(idx), _ptr(w),
        _ptr(counts), _stream(stream)))
    return idx, w, counts


def moe_permute(topk_idx, E: int, counts=None, ws=None, stream=None) -> dict:
    T, K = topk_idx.shape
    R = T * K
    dev = topk_idx.device
    if ws is None:
        ws = workspace(T, 0, E, K, 0, dev)
    out = dict(
        offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
        perm_token=torch.empty(R, dtype=torch.int32, device=dev),
        perm_slot=torch.empty(R, dtype=torch.int32, device=dev),
        row_of_slot=torch.empty(R, dtype=torch.int32, device=dev),
        tiles=torch.zeros((R // TILE_M + E, 4), dtype=torch.int32, device=dev),
        num_tiles=torch.empty(1, dtype=torch.int32, device=dev),
    )
    _check("moe_permute", lib().moe_permute(
        _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(counts, torch.int32, "counts"), T, E, K,
        _ptr(out["offsets"]), _ptr(out["perm_token"]), _ptr(out["perm_slot"]),
        _ptr(out["row_of_slot"]), _ptr(out["tiles"]), _ptr(out["num_tiles"]), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def moe_permute_noalloc(topk_idx, E: int, counts=None, out: dict | None = None, stream=None) -> dict:
    """moe_permute without a workspace: the library uses its built-in 4 MiB
    scratch array, so this call allocates no device memory of its own. `out`
    may hold preallocated output tensors (same keys as moe_permute returns)."""
    T, K = topk_idx.shape
    R = T * K
    dev = topk_idx.device
    if out is None:
        out = dict(
            offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            perm_token=torch.empty(R, dtype=torch.int32, device=dev),
            perm_slot=torch.empty(R, dtype=torch.int32, device=dev),
            row_of_slot=torch.empty(R, dtype=torch.int32, device=dev),
            tiles=torch.zeros((R // TILE_M + E, 4), dtype=torch.int32, device=dev),
            num_tiles=torch.empty(1, dtype=torch.int32, device=dev),
        )
    _check("moe_permute_noalloc", lib().moe_permute_noalloc(
        _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(counts, torch.int32, "counts"), T, E, K,
        _ptr(out["offsets"]), _ptr(out["perm_token"]), _ptr(out["perm_slot"]),
        _ptr(out["row_of_slot"]), _ptr(out["tiles"]), _ptr(out["num_tiles"]), _stream(stream)))
    return out


def moe_gemm_gate_up(X, W1, W3, perm_token, offsets, K: int, ws=None, stream=None):
    T, d = X.shape
    E, _, n = W1.shape
    if ws is None:
        ws = workspace(T, d, E, K, n, X.device)
    H = torch.empty((T * K, n), dtype=torch.bfloat16, device=X.device)
    _check("moe_gemm_gate_up", lib().moe_gemm_gate_up(
        _ptr(X, torch.bfloat16, "X"), _ptr(W1, torch.bfloat16, "W1"), _ptr(W3, torch.bfloat16, "W3"),
        _ptr(perm_token, torch.int32), _ptr(offsets, torch.int32), T, d, E, K, n, _ptr(H),
        _ptr(ws), ws.numel(), _stream(stream)))
    return H


def moe_gemm_gate_up_train(X, W1, W3, perm_token, offsets, K: int, ws=None, stream=None):
    """(H [T*K, n] bf16, A1, A3 [T*K, n] fp32): H as moe_gemm_gate_up gives it
    and the pre-activations x W1[e], x W3[e] of every grouped row."""
    T, d = X.shape
    E, _, n = W1.shape
    if ws is None:
        ws = workspace(T, d, E, K, n, X.device)
    H = torch.empty((T * K, n), dtype=torch.bfloat16, device=X.device)
    A1, A3 = (torch.empty((T * K, n), dtype=torch.float32, device=X.device) for _ in range(2))
    _check("moe_gemm_gate_up_train", lib().moe_gemm_gate_up_train(
        _ptr(X, torch.bfloat16, "X"), _ptr(W1, torch.bfloat16, "W1"), _ptr(W3, torch.bfloat16, "W3"),
        _ptr(perm_token, torch.int32, "perm_token"), _ptr(offsets, torch.int32, "offsets"),
        T, d, E, K, n, _ptr(H), _ptr(A1), _ptr(A3), _ptr(ws), ws.numel(), _stream(stream)))
    return H, A1, A3


def moe_backward_dh(dY, W2, A1, A3, topk_w, perm_token, perm_slot, offsets, K: int, ws=None,
                    stream=None):
    """(dA1, dA3 [T*K, n] bf16, dS [T*K] fp32) of the grouped rows: the backward's
    dH step with the routing-weight gradient."""
    T, d = dY.shape
    E, n, _ = W2.shape
    if ws is None:
        ws = workspace(T, d, E, K, n, dY.device)
    dA1, dA3 = (torch.empty((T * K, n), dtype=torch.bfloat16, device=dY.device) for _ in range(2))
    dS = torch.zeros(T * K, dtype=torch.float32, device=dY.device)
    _check("moe_backward_dh", lib().moe_backward_dh(
        _ptr(dY, torch.bfloat16, "dY"), _ptr(W2, torch.bfloat16, "W2"), _ptr(A1, torch.float32, "A1"),
        _ptr(A3, torch.float32, "A3"), _ptr(topk_w, torch.float32, "topk_w"),
        _ptr(perm_token, torch.int32, "perm_token"), _ptr(perm_slot, torch.int32, "perm_slot"),
        _ptr(offsets, torch.int32, "offsets"), T, d, E, K, n, _ptr(dA1), _ptr(dA3), _ptr(dS),
        _ptr(ws), ws.numel(), _stream(stream)))
    return dA1, dA3, dS


def moe_backward_dx(dA1, dA3, W1, W3, offsets, row_of_slot, K: int, ws=None, stream=None):
    """(dXg [T*K, d] bf16 grouped rows, dX [T, d] bf16): the experts' share of the
    input gradient."""
    R, n = dA1.shape
    E, d, _ = W1.shape
    T = R // K
    if ws is None:
        ws = torch.zeros(256, dtype=torch.uint8, device=dA1.device)
    dXg = torch.empty((R, d), dtype=torch.bfloat16, device=dA1.device)
    dX = torch.empty((T, d), dtype=torch.bfloat16, device=dA1.device)
    _check("moe_backward_dx", lib().moe_backward_dx(
        _ptr(dA1, torch.bfloat16, "dA1"), _ptr(dA3, torch.bfloat16, "dA3"),
        _ptr(W1, torch.bfloat16, "W1"), _ptr(W3, torch.bfloat16, "W3"),
        _ptr(offsets, torch.int32, "offsets"), _ptr(row_of_slot, torch.int32, "row_of_slot"),
        T, d, E, K, n, _ptr(dXg), _ptr(dX), _ptr(ws), ws.numel(), _stream(stream)))
    return dXg, dX


def moe_backward_router(X, Wr, logits, topk_idx, dS, row_of_slot, dXg, renorm: bool = True,
                        ws=None, stream=None) -> dict:
    """The router's backward and the full input gradient: dict of dX [T, d] bf16,
    dL [T, E], dWr [d, E], dbias [E] fp32."""
    T, d = X.shape
    E = Wr.shape[1]
    K = topk_idx.shape[1]
    if ws is None:
        ws = workspace(T, d, E, K, 0, X.device)
    out = dict(dX=torch.empty((T, d), dtype=torch.bfloat16, device=X.device),
               dL=torch.empty((T, E), dtype=torch.float32, device=X.device),
               dWr=torch.empty((d, E), dtype=torch.float32, device=X.device),
               dbias=torch.empty(E, dtype=torch.float32, device=X.device))
    _check("moe_backward_router", lib().moe_backward_router(
        _ptr(X, torch.bfloat16, "X"), _ptr(Wr, torch.float32, "Wr"),
        _ptr(logits, torch.float32, "logits"), _ptr(topk_idx, torch.int32, "topk_idx"),
        _ptr(dS, torch.float32, "dS"), _ptr(row_of_slot, torch.int32, "row_of_slot"),
        T, d, E, K, int(bool(renorm)), _ptr(dXg, torch.bfloat16, "dXg"), _ptr(out["dX"]),
        _ptr(out["dL"]), _ptr(out["dWr"]), _ptr(out["dbias"]), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def moe_backward_dw(X, dY, H, dA1, dA3, topk_w, perm_token, perm_slot, offsets, K: int,
                    scratch=None, stream=None) -> dict:
    """Weight gradients dW1, dW3 [E, d, n] and dW2 [E, n, d], fp32."""
    T, d = X.shape
    E = offsets.shape[0] - 1
    n = dA1.shape[1]
    if scratch is None:
        nbytes = int(lib().moe_backward_dw_scratch_bytes(T, d, E, K))
        scratch = torch.zeros(nbytes, dtype=torch.uint8, device=X.device)
    out = dict(dW1=torch.empty((E, d, n), dtype=torch.float32, device=X.device),
               dW3=torch.empty((E, d, n), dtype=torch.float32, device=X.device),
               dW2=torch.empty((E, n, d), dtype=torch.float32, device=X.device))
    _check("moe_backward_dw", lib().moe_backward_dw(
        _ptr(X, torch.bfloat16, "X"), _ptr(dY, torch.bfloat16, "dY"), _ptr(H, torch.bfloat16, "H"),
        _ptr(dA1, torch.bfloat16, "dA1"), _ptr(dA3, torch.bfloat16, "dA3"),
        _ptr(topk_w, torch.float32, "topk_w"), _ptr(perm_token, torch.int32, "perm_token"),
        _ptr(perm_slot, torch.int32, "perm_slot"), _ptr(offsets, torch.int32, "offsets"),
        T, d, E, K, n, _ptr(out["dW1"]), _ptr(out["dW3"]), _ptr(out["dW2"]), _ptr(scratch),
        scratch.numel(), _stream(stream)))
    out["scratch"] = scratch
    return out


def moe_gemm_down(H, W2, topk_w, perm_slot, offsets, T: int, K: int, ws=None, stream=None):
    E, n, d = W2.shape
    if ws is None:
        ws = workspace(T, d, E, K, n, H.device)
    Z = torch.empty((T * K, d), dtype=torch.bfloat16, device=H.device)
    _check("moe_gemm_down", lib().moe_gemm_down(
        _ptr(H, torch.bfloat16, "H"), _ptr(W2, torch.bfloat16, "W2"), _ptr(topk_w, torch.float32),
        _ptr(perm_slot, torch.int32), _ptr(offsets, torch.int32), T, d, E, K, n, _ptr(Z),
        _ptr(ws), ws.numel(), _stream(stream)))
    return Z


def moe_expert_mlp(X, W1, W3, W2, topk_w, perm_token, perm_slot, offsets, K: int, ws=None,
                   stream=None):
    T, d = X.shape
    E, _, n = W1.shape
    if ws is None:
        ws = workspace(T, d, E, K, n, X.device)
    H = torch.empty((T * K, n), dtype=torch.bfloat16, device=X.device)
    Z = torch.empty((T * K, d), dtype=torch.bfloat16, device=X.device)
    _check("moe_expert_mlp", lib().moe_expert_mlp(
        _ptr(X, torch.bfloat16), _ptr(W1, torch.bfloat16), _ptr(W3, torch.bfloat16),
        _ptr(W2, torch.bfloat16), _ptr(topk_w, torch.float32), _ptr(perm_token, torch.int32),
        _ptr(perm_slot, torch.int32), _ptr(offsets, torch.int32), T, d, E, K, n, _ptr(H), _ptr(Z),
        _ptr(ws), ws.numel(), _stream(stream)))
    return H, Z


def moe_combine(Z, row_of_slot, K: int, stream=None):
    R, d = Z.shape
    T = row_of_slot.numel() // K
    Y = torch.empty((T, d), dtype=torch.bfloat16, device=Z.device)
    _check("moe_combine", lib().moe_combine(
        _ptr(Z, torch.bfloat16, "Z"), _ptr(row_of_slot, torch.int32), T, K, d, _ptr(Y),
        _stream(stream)))
    return Y


def moe_forward(X, Wr, W1, W3, W2, K: int, bias=None, renorm: bool = True, ws=None, Y=None,
                topk_idx=None, topk_w=None, stream=None, events=None):
    """Y [T,d] bf16 for the whole layer. Optional topk_idx/topk_w receive the
    routing; `events` (list of torch.cuda.Event) are recorded between stages."""
    T, d = X.shape
    E, _, n = W1.shape
    if ws is None:
        ws = workspace(T, d, E, K, n, X.device)
    if Y is None:
        Y = torch.empty((T, d), dtype=torch.bfloat16, device=X.device)
    args = (_ptr(X, torch.bfloat16, "X"), _ptr(Wr, torch.float32, "Wr"),
            _ptr(bias, torch.float32, "bias"), _ptr(W1, torch.bfloat16, "W1"),
            _ptr(W3, torch.bfloat16, "W3"), _ptr(W2, torch.bfloat16, "W2"), T, d, E, K, n,
            int(bool(renorm)), _ptr(Y, torch.bfloat16, "Y"), _ptr(topk_idx, torch.int32),
            _ptr(topk_w, torch.float32), _ptr(ws), ws.numel(), _stream(stream))
    if events:
        for e in events:
            if e.cuda_event == 0:  # torch creates the CUDA event on first record
                e.record()
        arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
        _check("moe_forward_traced", lib().moe_forward_traced(*args, arr, len(events)))
    else:
        _check("moe_forward", lib().moe_forward(*args))
    return Y


def moe_forward_host(X_host, Y_host, X_dev, Y_dev, Wr, W1, W3, W2, K: int, bias=None,
                     renorm: bool = True, ws=None, stream=None):
    """End to end from host memory (X_host/Y_host CPU bf16 tensors, ideally pinned);
    returns after Y_host holds the result."""
    T, d = X_host.shape
    E, _, n = W1.shape
    for name, t in (("X_host", X_host), ("Y_host", Y_host)):
        if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a contiguous CPU bf16 tensor")
    if ws is None:
        ws = workspace(T, d, E, K, n, X_dev.device)
    _check("moe_forward_host", lib().moe_forward_host(
        ctypes.c_void_p(X_host.data_ptr()), ctypes.c_void_p(Y_host.data_ptr()),
        _ptr(X_dev, torch.bfloat16), _ptr(Y_dev, torch.bfloat16), _ptr(Wr, torch.float32),
        _ptr(bias, torch.float32), _ptr(W1, torch.bfloat16), _ptr(W3, torch.bfloat16),
        _ptr(W2, torch.bfloat16), T, d, E, K, n, int(bool(renorm)), _ptr(ws), ws.numel(),
        _stream(stream)))
    return Y_host


def moe_forward_host_stream(X_host, Y_host, X_dev2, Y_dev2, Wr, W1, W3, W2, K: int, bias=None,
                            renorm: bool = True, ws=None, stream=None, h2d_stream=None,
                            d2h_stream=None):
    """n batches from host memory with copies overlapped: X_host / Y_host are CPU
    bf16 [n, T, d] (pinned), X_dev2 / Y_dev2 CUDA bf16 [2, T, d]. Returns after
    Y_host holds every output."""
    nb, T, d = X_host.shape
    E, _, n = W1.shape
    for name, t in (("X_host", X_host), ("Y_host", Y_host)):
        if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a contiguous CPU bf16 tensor")
    if tuple(X_dev2.shape) != (2, T, d) or tuple(Y_dev2.shape) != (2, T, d):
        raise ValueError("X_dev2 / Y_dev2 must be [2, T, d]")
    if ws is None:
        ws = workspace(T, d, E, K, n, X_dev2.device)
    if stream is None:
        stream = torch.cuda.current_stream()
    h2d_stream = h2d_stream or torch.cuda.Stream(device=X_dev2.device)
    d2h_stream = d2h_stream or torch.cuda.Stream(device=X_dev2.device)
    _check("moe_forward_host_stream", lib().moe_forward_host_stream(
        ctypes.c_void_p(X_host.data_ptr()), ctypes.c_void_p(Y_host.data_ptr()), nb,
        _ptr(X_dev2, torch.bfloat16), _ptr(Y_dev2, torch.bfloat16), _ptr(Wr, torch.float32),
        _ptr(bias, torch.float32), _ptr(W1, torch.bfloat16), _ptr(W3, torch.bfloat16),
        _ptr(W2, torch.bfloat16), T, d, E, K, n, int(bool(renorm)), _ptr(ws), ws.numel(),
        _stream(stream), _stream(h2d_stream), _stream(d2h_stream)))
    return Y_host


def moe_selftest_wait_timeout(ws, stream=None):
    """Enqueue the bounded-wait self-test (sets MOE_DEVERR_TIMEOUT after ~1 s)."""
    _check("moe_selftest_wait_timeout", lib().moe_selftest_wait_timeout(
        _ptr(ws), ws.numel(), _stream(stream)))


def moe_sync_check(ws, stream=None):
    """(status, raw error word) after waiting for the stream; clears the word."""
    word = ctypes.c_uint32(0)
    st = lib().moe_sync_check(_ptr(ws), _stream(stream), ctypes.byref(word))
    return int(st), int(word.value)


# ------------------------------------------------------------ Token Rounding

def moe_round_capacity(T: int, E: int, K: int, M: int = TILE_M) -> int:
    return int(lib().moe_round_capacity(T, E, K, M))


def moe_round_routing(logits, topk_idx, counts, M: int = TILE_M, renorm: bool = True, ws=None,
                      stream=None) -> dict:
    """Token Rounding of a top-K routing (outputs of moe_route). Returns counts,
    offsets, perm_token [capacity], row_map [T,E], row_w [capacity], tiles and
    num_tiles; offsets[E] entries of perm_token/row_w are meaningful."""
    T, E = logits.shape
    K = topk_idx.shape[1]
    dev = logits.device
    cap = moe_round_capacity(T, E, K, M)
    if cap < 0:
        raise ValueError("invalid Token Rounding shape")
    if ws is None:
        ws = torch.zeros(int(lib().moe_round_workspace_bytes(T, E)), dtype=torch.uint8, device=dev)
    out = dict(
        counts=torch.empty(E, dtype=torch.int32, device=dev),
        offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
        perm_token=torch.full((max(cap, 1),), -1, dtype=torch.int32, device=dev),
        row_map=torch.empty((T, E), dtype=torch.int32, device=dev),
        row_w=torch.zeros(max(cap, 1), dtype=torch.float32, device=dev),
        tiles=torch.zeros((cap // TILE_M + E, 4), dtype=torch.int32, device=dev),
        num_tiles=torch.empty(1, dtype=torch.int32, device=dev),
    )
    _check("moe_round_routing", lib().moe_round_routing(
        _ptr(logits, torch.float32, "logits"), _ptr(topk_idx, torch.int32, "topk_idx"),
        _ptr(counts, torch.int32, "counts"), T, E, K, M, int(bool(renorm)),
        _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm_token"]), _ptr(out["row_map"]),
        _ptr(out["row_w"]), _ptr(out["tiles"]), _ptr(out["num_tiles"]), _ptr(ws), ws.numel(),
        _stream(stream)))
    out["ws"] = ws
    return out


def moe_combine_rows(Z, row_map, stream=None):
    R, d = Z.shape
    T, E = row_map.shape
    Y = torch.empty((T, d), dtype=torch.bfloat16, device=Z.device)
    _check("moe_combine_rows", lib().moe_combine_rows(
        _ptr(Z, torch.bfloat16, "Z"), _ptr(row_map, torch.int32, "row_map"), T, E, d, R,
        _ptr(Y), _stream(stream)))
    return Y


def workspace_rounded(T: int, d: int, E: int, K: int, n: int, device=None) -> torch.Tensor:
    """A zeroed workspace tensor for moe_forward_rounded."""
    nbytes = int(lib().moe_workspace_bytes_rounded(T, d, E, K, n))
    if nbytes == 0:
        raise ValueError("invalid layer shape")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def moe_forward_rounded(X, Wr, W1, W3, W2, K: int, bias=None, renorm: bool = True, ws=None,
                        Y=None, row_map=None, stream=None, events=None):
    """Y [T,d] bf16 for the layer under Token Rounding (tile size 128). An optional
    row_map [T,E] int32 receives each (token, expert) row or -1."""
    T, d = X.shape
    E, _, n = W1.shape
    if ws is None:
        ws = workspace_rounded(T, d, E, K, n, X.device)
    if Y is None:
        Y = torch.empty((T, d), dtype=torch.bfloat16, device=X.device)
    args = (_ptr(X, torch.bfloat16, "X"), _ptr(Wr, torch.float32, "Wr"),
            _ptr(bias, torch.float32, "bias"), _ptr(W1, torch.bfloat16, "W1"),
            _ptr(W3, torch.bfloat16, "W3"), _ptr(W2, torch.bfloat16, "W2"), T, d, E, K, n,
            int(bool(renorm)), _ptr(Y, torch.bfloat16, "Y"), _ptr(row_map, torch.int32, "row_map"),
            _ptr(ws), ws.numel(), _stream(stream))
    if events:
        for e in events:
            if e.cuda_event == 0:
                e.record()
        arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
        _check("moe_forward_rounded_traced", lib().moe_forward_rounded_traced(*args, arr,
                                                                               len(events)))
    else:
        _check("moe_forward_rounded", lib().moe_forward_rounded(*args))
    return Y
