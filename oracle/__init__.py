"""CPU oracle for the forward pass of one Mixture-of-Experts layer.

TEST INFRASTRUCTURE ONLY. The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers. The CUDA library never
imports, links or runs anything here, and nothing here comes from it.

The arithmetic lives in ``moe_oracle.c`` (plain C11, built with gcc); this module
builds it and marshals numpy arrays through ctypes. bf16 arrays are passed as
their raw uint16 bit patterns. See ``moe_oracle.h`` for the definition each
function follows and the page sections it cites.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library next to this file."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    hdr = os.path.join(_HERE, "moe_oracle.h")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC), os.path.getmtime(hdr))):
        return _LIB_PATH
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math"]
    if platform.machine() in ("x86_64", "AMD64"):
        cmd.append("-mfma")  # hardware fmaf; fmaf is correctly rounded with or without it
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd += [_SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            sig = {
                "oracle_bf16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
                "oracle_bf16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
                "oracle_router_logits": (None, [P, P, P, I64, I, I, P]),
                "oracle_gate_up_pre": (None, [P, P, P, P, P, I, I, I, P, P]),
                "oracle_topk_softmax": (None, [P, I64, I, I, I, P, P]),
                "oracle_expert_counts": (None, [P, I64, I, I, P]),
                "oracle_permute": (None, [P, I64, I, I, P, P, P, P]),
                "oracle_tile_schedule": (I, [P, I, I, P, I]),
                "oracle_gate_up": (None, [P, P, P, P, P, I, I, I, P]),
                "oracle_down": (None, [P, P, P, P, P, I, I, I, P]),
                "oracle_combine": (None, [P, P, I64, I, I, P]),
                "oracle_combine_bf16": (None, [P, P, I64, I, I, P]),
                "oracle_forward_tokens": (None, [P, P, P, P, P, P, I64, I, I, I, I, I, P, I64,
                                                 P, P, P]),
                "oracle_token_rounding": (I64, [P, P, I64, I, I, I, I, I64, P, P, P, P, P]),
                "oracle_combine_rows": (None, [P, P, I64, I, I, P]),
                "oracle_combine_rows_bf16": (None, [P, P, I64, I, I, P]),
                "oracle_forward_assigned": (None, [P, P, P, P, I64, I, I, I, P, P, P, I64, P]),
                "oracle_num_threads": (I, []),
                "oracle_forward_fixed": (None, [P, P, P, P, P, P, P, I64, I, I, I, I, I, P]),
                "oracle_backward": (None, [P, P, P, P, P, P, P, P, I64, I, I, I, I, I,
                                           P, P, P, P, P, P]),
                "oracle_backward_rows": (None, [P, P, P, P, P, P, P, P, P, I64, I, I, I, I, I,
                                                P, P, P, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().oracle_num_threads()


def bf16_from_double(v: float) -> int:
    return int(_load().oracle_bf16_from_double(float(v)))


def bf16_to_double(b: int) -> float:
    return float(_load().oracle_bf16_to_double(int(b)))


def router_logits(X: np.ndarray, Wr: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """L[T,E] fp32: an fma chain over j ascending from +0.0f (with E <= 32, one
    chain per 1024-step block of j, the block sums added in ascending block
    order), + bias. X uint16 (bf16) [T,d]."""
    X = _c(X, np.uint16)
    Wr = _c(Wr, np.float32)
    T, d = X.shape
    E = Wr.shape[1]
    assert Wr.shape[0] == d
    if bias is not None:
        bias = _c(bias, np.float32)
        assert bias.shape == (E,)
    L = np.empty((T, E), np.float32)
    _load().oracle_router_logits(_p(X), _p(Wr), _p(bias), T, d, E, _p(L))
    return L


def topk_softmax(L: np.ndarray, K: int, renorm: bool = True):
    """(idx int32 [T,K], w fp32 [T,K]) from logits L fp32 [T,E]."""
    L = _c(L, np.float32)
    T, E = L.shape
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    _load().oracle_topk_softmax(_p(L), T, E, K, int(bool(renorm)), _p(idx), _p(w))
    return idx, w


def near_ties(X: np.ndarray, Wr: np.ndarray, bias: np.ndarray | None, K: int,
               tol: float = 1e-5, L32: np.ndarray | None = None) -> dict:
    """How many routing decisions of a workload sit on a near-tie (a report:
    nothing fails).

    The float64 logits X Wr (+ bias) come from one library matrix product. A
    token is a near-tie when its K-th and (K+1)-th largest float64 logits lie
    within `tol` of each other: its top-K set can then depend on the rounding
    of the fp32 logits, i.e. on the fixed summation order of the router's fp32
    definition (router_logits). The report also counts the tokens whose top-K
    set under that fp32 definition (L32, computed when not given) differs from
    the float64 one. X uint16 (bf16) [T,d]."""
    Xf = bf16_bits_to_f64(_c(X, np.uint16))
    L64 = Xf @ _c(Wr, np.float32).astype(np.float64)
    if bias is not None:
        L64 = L64 + _c(bias, np.float32).astype(np.float64)
    T, E = L64.shape
    if L32 is None:
        L32 = router_logits(X, Wr, bias)
    idx32, _ = topk_softmax(L32, K, True)
    # float64 top-K set: sort by (-score, expert), the same tie rule
    order = np.lexsort((np.broadcast_to(np.arange(E), (T, E)), -L64), axis=1)
    set64 = np.sort(order[:, :K], axis=1)
    differs = int(np.sum(np.any(np.sort(idx32, axis=1) != set64, axis=1)))
    if K < E:
        srt = -np.sort(-L64, axis=1)
        gap = srt[:, K - 1] - srt[:, K]
        n_ties = int(np.sum(gap < tol))
        min_gap = float(gap.min())
    else:
        n_ties, min_gap = 0, float("inf")
    return dict(tokens=T, near_ties=n_ties, tol=tol, min_gap=min_gap,
                fp32_topk_differs_from_f64=differs)


def expert_counts(idx: np.ndarray, E: int) -> np.ndarray:
    idx = _c(idx, np.int32)
    T, K = idx.shape
    counts = np.empty(E, np.int32)
    _load().oracle_expert_counts(_p(idx), T, K, E, _p(counts))
    return counts


def permute(idx: np.ndarray, E: int):
    """(offsets [E+1], perm_token [R], perm_slot [R], row_of_slot [R]), all int32."""
    idx = _c(idx, np.int32)
    T, K = idx.shape
    R = T * K
    offsets = np.empty(E + 1, np.int32)
    perm_token = np.empty(R, np.int32)
    perm_slot = np.empty(R, np.int32)
    row_of_slot = np.empty(R, np.int32)
    _load().oracle_permute(_p(idx), T, E, K, _p(offsets), _p(perm_token), _p(perm_slot),
                           _p(row_of_slot))
    return offsets, perm_token, perm_slot, row_of_slot


def tile_schedule(offsets: np.ndarray, M: int) -> np.ndarray:
    """int32 [num_tiles, 4] = {expert, first row, rows, 0}."""
    offsets = _c(offsets, np.int32)
    E = offsets.shape[0] - 1
    max_tiles = int(offsets[E]) // M + E + 1
    tiles = np.zeros((max_tiles, 4), np.int32)
    nt = _load().oracle_tile_schedule(_p(offsets), E, M, _p(tiles), max_tiles)
    return tiles[:nt].copy()


def gate_up(X, W1, W3, perm_token, offsets) -> np.ndarray:
    """H uint16 (bf16) [R,n]."""
    X = _c(X, np.uint16)
    W1 = _c(W1, np.uint16)
    W3 = _c(W3, np.uint16)
    perm_token = _c(perm_token, np.int32)
    offsets = _c(offsets, np.int32)
    E, d, n = W1.shape
    assert W3.shape == W1.shape and X.shape[1] == d and offsets.shape[0] == E + 1
    R = int(offsets[E])
    H = np.empty((R, n), np.uint16)
    _load().oracle_gate_up(_p(X), _p(W1), _p(W3), _p(perm_token), _p(offsets), E, d, n, _p(H))
    return H


def gate_up_pre(X, W1, W3, perm_token, offsets):
    """(A1, A3) float64 [R,n]: the unrounded pre-activations x W1[e], x W3[e]."""
    X = _c(X, np.uint16)
    W1 = _c(W1, np.uint16)
    W3 = _c(W3, np.uint16)
    perm_token = _c(perm_token, np.int32)
    offsets = _c(offsets, np.int32)
    E, d, n = W1.shape
    assert W3.shape == W1.shape and X.shape[1] == d and offsets.shape[0] == E + 1
    R = int(offsets[E])
    A1 = np.empty((R, n), np.float64)
    A3 = np.empty((R, n), np.float64)
    _load().oracle_gate_up_pre(_p(X), _p(W1), _p(W3), _p(perm_token), _p(offsets), E, d, n,
                               _p(A1), _p(A3))
    return A1, A3


def down(H, W2, topk_w, perm_slot, offsets) -> np.ndarray:
    """Z float64 [R,d] = w * (H W2[e])."""
    H = _c(H, np.uint16)
    W2 = _c(W2, np.uint16)
    topk_w = _c(topk_w, np.float32)
    perm_slot = _c(perm_slot, np.int32)
    offsets = _c(offsets, np.int32)
    E, n, d = W2.shape
    R = int(offsets[E])
    assert H.shape == (R, n)
    Z = np.empty((R, d), np.float64)
    _load().oracle_down(_p(H), _p(W2), _p(topk_w), _p(perm_slot), _p(offsets), E, n, d, _p(Z))
    return Z


def combine(Z: np.ndarray, row_of_slot: np.ndarray, K: int) -> np.ndarray:
    Z = _c(Z, np.float64)
    row_of_slot = _c(row_of_slot, np.int32)
    R, d = Z.shape
    T = row_of_slot.shape[0] // K
    Y = np.empty((T, d), np.uint16)
    _load().oracle_combine(_p(Z), _p(row_of_slot), T, K, d, _p(Y))
    return Y


def combine_bf16(Z: np.ndarray, row_of_slot: np.ndarray, K: int) -> np.ndarray:
    Z = _c(Z, np.uint16)
    row_of_slot = _c(row_of_slot, np.int32)
    R, d = Z.shape
    T = row_of_slot.shape[0] // K
    Y = np.empty((T, d), np.uint16)
    _load().oracle_combine_bf16(_p(Z), _p(row_of_slot), T, K, d, _p(Y))
    return Y


def forward(X, Wr, bias, W1, W3, W2, K: int, renorm: bool = True, M: int = 128) -> dict:
    """The whole layer through the grouped steps; returns every intermediate."""
    E = Wr.shape[1]
    L = router_logits(X, Wr, bias)
    idx, w = topk_softmax(L, K, renorm)
    counts = expert_counts(idx, E)
    offsets, perm_token, perm_slot, row_of_slot = permute(idx, E)
    tiles = tile_schedule(offsets, M)
    H = gate_up(X, W1, W3, perm_token, offsets)
    Z = down(H, W2, w, perm_slot, offsets)
    Y = combine(Z, row_of_slot, K)
    return dict(logits=L, idx=idx, w=w, counts=counts, offsets=offsets, perm_token=perm_token,
                perm_slot=perm_slot, row_of_slot=row_of_slot, tiles=tiles, H=H, Z=Z, Y=Y)


def forward_tokens(X, Wr, bias, W1, W3, W2, K: int, tokens, renorm: bool = True):
    """(Y rows [n,d] uint16, idx rows [n,K], w rows [n,K]) for the listed tokens,
    computed token by token from the definition."""
    X = _c(X, np.uint16)
    Wr = _c(Wr, np.float32)
    if bias is not None:
        bias = _c(bias, np.float32)
    W1 = _c(W1, np.uint16)
    W3 = _c(W3, np.uint16)
    W2 = _c(W2, np.uint16)
    tokens = _c(np.asarray(tokens, np.int64), np.int64)
    T, d = X.shape
    E, _, n = W1.shape
    nt = tokens.shape[0]
    assert tokens.min(initial=0) >= 0 and tokens.max(initial=0) < T
    Y = np.empty((nt, d), np.uint16)
    idx = np.empty((nt, K), np.int32)
    w = np.empty((nt, K), np.float32)
    _load().oracle_forward_tokens(_p(X), _p(Wr), _p(bias), _p(W1), _p(W3), _p(W2), T, d, E, K, n,
                                  int(bool(renorm)), _p(tokens), nt, _p(Y), _p(idx), _p(w))
    return Y, idx, w


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact float64 values of an array of bf16 bit patterns."""
    a = np.ascontiguousarray(a, np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------ token rounding

def rounding_capacity(T: int, E: int, K: int, M: int) -> int:
    """Most rows Token Rounding can produce: each expert moves by at most M//2
    rows and keeps at most T."""
    return min(T * E, T * K + E * (M // 2))


def token_rounding(L: np.ndarray, idx: np.ndarray, M: int, renorm: bool = True) -> dict:
    """Token Rounding of a top-K routing (see oracle_token_rounding in moe_oracle.h).
    Returns counts [E], offsets [E+1], perm_token [R'], row_map [T,E], row_w [R']."""
    L = _c(L, np.float32)
    idx = _c(idx, np.int32)
    T, E = L.shape
    K = idx.shape[1]
    assert idx.shape[0] == T and M >= 1
    cap = rounding_capacity(T, E, K, M)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm_token = np.empty(max(cap, 1), np.int32)
    row_map = np.empty((T, E), np.int32)
    row_w = np.empty(max(cap, 1), np.float32)
    R = _load().oracle_token_rounding(_p(L), _p(idx), T, E, K, M, int(bool(renorm)), cap,
                                      _p(counts), _p(offsets), _p(perm_token), _p(row_map),
                                      _p(row_w))
    if R < 0:
        raise RuntimeError("token rounding produced more rows than its capacity bound")
    return dict(counts=counts, offsets=offsets, perm_token=perm_token[:R].copy(),
                row_map=row_map, row_w=row_w[:R].copy())


def combine_rows(Z: np.ndarray, row_map: np.ndarray) -> np.ndarray:
    """Y uint16 (bf16) [T,d] from double Z rows and row_map [T,E]."""
    Z = _c(Z, np.float64)
    row_map = _c(row_map, np.int32)
    T, E = row_map.shape
    d = Z.shape[1]
    Y = np.empty((T, d), np.uint16)
    _load().oracle_combine_rows(_p(Z), _p(row_map), T, E, d, _p(Y))
    return Y


def combine_rows_bf16(Z: np.ndarray, row_map: np.ndarray) -> np.ndarray:
    Z = _c(Z, np.uint16)
    row_map = _c(row_map, np.int32)
    T, E = row_map.shape
    d = Z.shape[1]
    Y = np.empty((T, d), np.uint16)
    _load().oracle_combine_rows_bf16(_p(Z), _p(row_map), T, E, d, _p(Y))
    return Y


def forward_rounded(X, Wr, bias, W1, W3, W2, K: int, renorm: bool = True, M: int = 128) -> dict:
    """The layer under Token Rounding, through the grouped steps."""
    L = router_logits(X, Wr, bias)
    idx, w = topk_softmax(L, K, renorm)
    tr = token_rounding(L, idx, M, renorm)
    R = int(tr["offsets"][-1])
    H = gate_up(X, W1, W3, tr["perm_token"], tr["offsets"])
    # the weight of grouped row p is row_w[p]: an identity slot map
    Z = down(H, W2, tr["row_w"], np.arange(R, dtype=np.int32), tr["offsets"])
    Y = combine_rows(Z, tr["row_map"])
    tiles = tile_schedule(tr["offsets"], 128)
    return dict(logits=L, idx=idx, w=w, tiles=tiles, H=H, Z=Z, Y=Y, **tr)


def forward_assigned(X, W1, W3, W2, row_map, row_w, tokens) -> np.ndarray:
    """Y rows [n,d] (bf16 bits) for the listed tokens under a given assignment,
    computed token by token."""
    X = _c(X, np.uint16)
    W1 = _c(W1, np.uint16)
    W3 = _c(W3, np.uint16)
    W2 = _c(W2, np.uint16)
    row_map = _c(row_map, np.int32)
    row_w = _c(row_w, np.float32)
    tokens = _c(np.asarray(tokens, np.int64), np.int64)
    T, d = X.shape
    E, _, n = W1.shape
    assert row_map.shape == (T, E)
    nt = tokens.shape[0]
    Y = np.empty((nt, d), np.uint16)
    _load().oracle_forward_assigned(_p(X), _p(W1), _p(W3), _p(W2), T, d, E, n, _p(row_map),
                                    _p(row_w), _p(tokens), nt, _p(Y))
    return Y


def _f64_input(a):
    # bf16 tensors arrive as uint16 bit patterns and widen exactly; others as floats
    a = np.asarray(a)
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else _c(a, np.float64)


def forward_fixed(X, Wr, bias, W1, W3, W2, idx, renorm: bool = True) -> np.ndarray:
    """Y [T,d] float64 of the layer with the top-K choice idx [T,K] held fixed,
    in double and without the bf16 roundings of H and Y (the function the
    backward differentiates). X, W1, W3, W2 as bf16 bits (uint16) or floats."""
    X, Wr, W1, W3, W2 = (_f64_input(a) for a in (X, Wr, W1, W3, W2))
    bias = None if bias is None else _f64_input(bias)
    idx = _c(idx, np.int32)
    T, d = X.shape
    E, _, n = W1.shape
    K = idx.shape[1]
    Y = np.empty((T, d), np.float64)
    _load().oracle_forward_fixed(_p(X), _p(Wr), _p(bias), _p(W1), _p(W3), _p(W2), _p(idx),
                                 T, d, E, K, n, int(renorm), _p(Y))
    return Y


def backward_rows(X, Wr, bias, W1, W3, W2, idx, perm_slot, dY, renorm: bool = True) -> dict:
    """The backward's per-row quantities in grouped row order (perm_slot as
    permute() gives it): dS [T*K], dA1, dA3 [T*K,n], dXg [T*K,d] and per token
    dL [T,E], all float64 (see oracle_backward_rows in moe_oracle.c)."""
    X, Wr, W1, W3, W2 = (_f64_input(a) for a in (X, Wr, W1, W3, W2))
    bias = None if bias is None else _f64_input(bias)
    idx = _c(idx, np.int32)
    perm_slot = _c(perm_slot, np.int32)
    dY = _c(dY, np.float64)
    T, d = X.shape
    E, _, n = W1.shape
    K = idx.shape[1]
    R = T * K
    out = {"dS": np.empty(R), "dA1": np.empty((R, n)), "dA3": np.empty((R, n)),
           "dXg": np.empty((R, d)), "dL": np.empty((T, E))}
    _load().oracle_backward_rows(_p(X), _p(Wr), _p(bias), _p(W1), _p(W3), _p(W2), _p(idx),
                                 _p(perm_slot), _p(dY), T, d, E, K, n, int(renorm),
                                 _p(out["dS"]), _p(out["dA1"]), _p(out["dA3"]), _p(out["dXg"]),
                                 _p(out["dL"]))
    return out


def backward(X, Wr, bias, W1, W3, W2, idx, dY, renorm: bool = True) -> dict:
    """Gradient of sum(Y * dY) for Y = forward_fixed(...): dX [T,d], dWr [d,E],
    dbias [E], dW1, dW3 [E,d,n], dW2 [E,n,d], all float64."""
    X, Wr, W1, W3, W2 = (_f64_input(a) for a in (X, Wr, W1, W3, W2))
    bias = None if bias is None else _f64_input(bias)
    idx = _c(idx, np.int32)
    dY = _c(dY, np.float64)
    T, d = X.shape
    E, _, n = W1.shape
    K = idx.shape[1]
    out = {"dX": np.empty((T, d)), "dWr": np.empty((d, E)), "dbias": np.empty(E),
           "dW1": np.empty((E, d, n)), "dW3": np.empty((E, d, n)), "dW2": np.empty((E, n, d))}
    _load().oracle_backward(_p(X), _p(Wr), _p(bias), _p(W1), _p(W3), _p(W2), _p(idx), _p(dY),
                            T, d, E, K, n, int(renorm), _p(out["dX"]), _p(out["dWr"]),
                            _p(out["dbias"]), _p(out["dW1"]), _p(out["dW3"]), _p(out["dW2"]))
    return out
