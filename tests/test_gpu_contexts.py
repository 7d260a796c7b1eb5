"""Kernels with large dynamic shared memory in several CUDA contexts.

A kernel's dynamic shared-memory limit is a property of the context it is set
in. The library raises it once per (kernel, context); a cache keyed by device
alone would skip a second context on the same device, and the launch there
would fail. The child process makes the grouped GEMM (217 KB of shared memory
per CTA) run in a created context, in the primary context, and in a new context
created after the first one was destroyed. It checks each result against the
oracle and that all three agree bit for bit.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

_CHILD = r"""
import ctypes, math, sys
import numpy as np
import torch
sys.path.insert(0, "tests")
import oracle
from gpu_common import check_hz
from top_routing_grouped_02_gb300 import moe, synth

cu = ctypes.CDLL("libcuda.so.1")
def ok(r, what):
    if r != 0:
        raise SystemExit(f"{what} failed: CUresult {r}")
ok(cu.cuInit(0), "cuInit")
dev = ctypes.c_int(0)
ok(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")

def create_context():
    ctx = ctypes.c_void_p()
    f = getattr(cu, "cuCtxCreate_v4", None)
    if f is not None:
        ok(f(ctypes.byref(ctx), None, 0, dev), "cuCtxCreate_v4")
    else:
        ok(cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, dev), "cuCtxCreate_v2")
    return ctx

T, d, E, K, n = 300, 256, 8, 2, 256
X = synth.bf16_bits(synth.normal("X", (T, d), 1.0, torch.bfloat16, "cpu"))
W1 = synth.bf16_bits(synth.normal("W1", (E, d, n), 1.0 / math.sqrt(d), torch.bfloat16, "cpu"))
W3 = synth.bf16_bits(synth.normal("W3", (E, d, n), 1.0 / math.sqrt(d), torch.bfloat16, "cpu"))
rng = np.random.default_rng(5)
idx = np.argsort(-rng.gumbel(size=(T, E)), axis=1, kind="stable")[:, :K].astype(np.int32)
off, pt, ps, ros = oracle.permute(idx, E)
R = T * K
H_ref = oracle.gate_up(X, W1, W3, pt, off)
L = moe.lib()
ws_bytes = int(L.moe_workspace_bytes(T, d, E, K, n))

def run_here(what):
    host = {"X": X, "W1": W1, "W3": W3, "pt": pt, "off": off}
    d_ = {}
    for k, a in host.items():
        a = np.ascontiguousarray(a)
        ptr = ctypes.c_uint64()
        ok(cu.cuMemAlloc_v2(ctypes.byref(ptr), ctypes.c_size_t(a.nbytes)), "cuMemAlloc")
        ok(cu.cuMemcpyHtoD_v2(ptr, a.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(a.nbytes)),
           "cuMemcpyHtoD")
        d_[k] = ptr.value
    for k, nbytes in (("H", R * n * 2), ("ws", ws_bytes)):
        ptr = ctypes.c_uint64()
        ok(cu.cuMemAlloc_v2(ctypes.byref(ptr), ctypes.c_size_t(nbytes)), "cuMemAlloc")
        d_[k] = ptr.value
    v = lambda k: ctypes.c_void_p(d_[k])
    st = L.moe_workspace_init(v("ws"), ws_bytes, None)
    if st != 0:
        raise SystemExit(f"{what}: moe_workspace_init returned {st}")
    st = L.moe_gemm_gate_up(v("X"), v("W1"), v("W3"), v("pt"), v("off"), T, d, E, K, n, v("H"),
                            v("ws"), ws_bytes, None)
    if st != 0:
        raise SystemExit(f"{what}: moe_gemm_gate_up returned {st}")
    ok(cu.cuCtxSynchronize(), "cuCtxSynchronize")
    H = np.empty((R, n), np.uint16)
    ok(cu.cuMemcpyDtoH_v2(H.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(d_["H"]),
                          ctypes.c_size_t(H.nbytes)), "cuMemcpyDtoH")
    for p in d_.values():
        ok(cu.cuMemFree_v2(ctypes.c_uint64(p)), "cuMemFree")
    check_hz(H, H_ref, "H")
    return H

a = create_context()                                   # current on this thread
Ha = run_here("created context")
popped = ctypes.c_void_p()
ok(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent")
prim = ctypes.c_void_p()
ok(cu.cuDevicePrimaryCtxRetain(ctypes.byref(prim), dev), "cuDevicePrimaryCtxRetain")
ok(cu.cuCtxPushCurrent_v2(prim), "cuCtxPushCurrent")
Hp = run_here("primary context")
ok(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent")
ok(cu.cuCtxDestroy_v2(a), "cuCtxDestroy")
b = create_context()
Hb = run_here("new context after the first was destroyed")
ok(cu.cuCtxDestroy_v2(b), "cuCtxDestroy")
ok(cu.cuDevicePrimaryCtxRelease_v2(dev), "cuDevicePrimaryCtxRelease")
assert np.array_equal(Ha, Hp) and np.array_equal(Ha, Hb)
print("CONTEXTS OK")
"""


def test_grouped_gemm_in_several_contexts():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _CHILD], cwd=root, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and "CONTEXTS OK" in r.stdout, (r.stdout[-2000:], r.stderr[-2000:])
