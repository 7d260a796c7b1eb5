"""The allocation-free grouping call (moe_permute_noalloc) against moe_permute.

moe_permute_noalloc serves callers that may not allocate device memory (for
example a plugin inside an inference engine that owns all device memory, or a
serving loop whose memory was planned at start-up): it keeps its scratch in an
array built into libmoe.so instead of a caller workspace. This file runs last
(named so that pytest collects it after the other test files) and passes both
on its own in a fresh process and after the rest of the suite.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from top_routing_grouped_02_gb300 import moe

pytestmark = pytest.mark.gpu

KEYS = ("offsets", "perm_token", "perm_slot", "row_of_slot", "tiles", "num_tiles")


def _routing(T, E, K, skew, seed):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** (-skew)
    g = rng.gumbel(size=(T, E)) + np.log(p / p.sum())
    return torch.from_numpy(np.argsort(-g, axis=1, kind="stable")[:, :K].astype(np.int32)).cuda()


def _same(got, ref, what):
    """Every output the grouping defines: offsets, the rows in use (up to
    offsets[E]; slots without a row leave the rest unwritten), row_of_slot and
    the tile list."""
    used = int(ref["offsets"][-1].item())
    assert torch.equal(got["offsets"], ref["offsets"]), f"offsets differ ({what})"
    for k in ("perm_token", "perm_slot"):
        assert torch.equal(got[k][:used], ref[k][:used]), f"{k} differs ({what})"
    assert torch.equal(got["row_of_slot"], ref["row_of_slot"]), f"row_of_slot differs ({what})"
    nt = int(ref["num_tiles"].item())
    assert torch.equal(got["num_tiles"], ref["num_tiles"]), f"num_tiles differs ({what})"
    assert torch.equal(got["tiles"][:nt], ref["tiles"][:nt]), f"tiles differ ({what})"


def test_noalloc_matches_workspace_call_on_two_calls_in_a_row():
    # different shapes back to back: a call must not see the previous one's scratch
    cases = [(8192, 256, 8, 1.1, 1), (4096, 8, 2, 0.0, 2), (8192, 256, 8, 1.1, 3)]
    for T, E, K, skew, seed in cases:
        idx = _routing(T, E, K, skew, seed)
        counts = torch.bincount(idx.view(-1).long(), minlength=E).to(torch.int32)
        ref = moe.moe_permute(idx, E, counts=counts)
        got = moe.moe_permute_noalloc(idx, E, counts=counts)
        torch.cuda.synchronize()
        for k in KEYS:
            assert torch.equal(got[k], ref[k]), f"{k} differs (T={T}, E={E}, K={K})"


def test_noalloc_without_counts():
    idx = _routing(3000, 16, 4, 0.7, 4)
    ref = moe.moe_permute(idx, 16)
    got = moe.moe_permute_noalloc(idx, 16)
    torch.cuda.synchronize()
    for k in KEYS:
        assert torch.equal(got[k], ref[k]), f"{k} differs"


def test_noalloc_bad_expert_then_good_call():
    # an index outside [0, E) and a repeated expert get no row (row_of_slot -1),
    # as with moe_permute; the next, valid call must match moe_permute exactly,
    # which shows that the control words the bad call left in the shared array
    # were cleared
    T, E, K = 1000, 8, 2
    idx = _routing(T, E, K, 0.0, 5)
    bad = idx.clone()
    bad[10, 1] = E + 3
    bad[20, 0] = -1
    bad[30, 1] = bad[30, 0]
    ref = moe.moe_permute(bad, E)
    got = moe.moe_permute_noalloc(bad, E)
    torch.cuda.synchronize()
    ros = got["row_of_slot"].cpu().numpy()
    assert ros[10 * K + 1] == -1 and ros[20 * K] == -1 and ros[30 * K + 1] == -1
    _same(got, ref, "bad indices")
    good = _routing(T, E, K, 0.3, 6)
    counts = torch.bincount(good.view(-1).long(), minlength=E).to(torch.int32)
    ref2 = moe.moe_permute(good, E, counts=counts)
    got2 = moe.moe_permute_noalloc(good, E, counts=counts)
    torch.cuda.synchronize()
    for k in KEYS:
        assert torch.equal(got2[k], ref2[k]), f"{k} differs after a bad call"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    T, E, K = 200000, 8, 8  # 1.6M slots: far beyond the 4 MiB scratch
    idx = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_permute_noalloc(idx, E)
    assert e.value.status == 2  # MOE_ERR_UNSUPPORTED_SHAPE, nothing enqueued


# Runs in a fresh process with no torch CUDA use: CUDA contexts made through the
# driver API (ctypes on libcuda), device buffers allocated in each, and
# moe_permute_noalloc called straight through the C ABI in each context. The
# built-in scratch has a separate address in every context, so the call must
# look it up again in a context it has not seen, including a new context made
# after the first was destroyed (its handle may be reused; its id is not).
_CONTEXTS_CHILD = r"""
import ctypes, sys
import numpy as np
import oracle
from top_routing_grouped_02_gb300 import moe

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

T, E, K = 1000, 16, 2
R = T * K
rng = np.random.default_rng(11)
idx = np.argsort(-rng.gumbel(size=(T, E)), axis=1, kind="stable")[:, :K].astype(np.int32)
off_r, pt_r, ps_r, ros_r = oracle.permute(idx, E)
tiles_r = oracle.tile_schedule(off_r, moe.TILE_M)
L = moe.lib()

def run_here(what):
    sizes = {"idx": R * 4, "off": (E + 1) * 4, "pt": R * 4, "ps": R * 4, "ros": R * 4,
             "tiles": (R // moe.TILE_M + E) * 16, "nt": 4}
    d = {}
    for k, n in sizes.items():
        ptr = ctypes.c_uint64()
        ok(cu.cuMemAlloc_v2(ctypes.byref(ptr), n), "cuMemAlloc")
        d[k] = ptr.value
    ok(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(d["idx"]), idx.ctypes.data_as(ctypes.c_void_p), R * 4),
       "cuMemcpyHtoD")
    v = lambda k: ctypes.c_void_p(d[k])
    st = L.moe_permute_noalloc(v("idx"), None, T, E, K, v("off"), v("pt"), v("ps"), v("ros"),
                               v("tiles"), v("nt"), None)
    if st != 0:
        raise SystemExit(f"{what}: moe_permute_noalloc returned {st}")
    ok(cu.cuCtxSynchronize(), "cuCtxSynchronize")
    def back(k, n):
        a = np.empty(n, np.int32)
        ok(cu.cuMemcpyDtoH_v2(a.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(d[k]), n * 4),
           "cuMemcpyDtoH")
        return a
    nt = int(back("nt", 1)[0])
    assert np.array_equal(back("off", E + 1), off_r), what
    assert np.array_equal(back("pt", R), pt_r), what
    assert np.array_equal(back("ps", R), ps_r), what
    assert np.array_equal(back("ros", R), ros_r), what
    assert nt == len(tiles_r), what
    assert np.array_equal(back("tiles", nt * 4).reshape(nt, 4), tiles_r), what
    for p in d.values():
        ok(cu.cuMemFree_v2(ctypes.c_uint64(p)), "cuMemFree")

a = create_context()                                   # current on this thread
run_here("created context")
popped = ctypes.c_void_p()
ok(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent")
prim = ctypes.c_void_p()
ok(cu.cuDevicePrimaryCtxRetain(ctypes.byref(prim), dev), "cuDevicePrimaryCtxRetain")
ok(cu.cuCtxPushCurrent_v2(prim), "cuCtxPushCurrent")
run_here("primary context")
ok(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent")
ok(cu.cuCtxPushCurrent_v2(a), "cuCtxPushCurrent")
run_here("created context again")
ok(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent")
ok(cu.cuCtxDestroy_v2(a), "cuCtxDestroy")
b = create_context()
run_here("new context after the first was destroyed")
ok(cu.cuCtxDestroy_v2(b), "cuCtxDestroy")
ok(cu.cuDevicePrimaryCtxRelease_v2(dev), "cuDevicePrimaryCtxRelease")
print("CONTEXTS OK")
"""


def test_noalloc_in_several_contexts():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _CONTEXTS_CHILD], cwd=root, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "CONTEXTS OK" in r.stdout, (r.stdout[-2000:], r.stderr[-2000:])
