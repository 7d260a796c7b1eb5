"""The C-ABI library on the host (no GPU needed): it loads, exports every entry
point include/moe.h declares, sizes workspaces and rejects bad arguments before
touching the device."""
import ctypes

import pytest
import torch

from top_routing_grouped_02_gb300 import _build, moe


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.lib()


def test_every_declared_symbol_is_exported(lib):
    declared = moe.header_symbols()
    assert len(declared) >= 15
    raw = ctypes.CDLL(moe.LIB_PATH)
    for name in declared:
        assert hasattr(raw, name), f"{name} declared in moe.h but not exported"
    assert set(declared) == set(moe._SIGS), "binding signatures out of sync with moe.h"


def test_abi_version_and_status_strings(lib):
    assert lib.moe_abi_version() == 101
    for code, name in moe.STATUS.items():
        assert lib.moe_status_string(code).decode() == name
    assert lib.moe_status_string(99).decode() == "MOE_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    T, d, E, K, n = 4096, 4096, 8, 2, 14336
    R = T * K
    b = moe.moe_workspace_bytes(T, d, E, K, n)
    # the gathered rows, H and Z dominate
    assert b >= 2 * R * (2 * d + n)
    assert b < 2 * R * (2 * d + n) + 64 * R + (1 << 20)
    assert b % 256 == 0
    assert moe.moe_workspace_bytes(0, d, E, K, n) == 0
    assert moe.moe_workspace_bytes(T, d, 300, K, n) == 0     # E > 256
    assert moe.moe_workspace_bytes(T, d, E, 9, n) == 0       # K > 8
    assert moe.moe_workspace_bytes(T, d, 4, 5, n) == 0       # K > E
    # grows with every dimension it should
    assert moe.moe_workspace_bytes(T, d, E, K, 2 * n) > b
    assert moe.moe_workspace_bytes(2 * T, d, E, K, n) > b


def test_forward_launch_counts(lib, monkeypatch):
    # kernels per forward: the router (1 for E <= 32 with E % 4 == 0: logits and
    # selection in one kernel; else 2), grouping 1 (3 above 65536 tokens; rounding
    # 3), combine 1, and
    # the expert GEMMs: two launches, a row gather more on CTA pairs (experts of
    # at least 8 row tiles on average), or one fused launch on request
    for var in ("MOE_GEMM_FUSED", "MOE_GEMM_CTA_PAIR"):
        monkeypatch.delenv(var, raising=False)
    assert moe.forward_launches(512, 256, 8, 2, 512) == 5            # tiny
    assert moe.forward_launches(16384, 1536, 128, 4, 256) == 6       # SonicMoE
    assert moe.forward_launches(16384, 1536, 128, 4, 256, True) == 8
    assert moe.forward_launches(8192, 7168, 256, 8, 2048) == 6       # DeepSeek-V3
    assert moe.forward_launches(4096, 4096, 8, 2, 14336) == 6        # Mixtral: CTA pairs
    assert moe.forward_launches(64, 256, 6, 2, 512) == 6             # E % 4 != 0: two router kernels
    assert moe.forward_launches(64, 33792, 8, 2, 512) == 6           # 33 blocks: two router kernels
    assert moe.forward_launches(70000, 256, 8, 2, 512) == 8          # T > 65536: three grouping kernels (and pairs)
    # (whether a fused launch's units fit its rounds depends on the device's SM
    # count, unknown here; these cases do not depend on it)
    assert moe.forward_launches(16384, 1536, 128, 4, 256, part="expert_mlp") == 2
    assert moe.forward_launches(4096, 4096, 8, 2, 14336, part="expert_mlp") == 3
    monkeypatch.setenv("MOE_GEMM_FUSED", "1")
    assert moe.forward_launches(512, 256, 8, 2, 512) == 4            # 80 units at most
    assert moe.forward_launches(512, 256, 8, 2, 512, part="expert_mlp") == 1
    assert moe.forward_launches(4096, 4096, 8, 2, 14336) == 6        # too wide to fuse
    assert moe.forward_launches(64, 256, 4, 1, 2176) == 5            # n > 2048
    monkeypatch.setenv("MOE_GEMM_FUSED", "0")
    assert moe.forward_launches(16384, 1536, 128, 4, 256) == 6
    with pytest.raises(ValueError):
        moe.forward_launches(512, 200, 8, 2, 512)
    assert lib.moe_forward_launches(512, 256, 8, 2, 512, 2) == -1


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails validation


@pytest.mark.parametrize("call,expect", [
    (lambda L: L.moe_route(None, FAKE, None, 16, 64, 8, 2, 1, FAKE, FAKE, FAKE, FAKE, None), 1),
    (lambda L: L.moe_route(FAKE, FAKE, None, 16, 64, 8, 2, 2, FAKE, FAKE, FAKE, FAKE, None), 1),
    (lambda L: L.moe_route(FAKE, FAKE, None, 16, 60, 8, 2, 1, FAKE, FAKE, FAKE, FAKE, None), 2),
    (lambda L: L.moe_route(FAKE, FAKE, None, 16, 64, 300, 2, 1, FAKE, FAKE, FAKE, FAKE, None), 2),
    (lambda L: L.moe_route(FAKE, FAKE, None, 0, 64, 8, 2, 1, FAKE, FAKE, FAKE, FAKE, None), 1),
    (lambda L: L.moe_route(ctypes.c_void_p((1 << 20) + 2), FAKE, None, 16, 64, 8, 2, 1, FAKE,
                           FAKE, FAKE, FAKE, None), 1),
    (lambda L: L.moe_route(FAKE, FAKE, None, 16, 64, 8, 2, 1, None, FAKE, FAKE, FAKE, None), 1),
    (lambda L: L.moe_route_logits(FAKE, 16, 8, 9, 1, FAKE, FAKE, FAKE, None), 2),
    (lambda L: L.moe_permute(FAKE, None, 16, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8,
                             None), 3),
    (lambda L: L.moe_permute(None, None, 16, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             1 << 30, None), 1),
    (lambda L: L.moe_gemm_gate_up(FAKE, FAKE, FAKE, FAKE, FAKE, 16, 200, 8, 2, 128, FAKE, FAKE,
                                  1 << 30, None), 2),
    (lambda L: L.moe_gemm_gate_up(FAKE, FAKE, FAKE, FAKE, FAKE, 16, 256, 8, 2, 100, FAKE, FAKE,
                                  1 << 30, None), 2),
    (lambda L: L.moe_gemm_down(FAKE, FAKE, FAKE, FAKE, FAKE, 16, 256, 8, 2, 128, FAKE, FAKE, 16,
                               None), 3),
    (lambda L: L.moe_combine(FAKE, FAKE, 16, 9, 64, FAKE, None), 2),
    (lambda L: L.moe_forward(FAKE, FAKE, None, FAKE, FAKE, FAKE, 16, 256, 8, 2, 128, 1, FAKE, None,
                             None, FAKE, 1024, None), 3),
    (lambda L: L.moe_forward(FAKE, FAKE, None, FAKE, FAKE, FAKE, 16, 256, 8, 2, 128, 1, None, None,
                             None, FAKE, 1 << 30, None), 1),
    (lambda L: L.moe_workspace_init(None, 64, None), 1),
    (lambda L: L.moe_sync_check(None, None, None), 1),
    # both expert GEMMs (two launches or one fused): null W2, unsupported d,
    # unaligned Z, workspace too small for the counter words
    (lambda L: L.moe_expert_mlp(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 16, 256, 8, 2, 128,
                                FAKE, FAKE, FAKE, 1 << 30, None), 1),
    (lambda L: L.moe_expert_mlp(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 200, 8, 2, 128,
                                FAKE, FAKE, FAKE, 1 << 30, None), 2),
    (lambda L: L.moe_expert_mlp(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 256, 8, 2, 128,
                                FAKE, ctypes.c_void_p((1 << 20) + 8), FAKE, 1 << 30, None), 1),
    (lambda L: L.moe_expert_mlp(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 256, 8, 2, 128,
                                FAKE, FAKE, FAKE, 4096, None), 3),
    # Token Rounding entry points
    (lambda L: L.moe_forward_rounded(FAKE, FAKE, None, FAKE, FAKE, FAKE, 16, 256, 8, 2, 128, 2,
                                     FAKE, None, FAKE, 1 << 30, None), 1),
    (lambda L: L.moe_forward_rounded(FAKE, FAKE, None, FAKE, FAKE, FAKE, 16, 256, 8, 2, 128, 1,
                                     FAKE, None, FAKE, 1024, None), 3),
    (lambda L: L.moe_combine_rows(None, FAKE, 16, 8, 64, 32, FAKE, None), 1),
    (lambda L: L.moe_combine_rows(FAKE, FAKE, 16, 8, 64, -1, FAKE, None), 1),
])
def test_bad_arguments_are_rejected_on_the_host(lib, call, expect):
    assert call(lib) == expect


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_a_device_reports_cuda_error(lib):
    st = lib.moe_route_logits(FAKE, 16, 8, 2, 1, FAKE, FAKE, FAKE, None)
    assert st == 5  # MOE_ERR_CUDA: no device to check the architecture of


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(moe, "_lib", None)
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        moe.lib()
