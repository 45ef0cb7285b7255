"""Host-side checks of the C ABI: the library builds, loads and exports every
function the header declares, and rejects bad sizes before touching a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe_b300.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    from mixture_experts_layer_98_b300 import build
    build.build()
    import mixture_experts_layer_98_b300 as m
    return m.lib()


def test_header_declares_the_forward():
    names = declared_functions()
    assert "moe_forward" in names and "moe_forward_ws" in names
    assert len(names) >= 10


def test_every_declared_symbol_is_exported(L):
    import mixture_experts_layer_98_b300 as m
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in moe_b300.h but not exported"
    assert set(m.EXPORTS) == set(declared_functions())


def test_strerror(L):
    for s in range(7):
        assert L.moe_strerror(s)
    assert b"unknown" in L.moe_strerror(99)


def test_set_expert_path(L):
    assert L.moe_set_expert_path(8) == -1
    assert L.moe_set_expert_path(7) == -1
    assert L.moe_set_expert_path(-1) == -1
    prev = L.moe_set_expert_path(1)
    assert L.moe_set_expert_path(4) == 1      # MOE_PATH_TCGEN05_PAIR
    assert L.moe_set_expert_path(6) == 4      # MOE_PATH_WARP_MMA
    assert L.moe_set_expert_path(prev) == 6


def test_workspace_bytes(L):
    ws = L.moe_workspace_bytes
    assert ws(4096, 2048, 128, 8, 768) > 4096 * 8 * (2048 * 2 + 768) * 2
    assert ws(-1, 2048, 128, 8, 768) == 0
    assert ws(16, 100, 8, 2, 256) == 0        # H not a multiple of 64
    assert ws(16, 128, 8, 9, 256) == 0        # K > E
    assert ws(16, 128, 300, 2, 256) == 0      # E > 256
    assert ws(16, 128, 64, 17, 256) == 0      # K > 16
    assert ws(16, 65600, 8, 2, 256) == 0      # H > 65536
    assert ws(4096, 4096, 8, 2, 14336) > 0    # few big experts (I = 14336)
    assert ws(1, 128, 8, 2, 256) <= ws(2, 128, 8, 2, 256)


def test_noalloc_scratch_limit(L):
    # moe_forward_noalloc's 32 MiB scratch holds the workspace of every batch up
    # to T = 212 on the H=4096, E=128, K=8, I=1536 layer (the limit its header
    # states) and not T = 213.  It takes no capacity, so it needs
    # moe_workspace_bytes less the T·K·H·2 bytes of fp32 expert outputs only a
    # capacity forward keeps.  The split-K plans of the decode kernels size
    # part of the workspace, so a plan change that grows it shows up here.
    def need(T):
        return L.moe_workspace_bytes(T, 4096, 128, 8, 1536) - T * 8 * 4096 * 2
    scratch = 32 << 20
    assert max(need(T) for T in range(1, 213)) <= scratch
    assert need(213) > scratch


def test_capacity_workspace_keeps_fp32_expert_outputs(L):
    # the fp32 expert outputs of a capacity forward take twice the bf16 bytes
    # at the end of the workspace: moe_workspace_bytes covers them
    for T, H, E, K, I in [(1, 128, 8, 2, 256), (300, 256, 16, 4, 128), (4096, 2048, 128, 8, 768)]:
        ws = L.moe_workspace_bytes(T, H, E, K, I)
        assert ws >= T * K * (2 * H * 2 + I * 2) + T * K * H * 2


@pytest.mark.parametrize("T,H,E,K,I", [(-1, 128, 8, 2, 256), (4, 96, 8, 2, 256),
                                       (4, 128, 0, 1, 256), (4, 128, 8, 0, 256),
                                       (4, 128, 8, 2, 100), (4, 128, 4, 5, 256)])
def test_forward_rejects_bad_sizes_before_any_work(L, T, H, E, K, I):
    z = ctypes.c_void_p(0)
    rc = L.moe_forward(z, T, H, z, z, z, z, E, K, I, 1, z, z, z, z, z, z)
    assert rc == 1  # MOE_ERR_INVALID_ARG, returned before any CUDA call


def test_forward_rejects_null_weights(L):
    z = ctypes.c_void_p(0)
    assert L.moe_forward(z, 0, 128, z, z, z, z, 8, 2, 256, 1, z, z, z, z, z, z) == 1


def test_forward_rejects_misaligned_pointers(L):
    z = ctypes.c_void_p(0)
    a = ctypes.c_void_p(0x1000)
    bad = ctypes.c_void_p(0x1002)
    assert L.moe_forward(a, 4, 128, a, bad, a, a, 8, 2, 256, 1, a, z, z, z, z, z) == 2


def test_python_binding_fails_loudly_without_library(monkeypatch):
    import mixture_experts_layer_98_b300.binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", "/nonexistent/libmoe_b300.so")
    with pytest.raises(RuntimeError, match="not built"):
        b.lib()


def test_packed_sizes_and_early_rejects(L):
    # 3·E·I·H·2 bytes for packable shapes (I % 128 == 0, H % 256 == 0), else 0
    assert L.moe_packed_experts_bytes(2048, 128, 768) == 3 * 128 * 768 * 2048 * 2
    assert L.moe_packed_experts_bytes(4096, 128, 1536) == 3 * 128 * 1536 * 4096 * 2
    assert L.moe_packed_experts_bytes(2048, 128, 320) == 0     # I % 128 != 0
    assert L.moe_packed_experts_bytes(1152, 8, 256) == 0       # H % 256 != 0
    assert L.moe_packed_experts_bytes(2048, 0, 768) == 0
    assert L.moe_packed_experts_bytes(2048, 300, 768) == 0
    z = ctypes.c_void_p(0)
    # shape checks come before any pointer or device check
    assert L.moe_pack_experts(z, z, z, 1152, 8, 256, z, z) == 1
    assert L.moe_forward_packed(z, 4, 1152, z, z, 8, 2, 256, 1, z, z, z, z, z, z, 0, z) == 1
    assert L.moe_forward_host_packed(z, 4, 1152, z, z, 8, 2, 256, 1, z, z, z, z, z, z) == 1


def test_q4_experts_bytes(L):
    # per matrix: codes E*R*C/2 bytes + scales E*R*(C/128)*4 bytes
    def mat(R, C, E):
        return E * R * C // 2 + E * R * (C // 128) * 4
    H, E, I = 2048, 128, 768
    assert L.moe_q4_experts_bytes(H, E, I) == 2 * mat(I, H, E) + mat(H, I, E)
    assert L.moe_q4_experts_bytes(128, 8, 256) == 0    # H % 256 != 0
    assert L.moe_q4_experts_bytes(256, 8, 192) == 0    # I % 128 != 0
    assert L.moe_q4_experts_bytes(256, 0, 128) == 0
    assert L.moe_quantize_experts_q4(None, None, None, 256, 8, 128, None, None) != 0
    assert L.moe_forward_q4(None, 1, 256, None, None, 8, 2, 128, 1, None, None, None, None,
                            None, None, 0, None) != 0


def test_q4_argument_checks(L):
    # every check below runs before the library touches a device (no GPU here);
    # the pointers are never dereferenced
    from mixture_experts_layer_98_b300.binding import (MOE_ERR_ALIGNMENT, MOE_ERR_INVALID_ARG,
                                                        _Options)
    import ctypes
    odd = ctypes.c_void_p(0x1008)    # 8-byte aligned only
    ok = ctypes.c_void_p(0x2000)
    # quantise / dequantise: unsupported shape, NULL, misaligned
    assert L.moe_quantize_experts_q4(ok, ok, ok, 128, 8, 256, ok, None) == MOE_ERR_INVALID_ARG
    assert L.moe_quantize_experts_q4(ok, ok, None, 256, 8, 128, ok, None) == MOE_ERR_INVALID_ARG
    assert L.moe_quantize_experts_q4(ok, ok, ok, 256, 8, 128, odd, None) == MOE_ERR_ALIGNMENT
    assert L.moe_dequantize_experts_q4(odd, 256, 8, 128, ok, ok, ok, None) == MOE_ERR_ALIGNMENT
    assert L.moe_dequantize_experts_q4(ok, 256, 8, 192, ok, ok, ok, None) == MOE_ERR_INVALID_ARG
    # forward: unsupported shape, misaligned buffer
    fwd = (ok, 4, 256, ok)
    rest = (ok, ok, ok, ok, ok, ok, 0, None)
    assert L.moe_forward_q4(*fwd, ok, 8, 2, 192, 1, *rest) == MOE_ERR_INVALID_ARG
    assert L.moe_forward_q4(*fwd, odd, 8, 2, 128, 1, *rest) == MOE_ERR_ALIGNMENT
    # options: 4-bit and packed weights together, 4-bit with an unsupported shape
    both = _Options(None, 0x2000, None, 0, 0.0, 0x4000)
    assert L.moe_forward_opts(*fwd, None, None, None, 8, 2, 128, 1, ok, ok, ok, ok, ok,
                              ctypes.byref(both), None) == MOE_ERR_INVALID_ARG
    bad_shape = _Options(None, None, None, 0, 0.0, 0x4000)
    assert L.moe_forward_opts(*fwd, None, None, None, 8, 2, 192, 1, ok, ok, ok, ok, ok,
                              ctypes.byref(bad_shape), None) == MOE_ERR_INVALID_ARG
    # host-buffer entry: unsupported shape, misaligned buffer
    assert L.moe_forward_host_q4(*fwd, ok, 8, 2, 192, 1, ok, ok, ok, ok, ok,
                                 None) == MOE_ERR_INVALID_ARG
    assert L.moe_forward_host_q4(*fwd, odd, 8, 2, 128, 1, ok, ok, ok, ok, ok,
                                 None) == MOE_ERR_ALIGNMENT
    misaligned = _Options(None, None, None, 0, 0.0, 0x4008)
    assert L.moe_forward_opts(*fwd, None, None, None, 8, 2, 128, 1, ok, ok, ok, ok, ok,
                              ctypes.byref(misaligned), None) == MOE_ERR_ALIGNMENT
