"""The C ABI on the host, without a GPU: the library builds for sm_103a,
loads, exports every function include/moe_w4a16.h declares, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

import w4a16_group_quantized_moe_gb300 as moe
from w4a16_group_quantized_moe_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe_w4a16.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return moe.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(moe.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # nothing but the C entry points is visible
    out = os.popen(f"nm -D --defined-only {moe.LIB_PATH}").read()
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert exported == declared_functions()


def test_status_strings(lib):
    for s in range(6):
        assert lib.moe_status_string(s)
    assert lib.moe_status_string(99) == b"unknown status"
    assert lib.moe_abi_version() == 1


def test_workspace_bytes(lib):
    # control block + per-block counters + fp32 per-pair projections
    n = lib.moe_workspace_bytes(8, 512, 10, 2560, 640)
    assert n >= 256 + 320 * 4 + 80 * 2560 * 4
    assert n % 256 == 0
    assert lib.moe_workspace_bytes(8, 512, 10, 2560, 641) == 0     # I % 32
    assert lib.moe_workspace_bytes(8, 512, 513, 2560, 640) == 0    # k > E
    assert lib.moe_workspace_bytes(8, 2048, 10, 2560, 640) == 0    # E > 1024
    assert lib.moe_workspace_bytes(0, 512, 10, 2560, 640) > 0


@pytest.mark.parametrize("T,E,k,status", [(-1, 16, 2, moe.MOE_ERR_INVALID_ARG),
                                          (4, 16, 17, moe.MOE_ERR_INVALID_ARG),
                                          (4, 0, 1, moe.MOE_ERR_INVALID_ARG),
                                          (4, 2048, 2, moe.MOE_ERR_UNSUPPORTED),
                                          (4, 64, 40, moe.MOE_ERR_UNSUPPORTED)])
def test_route_rejects_bad_sizes(lib, T, E, k, status):
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    assert lib.moe_topk_route(p, T, E, k, p, p, None) == status


def test_null_and_misaligned_pointers_rejected(lib):
    buf = (ctypes.c_uint8 * 256)()
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    assert lib.moe_topk_route(None, 4, 16, 2, p, p, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_topk_route(p + 4, 4, 16, 2, p, p, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_align_offsets(p, 4, 16, 2, p, p, None, p, None, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_get_device_error(None, 256, None, None) == moe.MOE_ERR_INVALID_ARG


def test_gate_up_and_down_validate_before_launch(lib):
    buf = (ctypes.c_uint8 * 512)()
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    args = lambda gs, H, I, ws, wsb: (p, p, p, p, gs, p, p, p, p, 4, 16, 2, H, I, p, ws, wsb, None)
    need = lib.moe_workspace_bytes(4, 16, 2, 256, 64)
    f = lib.moe_w4a16_gate_up_silu
    assert f(*args(32, 250, 64, p, need)) == moe.MOE_ERR_INVALID_ARG      # H % 32
    assert f(*args(16, 256, 64, p, need)) == moe.MOE_ERR_UNSUPPORTED      # group size
    assert f(*args(0, 256, 64, p, need)) == moe.MOE_ERR_INVALID_ARG
    assert f(*args(32, 256, 64, None, need)) == moe.MOE_ERR_WORKSPACE
    assert f(*args(32, 256, 64, p, need - 1)) == moe.MOE_ERR_WORKSPACE
    g = lib.moe_w4a16_down_combine
    dargs = lambda ws, wsb: (p, p, p, p, 32, p, p, p, p, p, 4, 16, 2, 256, 64, p, ws, wsb, None)
    assert g(*dargs(p, need - 256)) == moe.MOE_ERR_WORKSPACE
    assert g(p, p, p, p, 32, p, p, p, p, None, 4, 16, 2, 256, 64, p, p, need,
             None) == moe.MOE_ERR_INVALID_ARG                                  # null topk_w


def test_new_calls_validate_before_the_device(lib):
    """Forced-family, NVFP4, router and AWQ-import calls reject malformed
    arguments on the host (no device is touched: there is none here)."""
    buf = (ctypes.c_uint8 * 512)()
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    need = lib.moe_workspace_bytes(4, 16, 2, 256, 64)
    # _ex: an unknown family, and the usual checks
    gu = lambda path, H=256: lib.moe_w4a16_gate_up_silu_ex(p, p, p, p, 32, p, p, p, p, 4, 16, 2, H, 64, p, p,
                                                          need, path, None)
    assert gu(7) == moe.MOE_ERR_INVALID_ARG and gu(-1) == moe.MOE_ERR_INVALID_ARG
    assert gu(moe.MOE_PATH_DECODE, H=250) == moe.MOE_ERR_INVALID_ARG
    dn = lambda path: lib.moe_w4a16_down_combine_ex(p, p, p, p, 32, p, p, p, p, p, 4, 16, 2, 256, 64, p, p, need,
                                                    path, None)
    assert dn(4) == moe.MOE_ERR_INVALID_ARG
    # NVFP4: null scale pointer, short workspace, bad sizes
    assert lib.moe_nvfp4_gate_up_silu(p, p, None, p, p, p, p, p, 4, 16, 2, 256, 64, p, p, need,
                                      None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_nvfp4_down_combine(p, p, p, p, p, p, p, p, p, 4, 16, 2, 256, 64, p, p, need - 256,
                                      None) == moe.MOE_ERR_WORKSPACE
    assert lib.moe_nvfp4_moe_layer(p, p, p, p, p, p, p, p, 4, 16, 3, 256, 60, p, p, p, p, 1 << 20,
                                   None) == moe.MOE_ERR_INVALID_ARG                     # I % 32
    # router: H % 32, misaligned x, no workspace for the fused call
    assert lib.moe_router_logits(p, p, 4, 16, 250, p, None, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_router_logits(p + 2, p, 4, 16, 256, p, None, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_router_route_align(p, p, 4, 16, 2, 256, p, p, p, p, p, p, p, None, 0,
                                      None) == moe.MOE_ERR_WORKSPACE
    assert lib.moe_router_route_align(p, p, 4, 2048, 2, 256, p, p, p, p, p, p, p, p, 512,
                                      None) == moe.MOE_ERR_UNSUPPORTED                  # E > 1024
    # launch floor: the layer's size checks
    assert lib.moe_decode_layer_floor(1, 0, 10, 2560, 640, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_layer_floor(1, 512, 10, 2500, 640, None) == moe.MOE_ERR_INVALID_ARG
    # AWQ import: misplaced rows, K % 32, group size, overflowing destination
    imp = lambda E, K, N, g, Nd, r0: lib.moe_awq_import(p, p, p, E, K, N, g, p, p, p, Nd, r0, None)
    assert imp(1, 64, 16, 32, 32, 4) == moe.MOE_ERR_INVALID_ARG
    assert imp(1, 48, 16, 32, 32, 0) == moe.MOE_ERR_INVALID_ARG
    assert imp(1, 64, 16, 128, 32, 0) == moe.MOE_ERR_UNSUPPORTED
    assert imp(1, 64, 16, 32, 16, 8) == moe.MOE_ERR_INVALID_ARG
    assert imp(2048, 64, 16, 32, 16, 0) == moe.MOE_ERR_UNSUPPORTED


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.dirname(moe.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "moe_oracle" not in text, f
