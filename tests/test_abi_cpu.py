"""The C-ABI library without a GPU: it builds, loads, exports every entry
point include/moe.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import nvfp4_routed_expert_gb300 as nv
from nvfp4_routed_expert_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "moe.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return nv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for required in ("moe_layer_create", "moe_quantize_act", "moe_forward", "moe_destroy",
                     "moe_workspace_bytes", "moe_layer_status", "moe_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(nv.EXPORTED)


def test_status_strings(lib):
    for code, name in ((0, "MOE_OK"), (1, "MOE_ERR_INVALID_ARGUMENT"), (5, "MOE_ERR_DEVICE_TIMEOUT")):
        assert nv.status_string(code) == name
    assert nv.status_string(99) == "MOE_ERR_UNKNOWN"


def test_workspace_sizing(lib):
    small = nv.make_desc(256, 16, 2, 128, 4)
    big = nv.make_desc(2048, 512, 10, 512, 65536)
    assert 0 < nv.moe_workspace_bytes(small) < nv.moe_workspace_bytes(big)
    # hq/hs + xq alone at 64k tokens
    assert nv.moe_workspace_bytes(big) > 65536 * 10 * (256 + 32) + 65536 * (1024 + 128)
    for bad in (nv.make_desc(100, 16, 2, 128, 4), nv.make_desc(256, 16, 17, 128, 4),
                nv.make_desc(256, 2000, 2, 128, 4), nv.make_desc(256, 16, 2, 96, 4),
                nv.make_desc(256, 16, 2, 128, 0), nv.make_desc(256, 16, 2, 128, 4, h_tensor_scale=0.0),
                nv.make_desc(256, 16, 2, 128, 4, flags=2)):
        assert nv.moe_workspace_bytes(bad) == 0


def test_create_rejects_bad_arguments_before_cuda(lib):
    out = ctypes.c_void_p(123)
    w = nv.NVFP4(None, None, None)
    bad = nv.make_desc(100, 16, 2, 128, 4)
    st = lib.moe_layer_create(ctypes.byref(bad), None, None, ctypes.byref(w), ctypes.byref(w),
                              ctypes.byref(w), None, None, ctypes.byref(out))
    assert st == nv.MOE_ERR_UNSUPPORTED_SHAPE and out.value is None
    good = nv.make_desc(256, 16, 2, 128, 4)
    st = lib.moe_layer_create(ctypes.byref(good), None, None, ctypes.byref(w), ctypes.byref(w),
                              ctypes.byref(w), None, None, ctypes.byref(out))
    assert st == nv.MOE_ERR_INVALID_ARGUMENT
    st = lib.moe_layer_create(ctypes.byref(good), None, None, None, None, None, None, None, None)
    assert st == nv.MOE_ERR_INVALID_ARGUMENT


def test_calls_reject_null_handles(lib):
    assert lib.moe_forward(None, None, None, None, None, 1, None, None, None, None, None,
                           None) == nv.MOE_ERR_INVALID_ARGUMENT
    assert lib.moe_quantize_act(None, None, 1, None, None, None, None, None) == \
        nv.MOE_ERR_INVALID_ARGUMENT
    assert lib.moe_layer_status(None, None) == nv.MOE_ERR_INVALID_ARGUMENT
    assert lib.moe_quantize_weights(None, 1, 1, 64, None, None, None, None) == \
        nv.MOE_ERR_INVALID_ARGUMENT
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf)
    assert lib.moe_quantize_weights(p, 1, 1, 96, p, p, p, None) == nv.MOE_ERR_UNSUPPORTED_SHAPE
    lib.moe_destroy(None)  # no-op


def test_packed_weight_bytes(lib):
    # only layers that can take the tensor-core path (more than 8 tokens, H and
    # I multiples of 256) have a packed buffer: the bf16 hi/lo copy of Wr
    # (2 parts x E x H x 2 bytes) and the tiled gate, up and down block scales
    # (E x I x H / 16 bytes each)
    def expect(H, E, I):
        return 2 * E * H * 2 + 3 * E * I * H // 16
    assert nv.moe_packed_weight_bytes(nv.make_desc(256, 16, 2, 256, 4)) == 0
    assert nv.moe_packed_weight_bytes(nv.make_desc(256, 16, 2, 256, 9)) == expect(256, 16, 256) == 212992
    assert nv.moe_packed_weight_bytes(nv.make_desc(2048, 512, 10, 512, 65536)) == \
        expect(2048, 512, 512) == 104857600
    assert nv.moe_packed_weight_bytes(
        nv.make_desc(256, 16, 2, 256, 64, flags=nv.MOE_FLAG_MULTI_KERNEL)) == 0
    assert nv.moe_packed_weight_bytes(nv.make_desc(256, 16, 2, 128, 64)) == 0   # I % 256 != 0
    assert nv.moe_packed_weight_bytes(nv.make_desc(100, 16, 2, 128, 64)) == 0   # invalid desc
