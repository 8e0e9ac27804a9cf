"""Host-side checks of the C ABI: the library loads without a GPU, exports every
entry point that include/moe_ffn.h declares, sizes workspaces and rejects bad
arguments before touching the device."""

import ctypes
import os
import re

import pytest

import mixture_experts_ffn_infer_gb300 as mx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"^[A-Za-z_][\w \t\*]*?\b(moe_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_ffn_infer_gb300 import build
    build.build()
    return mx.load_library()


def test_header_declares_the_boundary():
    assert set(_declared()) >= {"moe_workspace_size", "moe_permute", "moe_experts_forward", "moe_combine",
                                "moe_infer", "moe_layer_forward", "moe_get_error", "moe_status_string"}


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) == set(mx.exported_symbols())


def test_status_strings(lib):
    for code, name in mx.STATUS.items():
        assert mx.moe_status_string(code) == name


def test_workspace_size_rules(lib):
    dm = mx.dims(7168, 2048, 384, 8)
    a = mx.moe_workspace_size(dm, 16)
    b = mx.moe_workspace_size(dm, 4096)
    c = mx.moe_workspace_size(dm, 4096, 2048)
    assert 0 < a < b < c
    # the big buffers dominate: sorted f16 rows, h and the weighted rows
    R = 4096 * 8
    assert b >= 2 * R * 7168 * 2 + 2 * R * 2048
    assert mx.moe_workspace_size(mx.dims(7168 + 64, 2048, 384, 8), 16) == 0      # d not a multiple of 128
    assert mx.moe_workspace_size(mx.dims(7168, 2048, 2000, 8), 16) == 0          # too many experts
    assert mx.moe_workspace_size(mx.dims(7168, 2048, 384, 33), 16) == 0          # k too large
    assert mx.moe_workspace_size(mx.dims(7168, 2048, 384, 8), 1 << 29) == 0     # n*k >= 2^31
    assert mx.moe_workspace_size(dm, 16, 100) == 0                              # shared width not x128
    # the activation scheme: dynamic FP8 uses the same workspace; unknown schemes are unsupported
    fp8 = mx.dims(7168, 2048, 384, 8, mx.MOE_ACT_FP8_DYNAMIC)
    assert mx.moe_workspace_size(fp8, 4096, 2048) == c
    for bad in (2, -1):
        assert mx.moe_workspace_size(mx.dims(7168, 2048, 384, 8, bad), 16) == 0


def test_host_argument_errors_return_codes_without_a_device(lib):
    dm = mx.dims(1024, 256, 16, 4)
    w = mx.moe_weights()
    L = lib
    # n = 0 is a no-op (needs a workspace pointer only for size checks)
    buf = (ctypes.c_uint8 * 512)()
    addr = (ctypes.addressof(buf) + 255) & ~255
    assert L.moe_combine(ctypes.byref(dm), 0, None, None, None, None, 0, None) == 0
    # missing workspace
    assert L.moe_infer(ctypes.byref(dm), 8, None, None, None, ctypes.byref(w), None, 0, None, 0, None, None) == 3
    # workspace too small
    assert L.moe_infer(ctypes.byref(dm), 8, None, None, None, ctypes.byref(w), None, 0, ctypes.c_void_p(addr), 256,
                       None, None) == 3
    # unsupported dims
    bad = mx.dims(1000, 256, 16, 4)
    assert L.moe_infer(ctypes.byref(bad), 8, None, None, None, ctypes.byref(w), None, 0, ctypes.c_void_p(addr),
                       1 << 30, None, None) == 2
    # negative n
    assert L.moe_combine(ctypes.byref(dm), -1, None, None, None, None, 0, None) == 1
    # null pointers with a large enough (claimed) workspace
    assert L.moe_infer(ctypes.byref(dm), 8, None, None, None, ctypes.byref(w), None, 0, ctypes.c_void_p(addr),
                       1 << 30, None, None) == 1
    # shared expert given without its width
    assert L.moe_layer_forward(ctypes.byref(dm), 8, None, None, 1e-6, None, None, ctypes.byref(w), ctypes.byref(w),
                               0, None, 0, ctypes.c_void_p(addr), 1 << 30, None, None) == 1
    assert L.moe_combine(ctypes.byref(dm), 8, None, None, None, None, 0, None) == 1
    assert L.moe_get_error(None, None) == 1
    # the MLP entry point takes one expert and k = 1 only, then checks like moe_infer
    one = mx.dims(1024, 256, 1, 1)
    assert L.moe_mlp_forward(ctypes.byref(dm), 8, None, ctypes.byref(w), None, 0, ctypes.c_void_p(addr), 1 << 30,
                             None) == 2
    assert L.moe_mlp_forward(ctypes.byref(one), 8, None, ctypes.byref(w), None, 0, None, 0, None) == 3
    assert L.moe_mlp_forward(ctypes.byref(one), 8, None, ctypes.byref(w), None, 0, ctypes.c_void_p(addr), 1 << 30,
                             None) == 1
    assert L.moe_mlp_forward(ctypes.byref(one), 0, None, ctypes.byref(w), None, 0, ctypes.c_void_p(addr), 1 << 30,
                             None) == 0


def test_tiled_bytes_and_permute_workspace(lib):
    # gate and up interleaved: twice one matrix; down in row-block pairs, padded to an even count
    assert mx.moe_tiled_bytes(0, 384, 7168, 2048) == 2 * 384 * 2048 * 7168
    assert mx.moe_tiled_bytes(2, 384, 7168, 2048) == 384 * 7168 * 2048
    assert mx.moe_tiled_bytes(2, 3, 384, 256) == 3 * 4 * 128 * 256          # 3 row blocks -> 2 pairs
    assert mx.moe_tiled_bytes(1, 3, 384, 256) == 0                          # w_up is not a tiled buffer
    assert mx.moe_tiled_bytes(0, 3, 300, 256) == 0                          # d not a multiple of 128
    # the routing prefix of the workspace: the error word only for small batches,
    # plus per-chunk counts above 8192 entries, and never more than the whole workspace
    dm = mx.dims(7168, 2048, 384, 8)
    small = mx.moe_permute_workspace_size(dm, 16)
    large = mx.moe_permute_workspace_size(dm, 32768)
    assert 256 <= small <= 4096
    assert large >= small + (32768 * 8 // 2048) * 384 * 4
    assert large < mx.moe_workspace_size(dm, 32768)
    assert mx.moe_permute_workspace_size(mx.dims(7168, 2048, 2000, 8), 16) == 0


def test_permute_rejects_a_workspace_shorter_than_its_prefix(lib):
    dm = mx.dims(128, 128, 384, 8)
    n = 4096                                   # 32768 entries: the chunked plan needs scratch
    need = mx.moe_permute_workspace_size(dm, n)
    buf = (ctypes.c_uint8 * (need + 256))()
    addr = (ctypes.addressof(buf) + 255) & ~255
    dummy = ctypes.c_void_p(addr)
    st = lib.moe_permute(ctypes.byref(dm), n, dummy, dummy, dummy, dummy, None, 0, ctypes.c_void_p(addr), need - 1,
                         None)
    assert st == 3


def test_static_scratch_size_matches_header():
    # the binding's copy of the built-in scratch size is the header's macro, the one the library is built with
    text = open(os.path.join(ROOT, "include", "moe_ffn.h")).read()
    m = re.search(r"#define\s+MOE_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m, "MOE_STATIC_SCRATCH_BYTES not found"
    assert mx.MOE_STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
    # K2 sizes: 24 tokens fit, 25 do not
    dm = mx.dims(7168, 2048, 384, 8)
    assert mx.moe_workspace_size(dm, 24) <= mx.MOE_STATIC_SCRATCH_BYTES < mx.moe_workspace_size(dm, 25)
