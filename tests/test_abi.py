"""The C-ABI library without a GPU: it builds, loads, exports every function
include/*.h declares, and rejects bad arguments on the host (no CUDA call is
made before the arguments pass)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_quantized_moe_layer_gb300 import build
    import bit_quantized_moe_layer_gb300 as moe
    build.build()
    return moe.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(moe_\w+)\s*\(", src, flags=re.M))
    return names


def test_exports_every_declared_function(lib):
    import bit_quantized_moe_layer_gb300 as moe
    names = declared_functions()
    assert names, "no declarations found"
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    assert names <= exported, f"declared but not exported: {names - exported}"
    assert set(moe.EXPORTS) == names, "binding's export list out of date"


def test_status_strings(lib):
    for s in range(0, 9):
        assert lib.moe_status_str(s)
    assert lib.moe_status_str(99) == b"unknown status"


def test_workspace_bytes(lib):
    import bit_quantized_moe_layer_gb300 as moe
    d = moe.dims(256, 2816, 128, 8, 704)
    n = moe.workspace_bytes(d)
    S = 256 * 8
    assert n >= S * 2816 * 2 * 2 + S * 704 * 2
    assert moe.workspace_bytes(moe.dims(256, 2816, 128, 8, 704, bits=8)) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(group=32), 4), (dict(bits=8), 4), (dict(k=33, E=64), 4), (dict(E=300), 4), (dict(k=9, E=8), 4),
    (dict(H=2880), 4), (dict(inter=700), 4), (dict(T=-1), 2), (dict(H=0), 2),
])
def test_bad_dims_rejected(lib, kw, status):
    import bit_quantized_moe_layer_gb300 as moe
    base = dict(T=8, H=256, E=8, k=2, inter=128)
    base.update(kw)
    d = moe.dims(**base)
    buf = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(buf) + 15) & ~15
    rc = lib.moe_route(ctypes.byref(d), p, p, p, p, p, p, None)
    assert rc == status


def test_null_and_alignment(lib):
    import bit_quantized_moe_layer_gb300 as moe
    d = moe.dims(8, 256, 8, 2, 128)
    buf = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(buf) + 15) & ~15
    assert lib.moe_route(ctypes.byref(d), None, p, p, p, p, p, None) == 1
    assert lib.moe_route(ctypes.byref(d), p + 2, p, p, p, p, p, None) == 3
    assert lib.moe_route(None, p, p, p, p, p, p, None) == 1
    q = moe.qweight(p, p, None)
    assert lib.moe_experts(ctypes.byref(d), p, p, p, ctypes.byref(q), ctypes.byref(q), p, None, 0, None) == 1
    good = moe.qweight(p, p, p)
    # workspace too small is a host-side error too (checked before any launch)
    rc = lib.moe_experts(ctypes.byref(d), p, p, p, ctypes.byref(good), ctypes.byref(good), p, p, 16, None)
    assert rc in (5, 8)  # 8 when the host has no GPU: the device check comes first


def test_zero_tokens_is_a_no_op(lib):
    import bit_quantized_moe_layer_gb300 as moe
    d = moe.dims(0, 256, 8, 2, 128)
    buf = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(buf) + 15) & ~15
    assert lib.moe_route(ctypes.byref(d), p, p, p, p, p, p, None) == 0


def test_dense_calls_check_arguments(lib):
    """The dense MLP calls are the one-expert, top-1 case: other E or k is a
    shape error; null and misaligned pointers and T = 0 as for the layer."""
    import bit_quantized_moe_layer_gb300 as moe
    buf = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(buf) + 15) & ~15
    q = moe.qweight(p, p, p)
    Q = ctypes.byref(q)
    for E, k, status in ((8, 2, 2), (2, 1, 2), (1, 2, 4)):  # k > E fails the layer's own check first
        d = moe.dims(8, 256, E, k, 192)
        assert lib.moe_dense_mlp(ctypes.byref(d), p, Q, Q, p, None, 0, None) == status
        assert lib.moe_dense_branch(ctypes.byref(d), p, p, p, Q, Q, p, None, 0, None) == status
        assert lib.moe_self_conditioning(ctypes.byref(d), p, p, p, Q, Q, p, None, 0, None) == status
    d = moe.dims(8, 256, 1, 1, 192)
    assert lib.moe_dense_mlp(ctypes.byref(d), None, Q, Q, p, None, 0, None) == 1
    assert lib.moe_dense_branch(ctypes.byref(d), p, None, p, Q, Q, p, None, 0, None) == 1
    assert lib.moe_self_conditioning(ctypes.byref(d), p + 2, p, p, Q, Q, p, None, 0, None) == 3
    assert lib.moe_dense_mlp(ctypes.byref(moe.dims(8, 256, 1, 1, 100)), p, Q, Q, p, None, 0, None) == 4
    d0 = moe.dims(0, 256, 1, 1, 192)
    assert lib.moe_self_conditioning(ctypes.byref(d0), p, p, p, Q, Q, p, None, 0, None) == 0


def test_lm_head_checks_arguments(lib):
    """moe_lm_head: E = k = 1, vocab a positive multiple of 128, a finite
    non-negative softcap, non-null aligned pointers; T = 0 is a no-op."""
    import bit_quantized_moe_layer_gb300 as moe
    buf = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(buf) + 15) & ~15
    q = moe.qweight(p, p, p)
    Q = ctypes.byref(q)
    cap = ctypes.c_float(30.0)
    d = moe.dims(8, 256, 1, 1, 64)
    assert lib.moe_lm_head(ctypes.byref(moe.dims(8, 256, 8, 2, 64)), 1024, cap, p, Q, p, None, 0, None) == 2
    assert lib.moe_lm_head(ctypes.byref(d), 0, cap, p, Q, p, None, 0, None) == 2
    assert lib.moe_lm_head(ctypes.byref(d), 1000, cap, p, Q, p, None, 0, None) == 4
    assert lib.moe_lm_head(ctypes.byref(d), 1024, ctypes.c_float(float("nan")), p, Q, p, None, 0, None) == 2
    assert lib.moe_lm_head(ctypes.byref(d), 1024, ctypes.c_float(-1.0), p, Q, p, None, 0, None) == 2
    assert lib.moe_lm_head(ctypes.byref(d), 1024, cap, None, Q, p, None, 0, None) == 1
    assert lib.moe_lm_head(ctypes.byref(d), 1024, cap, p, Q, p + 4, None, 0, None) == 3
    assert lib.moe_lm_head(ctypes.byref(moe.dims(0, 256, 1, 1, 64)), 1024, cap, p, Q, p, None, 0, None) == 0
