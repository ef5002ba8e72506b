"""The small-token dequant-GEMV path (moe_set_small_t_path(1)): the decode
workload and ragged token counts through the C ABI against the oracle with
the layer's comparison rules, and against the tcgen05 path on the same
inputs (the two dequantise identically; only the order of the fp32 sums
differs). The path is switched back to the default after each test."""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_moe_layer_gb300 import build
    build.build()
    oracle.build()
    import bit_quantized_moe_layer_gb300 as m
    m.load()
    return m


@pytest.fixture
def gemv(moe):
    prev = moe.set_small_t_path(1)
    yield moe
    moe.set_small_t_path(prev)


def test_path_switch(moe):
    assert moe.set_small_t_path(0) == 0
    assert moe.set_small_t_path(1) == 0
    assert moe.set_small_t_path(0) == 1
    with pytest.raises(moe.MoeError):
        moe.set_small_t_path(2)


@pytest.mark.parametrize("name,T", [("decode", None), ("canvas", 1), ("canvas", 17), ("canvas", 32)])
def test_gemv_experts_and_forward(gemv, name, T):
    inp = ms.make_layer(name, T=T, seed=14 if T else 0)
    d = inp.dims
    assert d.T * d.k <= 2 * d.E  # the call takes the GEMV path
    g = gh.upload(inp)
    ref = gh.oracle_route(inp)
    out = gh.gpu_experts(g, ref["idx"], ref["w"])
    want = gh.oracle_experts_rows(inp, ref["idx"], ref["w"])
    stats = gh.compare_out(out, want, f"gemv {name} T={d.T} experts", gh.explainer(inp, ref["idx"], ref["w"]))
    print(f"gemv {name} T={d.T} experts: {stats}")
    fo, idx, w = gh.gpu_forward(g)
    gh.check_routing(d, ref, idx, w, inp.router_w)
    same = np.array([set(idx[t]) == set(ref["idx"][t]) for t in range(d.T)])
    gh.compare_out(fo[same], want[same], f"gemv {name} forward")
    assert gemv.device_error() == 0


def test_gemv_matches_tensor_core_path(moe):
    """Same inputs through both paths: equal but for fp32 summation order, so
    within the layer tolerance of each other (a one-ulp flip of an
    intermediate z, m or y carries through the later products, so they are
    not ulp-close element by element)."""
    inp = ms.make_layer("decode", seed=15)
    g = gh.upload(inp)
    ref = gh.oracle_route(inp)
    a = gh.gpu_experts(g, ref["idx"], ref["w"])
    prev = moe.set_small_t_path(1)
    try:
        b = gh.gpu_experts(g, ref["idx"], ref["w"])
    finally:
        moe.set_small_t_path(prev)
    stats = gh.compare_out(b, a, "gemv vs tcgen05")
    print(f"gemv vs tcgen05: {stats}")


def test_gemv_dispatch_in_workspace(gemv):
    """The GEMV path's in-call dispatch (token tiles of up to 4 rows) read
    back from the caller workspace, bit for bit."""
    inp = ms.make_layer("decode", seed=16)
    d = inp.dims
    g = gh.upload(inp)
    ws = torch.full((gemv.workspace_bytes(g.d),), 0x33, dtype=torch.uint8, device="cuda")
    out, idx, w = gh.gpu_forward(g, workspace=ws)
    perm, off, inv = gh.workspace_dispatch(g.d, ws)
    operm, ooff, oinv = oracle.dispatch(d.T, d.k, d.E, idx)
    assert np.array_equal(off, ooff) and np.array_equal(perm, operm) and np.array_equal(inv, oinv)
