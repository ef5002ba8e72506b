"""The router with the pages' 4-bit group-64 projection (moe_route_q4 and
moe_forward_q4router, through the C ABI) against the oracle, and against the
dense router on the same weight dequantised independently."""
import dataclasses

import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
import gpu_helpers as gh
import oracle_checks as oc
import bit_quantized_moe_layer_gb300 as moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_moe_layer_gb300 import build
    build.build()
    oracle.build()


def dequantised(rq, d):
    """The 4-bit router weight dequantised independently (bf16 bits [E, H])."""
    return oc.torch_bf16_bits(oc.dense_dequant(rq[0][None], rq[1][None], rq[2][None], d.H, d.group)[0])


def upload_rq(rq):
    ts = (gh.dev32(rq[0]), gh.dev16(rq[1]), gh.dev16(rq[2]))
    return ts, moe.qweight(*ts)


def gpu_route_q4(g, rq_q):
    T, k = g.d.T, g.d.k
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.int16, device="cuda")
    moe.moe_route_q4(g.d, g.x, rq_q, g.layer.router_scale, g.layer.pes, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), gh.host16(w)


@pytest.mark.parametrize("name", ["tiny", "decode", "canvas", "prefill"])
def test_route_q4(name):
    inp = ms.make_layer(name)
    d = inp.dims
    rq = ms.make_router_q4(d, seed=30)
    g = gh.upload(inp)
    _, rq_q = upload_rq(rq)
    idx, w = gpu_route_q4(g, rq_q)
    ref = oracle.route_q4(d, inp.x, rq, inp.router_scale, inp.pes, taps=True)
    c = gh.check_routing(d, ref, idx, w, dequantised(rq, d))
    print(f"{name} q4 router: routing {c} of {d.T} tokens")


def test_route_q4_equals_dense_on_dequantised_weight():
    """Same kernel after the in-kernel dequantisation: the 4-bit router and the
    dense router on bf16(S q + B) (dequantised here) agree bit for bit."""
    inp = ms.make_layer("canvas")
    d = inp.dims
    rq = ms.make_router_q4(d, seed=31)
    dense = oc.torch_bf16_bits(oc.dense_dequant(rq[0][None], rq[1][None], rq[2][None], d.H, d.group)[0])
    g = gh.upload(dataclasses.replace(inp, router_w=dense))
    _, rq_q = upload_rq(rq)
    idx_q, w_q = gpu_route_q4(g, rq_q)
    prev = moe.set_router_path(1)  # the dense weight through the same (cluster) kernel
    try:
        idx_d, w_d = gh.gpu_route(g)
    finally:
        moe.set_router_path(prev)
    assert np.array_equal(idx_q, idx_d) and np.array_equal(w_q, w_d), "4-bit router != dense router on its weight"


def test_forward_q4router():
    inp = ms.make_layer("canvas")
    d = inp.dims
    rq = ms.make_router_q4(d, seed=32)
    g = gh.upload(inp)
    _, rq_q = upload_rq(rq)
    out = torch.empty((d.T, d.H), dtype=torch.int16, device="cuda")
    idx = torch.empty((d.T, d.k), dtype=torch.int32, device="cuda")
    w = torch.empty((d.T, d.k), dtype=torch.int16, device="cuda")
    moe.moe_forward_q4router(g.d, g.x, rq_q, g.layer.router_scale, g.layer.pes, g.layer.gate_up, g.layer.down, out,
                             idx, w)
    torch.cuda.synchronize()
    idx, w, out = idx.cpu().numpy(), gh.host16(w), gh.host16(out)
    ref = oracle.route_q4(d, inp.x, rq, inp.router_scale, inp.pes, taps=True)
    gh.check_routing(d, ref, idx, w, dequantised(rq, d))
    same = np.array([set(idx[t]) == set(ref["idx"][t]) for t in range(d.T)])
    want = gh.oracle_experts_rows(inp, ref["idx"], ref["w"], np.flatnonzero(same))
    print(f"canvas q4router forward: {gh.compare_out(out[same], want, 'q4router forward')}")
