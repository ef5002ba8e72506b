"""Parity of the decoder layer's MoE branch (moe_forward_branch, through the
C ABI) with the oracle's branch: the router on the residual, the experts on
RMSNorm(residual, pre_feedforward_layernorm_2), RMSNorm(., post_feedforward_
layernorm_2) of their combined output. Comparison rules: tests/gpu_helpers.py.
"""
import dataclasses

import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
import gpu_helpers as gh
import bit_quantized_moe_layer_gb300 as moe

pytestmark = pytest.mark.gpu

FULL = ("tiny", "decode", "canvas")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_moe_layer_gb300 import build
    build.build()
    oracle.build()


def gpu_branch(g, pre, post):
    T, k, H = g.d.T, g.d.k, g.d.H
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    xe = torch.empty((T, H), dtype=torch.int16, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.int16, device="cuda")
    moe.moe_forward_branch(g.d, g.x, g.layer.router_w, g.layer.router_scale, g.layer.pes, gh.dev16(pre),
                           gh.dev16(post), g.layer.gate_up, g.layer.down, out, idx, w, xe)
    torch.cuda.synchronize()
    return gh.host16(out), idx.cpu().numpy(), gh.host16(w), gh.host16(xe)


def check_expert_input(got, want, what):
    """The expert input is the same fp32 steps and one rounding on both sides
    from the same per-token rms, so it is bit-exact except where the two ways
    of forming the fp32 mean can differ (within ~2^-40 of a rounding boundary
    of the mean): at most one ulp, on a vanishing fraction of tokens."""
    g, o = gh.f64(got), gh.f64(want)
    diff = g != o
    if diff.any():
        assert np.all(np.abs(g - o)[diff] <= gh.bf16_ulp(o)[diff]), f"{what}: expert input off by more than an ulp"
        rows = np.unique(np.nonzero(diff)[0])
        assert rows.size <= max(1, got.shape[0] // 1000), f"{what}: expert input differs on {rows.size} tokens"


def run_case(inp, rows=None, seed=0):
    d = inp.dims
    pre, post = ms.make_branch_norms(d, seed)
    g = gh.upload(inp)
    out, idx, w, xe = gpu_branch(g, pre, post)
    ref = gh.oracle_route(inp)
    gh.check_routing(d, ref, idx, w, inp.router_w)
    xe_ref = oracle.rms_norm(inp.x, pre, d.eps)
    check_expert_input(xe, xe_ref, f"T={d.T}")
    rows = np.arange(d.T) if rows is None else rows
    same = np.array([set(idx[t]) == set(ref["idx"][t]) for t in rows])
    rows = rows[same]
    dr = dataclasses.replace(d, T=len(rows))
    y = oracle.experts(dr, xe_ref[rows], ref["idx"][rows], ref["w"][rows], (inp.gu_w, inp.gu_s, inp.gu_b),
                       (inp.dn_w, inp.dn_s, inp.dn_b))
    want = oracle.rms_norm(y, post, d.eps)
    return gh.compare_normed_out(out[rows], want, y, post, d.eps, f"branch T={d.T}")


@pytest.mark.parametrize("name", FULL)
def test_branch(name):
    stats = run_case(ms.make_layer(name))
    print(f"{name} branch: {stats}")


def test_branch_prefill_sampled():
    inp = ms.make_layer("prefill")
    rng = np.random.default_rng(5)
    rows = np.sort(np.concatenate([[0, inp.dims.T - 1], rng.choice(np.arange(1, inp.dims.T - 1), 46, False)]))
    print(f"prefill branch: {run_case(inp, rows, seed=1)}")


@pytest.mark.parametrize("T", [17, 256])
def test_branch_row_router(T):
    """The branch with the row router forced (moe_set_router_path(2)), which
    the default picks only at large T: its expert input and routing against
    the oracle at small T."""
    prev = moe.set_router_path(2)
    try:
        stats = run_case(ms.make_layer("canvas", T=T, seed=8), seed=3)
    finally:
        moe.set_router_path(prev)
    print(f"T={T} branch, row router: {stats}")


@pytest.mark.parametrize("T", [1, 17, 130])
def test_branch_ragged(T):
    run_case(ms.make_layer("canvas", T=T, seed=6), seed=2)


def test_branch_matches_composition():
    """The branch equals moe_route(residual), then moe_experts on the
    returned expert input, then the post norm's oracle, bit for bit on the
    routing and the expert input (same kernels), within tolerance on out."""
    inp = ms.make_layer("canvas", T=64, seed=7)
    d = inp.dims
    pre, post = ms.make_branch_norms(d, 7)
    g = gh.upload(inp)
    out, idx, w, xe = gpu_branch(g, pre, post)
    idx2, w2 = gh.gpu_route(g)
    assert np.array_equal(idx, idx2) and np.array_equal(w, w2), "branch routing != moe_route(residual)"
    g2 = dataclasses.replace(g, x=gh.dev16(xe))
    y = gh.gpu_experts(g2, idx, w)
    gh.compare_normed_out(out, oracle.rms_norm(y, post, d.eps), y, post, d.eps, "branch vs composition")
