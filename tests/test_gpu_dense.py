"""Parity of the dense 4-bit GeGLU MLP calls (moe_dense_mlp, moe_dense_branch
and moe_self_conditioning, through the C ABI) with the oracle, on the
decoder-sized MLP (H = 2816, I = 2112) and a small one. Comparison rules:
tests/gpu_helpers.py (compare_out for the MLP output, compare_normed_out
for the outputs of a post norm)."""
import dataclasses

import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
import gpu_helpers as gh
import bit_quantized_moe_layer_gb300 as moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_moe_layer_gb300 import build
    build.build()
    oracle.build()


@dataclasses.dataclass
class GpuDense:
    d: moe.Dims
    x: torch.Tensor
    embeds: torch.Tensor
    pre_w: torch.Tensor
    post_w: torch.Tensor
    gu: tuple
    dn: tuple


def upload(dn: ms.DenseInputs) -> GpuDense:
    """gate_up = gate_proj rows then up_proj rows (with their scales and biases)."""
    gu = [np.concatenate([a, b])[None] for a, b in zip(dn.gate, dn.up)]
    down = [a[None] for a in dn.down]
    return GpuDense(moe.dims(dn.T, dn.H, 1, 1, dn.I, eps=dn.eps), gh.dev16(dn.x), gh.dev16(dn.embeds),
                    gh.dev16(dn.pre_w), gh.dev16(dn.post_w), (gh.dev32(gu[0]), gh.dev16(gu[1]), gh.dev16(gu[2])),
                    (gh.dev32(down[0]), gh.dev16(down[1]), gh.dev16(down[2])))


def run(g: GpuDense, kind: str):
    out = torch.empty((g.d.T, g.d.H), dtype=torch.int16, device="cuda")
    gu, dn = moe.qweight(*g.gu), moe.qweight(*g.dn)
    if kind == "mlp":
        moe.moe_dense_mlp(g.d, g.x, gu, dn, out)
    elif kind == "branch":
        moe.moe_dense_branch(g.d, g.x, g.pre_w, g.post_w, gu, dn, out)
    else:
        moe.moe_self_conditioning(g.d, g.embeds, g.x, g.pre_w, gu, dn, out)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    return gh.host16(out)


def sub(dn: ms.DenseInputs, rows: np.ndarray) -> ms.DenseInputs:
    return dataclasses.replace(dn, T=len(rows), x=dn.x[rows], embeds=dn.embeds[rows])


def check_mlp(dn, got, rows=None, what="dense MLP"):
    ref = sub(dn, rows) if rows is not None else dn
    want = oracle.dense_mlp(ref.x, ref.gate, ref.up, ref.down)
    return gh.compare_out(got if rows is None else got[rows], want, what)


def check_branch(dn, got, rows=None):
    ref = sub(dn, rows) if rows is not None else dn
    y = oracle.dense_mlp(oracle.rms_norm(ref.x, ref.pre_w, ref.eps), ref.gate, ref.up, ref.down)
    want = oracle.dense_branch(ref.x, ref.pre_w, ref.post_w, ref.gate, ref.up, ref.down, ref.eps)
    return gh.compare_normed_out(got if rows is None else got[rows], want, y, ref.post_w, ref.eps, "dense branch")


def check_self_conditioning(dn, got, rows=None):
    """c = bf16(embeds + s): the GPU's s is within the layer bound of the
    oracle's, and the add may round one ulp apart, so c_err = 2e-2 RMS(s) +
    ulp(s) + ulp(c)."""
    ref = sub(dn, rows) if rows is not None else dn
    s = oracle.dense_mlp(oracle.rms_norm(ref.x, ref.pre_w, ref.eps), ref.gate, ref.up, ref.down)
    c = ms.bf16_bits(ms.bits_to_f32(ref.embeds) + ms.bits_to_f32(s))
    sf, cf = gh.f64(s), gh.f64(c)
    c_err = 2e-2 * float(np.sqrt(np.mean(sf * sf))) + gh.bf16_ulp(sf) + gh.bf16_ulp(cf)
    want = oracle.self_conditioning(ref.embeds, ref.x, ref.pre_w, ref.gate, ref.up, ref.down, ref.eps)
    return gh.compare_normed_out(got if rows is None else got[rows], want, c, None, ref.eps, "self-conditioning",
                                 c_err=c_err)


CASES = {
    "small": dict(T=16, H=256, I=192),
    "decode": dict(T=8),
    "canvas": dict(T=256),
    "ragged1": dict(T=1),
    "ragged17": dict(T=17),
    "ragged130": dict(T=130),
}


@pytest.mark.parametrize("name", list(CASES))
def test_dense_mlp(name):
    dn = ms.make_dense(seed=40, **CASES[name])
    stats = check_mlp(dn, run(upload(dn), "mlp"))
    print(f"{name} dense MLP: {stats}")


@pytest.mark.parametrize("name", ["small", "decode", "canvas", "ragged17"])
def test_dense_branch(name):
    dn = ms.make_dense(seed=41, **CASES[name])
    print(f"{name} dense branch: {check_branch(dn, run(upload(dn), 'branch'))}")


@pytest.mark.parametrize("name", ["small", "decode", "canvas", "ragged17"])
def test_self_conditioning(name):
    dn = ms.make_dense(seed=42, **CASES[name])
    print(f"{name} self-conditioning: {check_self_conditioning(dn, run(upload(dn), 'selfcond'))}")


def sample_rows(T, n, seed):
    rng = np.random.default_rng(seed)
    return np.sort(np.concatenate([[0, T - 1], rng.choice(np.arange(1, T - 1), n - 2, False)]))


def test_dense_prefill_sampled():
    """T = 4096 (128-row token tiles, many per SM): every call on the full
    batch, checked on 48 sampled rows (rows are independent)."""
    dn = ms.make_dense(T=4096, seed=43)
    g = upload(dn)
    rows = sample_rows(dn.T, 48, 44)
    print(f"prefill dense MLP: {check_mlp(dn, run(g, 'mlp'), rows)}")
    print(f"prefill dense branch: {check_branch(dn, run(g, 'branch'), rows)}")
    print(f"prefill self-conditioning: {check_self_conditioning(dn, run(g, 'selfcond'), rows)}")


def test_dense_mlp_matches_one_expert_layer():
    """moe_dense_mlp against moe_experts with one expert, top-1, weight 1 on
    the same weights: both are within the layer bound of the oracle, and the
    two GPU outputs agree within one ulp (same products, tile shapes may
    differ)."""
    dn = ms.make_dense(T=64, seed=45)
    g = upload(dn)
    a = run(g, "mlp")
    idx = torch.zeros((dn.T, 1), dtype=torch.int32, device="cuda")
    w = torch.full((dn.T, 1), 0x3F80, dtype=torch.int16, device="cuda")
    out = torch.empty((dn.T, dn.H), dtype=torch.int16, device="cuda")
    moe.moe_experts(g.d, g.x, idx, w, moe.qweight(*g.gu), moe.qweight(*g.dn), out)
    torch.cuda.synchronize()
    b = gh.host16(out)
    fa, fb = gh.f64(a), gh.f64(b)
    assert np.all(np.abs(fa - fb) <= gh.bf16_ulp(np.maximum(np.abs(fa), np.abs(fb)))), "dense MLP != one-expert layer"
    check_mlp(dn, b, what="one-expert layer")
