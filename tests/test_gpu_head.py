"""Parity of the tied 4-bit head with its final-logit softcap (moe_lm_head,
through the C ABI) with the oracle, at a vocabulary of 2^18 and smaller.

Comparison rule: the GPU's bf16 logit x may differ from the oracle's within
the layer bound max(2e-2 RMS(x), 1 bf16 ulp) (fp32 accumulation against the
exact sum); the softcap's derivative is at most 1, and both sides round
three fp32 steps (CUDA's tanhf within 2 ulps), so
|out - ref| <= max(2e-2 RMS(x), ulp(x)) + 4 fp32 ulps of ref, and the RMS
error stays below 1e-3 of the RMS.
"""
import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
import gpu_helpers as gh
import bit_quantized_moe_layer_gb300 as moe

pytestmark = pytest.mark.gpu
CAP = 30.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_moe_layer_gb300 import build
    build.build()
    oracle.build()


def upload(h, emb):
    return gh.dev16(h), (gh.dev32(emb[0]), gh.dev16(emb[1]), gh.dev16(emb[2]))


def run(h_d, emb_d, T, H, V, cap):
    d = moe.dims(T, H, 1, 1, 64)
    out = torch.empty((T, V), dtype=torch.float32, device="cuda")
    moe.moe_lm_head(d, V, cap, h_d, moe.qweight(*emb_d), out)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    return out.cpu().numpy()


def compare(got, want, logits_ref, what):
    x = gh.f64(logits_ref)
    rms = float(np.sqrt(np.mean(x * x)))
    o, g = want.astype(np.float64), got.astype(np.float64)
    err = np.abs(g - o)
    tol = np.maximum(2e-2 * rms, gh.bf16_ulp(x)) + 4 * 2.0 ** -24 * np.abs(o)
    bad = np.flatnonzero((err > tol).ravel())
    stats = dict(logit_rms=rms, max_err_over_tol=float((err / tol).max()),
                 rms_err_over_rms=float(np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(o ** 2))),
                 n_diff=int((err > 0).sum()), n=int(err.size))
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    assert bad.size == 0, f"{what}: {bad.size} elements beyond tolerance {stats}"
    assert stats["rms_err_over_rms"] <= 1e-3, f"{what}: RMS error too large {stats}"
    return stats


CASES = {
    "small_saturating": dict(T=5, H=256, V=384, h_scale=40.0),
    "ragged17": dict(T=17, H=2816, V=4096, h_scale=1.0),
    "tiles300": dict(T=300, H=2816, V=2048, h_scale=3.0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_head(name):
    c = CASES[name]
    h, emb = ms.make_head(c["T"], H=c["H"], V=c["V"], seed=60, h_scale=c["h_scale"])
    got = run(*upload(h, emb), c["T"], c["H"], c["V"], CAP)
    want, lg = oracle.lm_head(h, emb, cap=CAP, taps=True)
    print(f"{name} head: {compare(got, want, lg, name)}")


def test_head_no_cap_is_bf16_logits():
    """Cap 0: the output is the bf16 logit widened (exactly representable in
    bf16), within the layer bound of the oracle's logits."""
    h, emb = ms.make_head(9, H=2816, V=1024, seed=61)
    got = run(*upload(h, emb), 9, 2816, 1024, 0.0)
    bits = got.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "cap 0 output is not a widened bf16"
    want, lg = oracle.lm_head(h, emb, cap=0.0, taps=True)
    compare(got, want, lg, "no cap")


def test_head_softcap_of_own_logits():
    """The epilogue's softcap on the GPU's own logits: cap * tanh(x / cap)
    in float64 of the cap-0 output, within 4 fp32 ulps (three fp32 roundings,
    CUDA's tanhf within 2 ulps). Saturating logits."""
    h, emb = ms.make_head(6, H=256, V=512, seed=62, h_scale=40.0)
    hd, ed = upload(h, emb)
    x = run(hd, ed, 6, 256, 512, 0.0).astype(np.float64)
    got = run(hd, ed, 6, 256, 512, CAP).astype(np.float64)
    assert np.abs(x).max() > 2 * CAP
    exact = CAP * np.tanh(x / CAP)
    assert np.all(np.abs(got - exact) <= 4 * 2.0 ** -24 * np.abs(exact) + 1e-30), "softcap epilogue"


@pytest.mark.parametrize("T,rows", [(8, None), (256, [0, 1, 127, 128, 255])])
def test_head_full_vocab(T, rows):
    """Vocabulary 2^18 (decode T = 8: every row; canvas T = 256: sampled rows
    across both 128-row token tiles), every vocabulary column."""
    V, H = ms.VOCAB, 2816
    h, emb = ms.make_head(T, H=H, V=V, seed=63)
    got = run(*upload(h, emb), T, H, V, CAP)
    r = np.arange(T) if rows is None else np.array(rows)
    want, lg = oracle.lm_head(h[r], emb, cap=CAP, taps=True)
    print(f"T={T} head, vocab {V}: {compare(got[r], want, lg, f'T={T} vocab {V}')}")
