"""moe_experts_noalloc: the experts path for callers that cannot let the
library allocate (their device memory belongs to their own pool, or a
cudaMalloc's device synchronisation is not affordable in their loop). It uses
a fixed scratch array inside the library instead of a workspace.

Checked through the C ABI against moe_experts, the allocating entry point:
the two run the same kernels on the same inputs, so their outputs must be
equal bit for bit (the statistics of the usual layer tolerance are printed
too), on two calls in a row with different sizes (the second call reuses
the scratch the first one left behind); a call with an out-of-range expert
id after a large call (a stale inverse index left in the scratch must not
be read); and the rejection of sizes beyond the fixed scratch. This file
is collected last so that a run stopping at the first failure has already
run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import moe_synth as ms
import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_moe_layer_gb300 import build
    build.build()
    import bit_quantized_moe_layer_gb300 as m
    m.load()
    return m


def _routing(inp):
    rng = np.random.default_rng(inp.dims.T)
    d = inp.dims
    idx = np.stack([rng.choice(d.E, d.k, replace=False) for _ in range(d.T)]).astype(np.int32)
    w = ms.bf16_bits(rng.uniform(0.05, 0.3, (d.T, d.k)))
    return idx, w


def _noalloc(moe, g, idx, w):
    idx_d = torch.from_numpy(idx).cuda()
    w_d = gh.dev16(w)
    out = torch.full((g.d.T, g.d.H), -1, dtype=torch.int16, device="cuda")
    moe.moe_experts_noalloc(g.d, g.x, idx_d, w_d, g.layer.gate_up, g.layer.down, out)
    torch.cuda.synchronize()
    return gh.host16(out)


def test_noalloc_matches_allocating_call_twice(moe):
    for name, T in (("canvas", None), ("decode", None)):
        inp = ms.make_layer(name, T=T, seed=21)
        g = gh.upload(inp)
        idx, w = _routing(inp)
        got = _noalloc(moe, g, idx, w)
        want = gh.gpu_experts(g, idx, w)
        print(f"noalloc {name}: {gh.compare_out(got, want, f'noalloc {name}')}")
        assert np.array_equal(got, want), f"noalloc {name}: output differs from moe_experts"
    assert moe.device_error() == 0


def test_noalloc_bad_expert_after_large_call(moe):
    """A canvas-sized call leaves its inverse permutation in the scratch; a
    small call with an out-of-range id must drop that slot (adding nothing),
    raise the error word and stay finite, equal to moe_experts with the slot
    moved to a valid expert with weight 0."""
    big = ms.make_layer("canvas", seed=22)
    gb = gh.upload(big)
    _noalloc(moe, gb, *_routing(big))
    inp = ms.make_layer("canvas", T=8, seed=23)
    g = gh.upload(inp)
    idx, w = _routing(inp)
    bad, zero_w = idx.copy(), w.copy()
    bad[5, 2] = 300
    zero_w[5, 2] = 0
    moe.device_error()
    got = _noalloc(moe, g, bad, w)
    assert moe.device_error() & 2
    assert np.all(np.isfinite(gh.f64(got)))
    assert np.array_equal(got, gh.gpu_experts(g, idx, zero_w))


def test_noalloc_rejects_sizes_beyond_its_scratch(moe):
    d = moe.dims(4096, 2816, 128, 8, 704)
    assert moe.workspace_bytes(d) > (32 << 20)
    dummy = torch.zeros(64, dtype=torch.int32, device="cuda")
    q = moe.qweight(dummy, dummy, dummy)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_experts_noalloc(d, dummy, dummy, dummy, q, q, dummy)
    assert e.value.status == 5
