"""The seeded input generator (CPU only)."""
import json
import os

import numpy as np

import moe_synth as ms

HERE = os.path.dirname(os.path.abspath(__file__))


def test_skew_kappa_matches_calibration():
    with open(os.path.join(HERE, "golden", "skew_calibration.json")) as fh:
        cal = json.load(fh)
    assert ms.SKEW_KAPPA == cal["chosen"]["kappa"]
    assert abs(cal["chosen"]["top10pct_share"] - 0.60) <= 0.05
    assert cal["chosen"]["empty_experts"] >= 3


def test_deterministic_and_shared_layer():
    a = ms.make_layer("canvas", T=4)
    b = ms.make_layer("canvas", T=4)
    for f in ("x", "router_w", "gu_w", "gu_s", "dn_b"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    c = ms.make_layer("decode")
    assert np.array_equal(a.gu_w, c.gu_w) and np.array_equal(a.router_w, c.router_w)


def test_shapes_and_distributions():
    inp = ms.make_layer("tiny")
    d = inp.dims
    assert inp.x.shape == (d.T, d.H) and inp.x.dtype == np.uint16
    assert inp.gu_w.shape == (d.E, 2 * d.inter, d.H // 8) and inp.gu_w.dtype == np.uint32
    assert inp.gu_s.shape == (d.E, 2 * d.inter, d.H // d.group)
    assert inp.dn_w.shape == (d.E, d.H, d.inter // 8)
    s = ms.bits_to_f32(inp.gu_s)
    assert s.min() >= 0.0049 and s.max() <= 0.0201
    assert np.array_equal(ms.bits_to_f32(inp.gu_b), -8.0 * s)
    codes = (inp.gu_w[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & 0xF
    hist = np.bincount(codes.ravel(), minlength=16) / codes.size
    assert np.all(np.abs(hist - 1 / 16) < 0.01)
    wr = ms.bits_to_f32(inp.router_w)
    assert abs(wr.std() - 0.05) < 0.005
    x = ms.bits_to_f32(inp.x)
    assert abs(x.mean()) < 0.1 and abs(x.std() - 1.0) < 0.1
