"""Pins of the CPU oracle against facts that do not come from the oracle.

Each check takes a loaded oracle library, so the same checks run against the
oracle proper (tests/test_oracle_pins.py) and against builds of it with one
planted mistake (tests/test_oracle_mutants.py), which they must catch.

The references used here are independent of the oracle's code: closed forms,
invariants, brute force over tiny inputs, numpy/torch library routines
(float64 matmul, stable argsort, topk, gelu(approximate='tanh'), torch's
float32 -> bf16 rounding), and a "nearest bf16" property that checks a
rounded value against the exact one without re-implementing the rounding.
"""
from __future__ import annotations

import dataclasses
import json
import math
import os

import numpy as np
import torch

import moe_synth as ms
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


# ----------------------------------------------------------------- helpers --
def f64(bits) -> np.ndarray:
    return ms.bits_to_f32(bits).astype(np.float64)


def torch_bf16_bits(x_f32) -> np.ndarray:
    """float32 -> bf16 bits via torch's own conversion (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def neighbours(bits):
    """The two bf16 values adjacent to each given bf16 value (as float64)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int32)
    sign = b & 0x8000
    mag = b & 0x7FFF
    away = sign | np.minimum(mag + 1, 0x7F80)
    toward = np.where(mag == 0, (sign ^ 0x8000) | 1, sign | (mag - 1))
    return f64(away.astype(np.uint16)), f64(toward.astype(np.uint16))


def assert_nearest_bf16(bits, exact, what: str, rel_slack: float = 0.0):
    """Every bf16 value in `bits` is a nearest bf16 to the float64 `exact`."""
    c = f64(bits)
    exact = np.asarray(exact, dtype=np.float64)
    a, t = neighbours(bits)
    d0 = np.abs(c - exact)
    slack = rel_slack * np.abs(exact)
    ok = (d0 <= np.abs(a - exact) + slack) & (d0 <= np.abs(t - exact) + slack)
    bad = np.flatnonzero(~ok.ravel())
    assert bad.size == 0, (f"{what}: {bad.size} of {ok.size} values are not the nearest bf16; "
                           f"first at {bad[0]}: got {c.ravel()[bad[0]]!r} for exact {exact.ravel()[bad[0]]!r}")


def unpack_codes(w_words: np.ndarray, K: int) -> np.ndarray:
    """[.., N, K/8] uint32 -> [.., N, K] codes, nibble j of word i is element 8i+j."""
    shifts = (4 * np.arange(8, dtype=np.uint32))
    q = (w_words[..., :, None] >> shifts) & np.uint32(0xF)
    return q.reshape(*w_words.shape[:-1], K).astype(np.float64)


def dense_dequant(w_words, s_bits, b_bits, K: int, g: int) -> np.ndarray:
    """Dense dequantised weight bf16(S q + B) as float64, via float32 (where
    S q + B is exact for these inputs) and torch's bf16 rounding."""
    q = unpack_codes(w_words, K)
    S = np.repeat(f64(s_bits), g, axis=-1)
    B = np.repeat(f64(b_bits), g, axis=-1)
    v = S * q + B
    v32 = v.astype(np.float32)
    assert np.array_equal(v32.astype(np.float64), v), "test input not exact in float32"
    return f64(torch_bf16_bits(v32))


def geglu_exact(gate, up) -> np.ndarray:
    """gelu_approx(gate) * up in 100-digit arithmetic (mpmath), as float64."""
    import mpmath
    mpmath.mp.dps = 100
    c = mpmath.sqrt(2 / mpmath.pi)
    out = np.empty(len(gate))
    for i, (g, u) in enumerate(zip(gate, up)):
        g = mpmath.mpf(float(g))
        out[i] = float(g / 2 * (1 + mpmath.tanh(c * (g + mpmath.mpf("0.044715") * g ** 3))) * mpmath.mpf(float(u)))
    return out


def small_dims(**kw) -> ms.Dims:
    base = dict(T=16, H=256, E=8, k=2, inter=128, group=64)
    base.update(kw)
    return ms.Dims(**base)


def load_golden(name: str) -> dict:
    with open(os.path.join(HERE, "golden", name)) as fh:
        return json.load(fh)


# --------------------------------------------------------- rounding pins --
def check_bf16_from_float(lib):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(2000).astype(np.float32),
        (rng.standard_normal(500) * 1e30).astype(np.float32),
        (rng.standard_normal(500) * 1e-38).astype(np.float32),   # subnormal range
        np.array([0.0, -0.0, 1.0, -1.0, 3.4e38, -3.4e38, 1.00390625, 1.01171875], np.float32),
    ])
    got = np.array([oracle.bf16_from_float(float(v), lib) for v in vals], np.uint16)
    want = torch_bf16_bits(vals)
    assert np.array_equal(got, want), "bf16_from_float disagrees with torch's RNE conversion"


def check_bf16_from_double(lib):
    rng = np.random.default_rng(2)
    # float32-exact doubles: one rounding must equal torch's float32 -> bf16.
    v32 = rng.standard_normal(1000).astype(np.float32)
    got = np.array([oracle.bf16_from_double(float(v), lib) for v in v32], np.uint16)
    assert np.array_equal(got, torch_bf16_bits(v32)), "bf16_from_double on float32-exact values"
    # general doubles: nearest property.
    vd = rng.standard_normal(1000) * np.exp(rng.uniform(-20, 20, 1000))
    got = np.array([oracle.bf16_from_double(float(v), lib) for v in vd], np.uint16)
    assert_nearest_bf16(got, vd, "bf16_from_double")
    # exact ties go to even; a tie nudged by 2^-40 goes up (no double rounding).
    one_plus = 1.0 + 2.0 ** -8            # halfway between 1 and 1+2^-7
    assert oracle.bf16_from_double(one_plus, lib) == 0x3F80
    assert oracle.bf16_from_double(one_plus + 2.0 ** -40, lib) == 0x3F81
    three_half = 1.0 + 3 * 2.0 ** -8      # halfway between 1+2^-7 and 1+2^-6 -> even (1+2^-6)
    assert oracle.bf16_from_double(three_half, lib) == 0x3F82
    assert oracle.bf16_from_double(-one_plus - 2.0 ** -40, lib) == 0xBF81


# ------------------------------------------------------------ router pins --
def _route(lib, d, x, wr, sc, pes):
    return oracle.route(d, x, wr, sc, pes, taps=True, lib=lib)


def check_router_constant_row(lib):
    """x = 1 everywhere, scale = 1: the norm gives 1 and the output is the
    hidden**-0.5 scalar itself (H=256: 1/16 exactly; H=2816: golden)."""
    golden = load_golden("router_root_bf16.json")
    for H, want in ((256, 0x3D80), (golden["H"], int(golden["root_bits"], 16))):
        d = small_dims(T=2, H=H, E=4, k=2)
        x = np.full((d.T, H), 0x3F80, np.uint16)
        _, sc, pes = ms.make_router(d)
        sc = np.full(H, 0x3F80, np.uint16)
        wr = ms.make_router(d)[0]
        r = _route(lib, d, x, wr, sc, pes)
        assert np.all(r["normed"] == want), f"constant row, H={H}: normed != {want:#06x}"



def _golden_row(g) -> np.ndarray:
    """The hand-built row of the norm-rounding goldens: x[0] = 64, else 1."""
    x = np.full(g["H"], 0x3F80, np.uint16)
    x[0] = 0x4280
    return x


def check_router_norm_rounding_golden(lib):
    """Hand-derived bits of n3 = bf16(bf16(bf16(x r) scale) bf16(H^-0.5)) on
    a row where the bf16 scalar and the fp32 scalar, and a rounded and an
    unrounded n, give different results (golden: router_norm_rounding.json)."""
    g = load_golden("router_norm_rounding.json")
    H = g["H"]
    d = dataclasses.replace(small_dims(T=2, H=H, E=4, k=2), eps=g["eps"])
    x = np.tile(_golden_row(g), (d.T, 1))
    sc = np.full(H, 0x3F80, np.uint16)
    sc[1], sc[2] = 0x3F10, 0x3F04
    wr, _, pes = ms.make_router(d)
    r = _route(lib, d, x, wr, sc, pes)
    for h, want in g["normed_bits"].items():
        got = r["normed"][:, int(h)]
        assert np.all(got == int(want, 16)), f"normed[{h}] = {got[0]:#06x}, golden {want}"

def check_router_zero_row(lib):
    """x = 0: every score is 0, the tie goes to the lowest ids and the
    softmax is uniform: w_j = bf16(bf16(1/k) * pes[j])."""
    d = small_dims(T=3, E=8, k=3)
    inp = ms.make_custom(d)
    x = np.zeros((d.T, d.H), np.uint16)
    r = _route(lib, d, x, inp.router_w, inp.router_scale, inp.pes)
    assert np.all(r["normed"] == 0)
    assert np.array_equal(r["idx"], np.tile(np.arange(d.k, dtype=np.int32), (d.T, 1)))
    p = torch.tensor(1.0 / d.k, dtype=torch.float32).to(torch.bfloat16)
    pes = torch.from_numpy(ms.bits_to_f32(inp.pes[: d.k])).to(torch.bfloat16)
    want = (p * pes).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(r["w"], np.tile(want, (d.T, 1))), "zero row: weights"


def check_router_scale_invariance(lib):
    """With eps = 0 the layer's router is invariant under x -> 2x, bit for bit."""
    d = dataclasses.replace(small_dims(T=32, E=16, k=4), eps=0.0)
    inp = ms.make_custom(d, seed=3)
    x2 = ms.bf16_bits(ms.bits_to_f32(inp.x) * 2.0)
    a = _route(lib, d, inp.x, inp.router_w, inp.router_scale, inp.pes)
    b = _route(lib, d, x2, inp.router_w, inp.router_scale, inp.pes)
    for key in ("normed", "idx", "w"):
        assert np.array_equal(a[key], b[key]), f"x -> 2x changed {key}"


def check_router_exact_math(lib):
    """normed ~ x / sqrt(mean(x^2) + eps) * scale * H^-0.5 within the error of
    its four roundings; mean(normed^2 / (scale H^-0.5)^2) ~ 1."""
    d = small_dims(T=32, E=16, k=4)
    inp = ms.make_custom(d, seed=4)
    r = _route(lib, d, inp.x, inp.router_w, inp.router_scale, inp.pes)
    x = f64(inp.x)
    exact = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + d.eps) * f64(inp.router_scale) * d.H ** -0.5
    n = f64(r["normed"])
    tol = 5 * 2.0 ** -8 * np.abs(exact) + 1e-30
    assert np.all(np.abs(n - exact) <= tol), "normed far from the exact RMS-norm * scale * H^-0.5"


def check_router_logits_topk(lib):
    """scores = nearest bf16 of normed . W_r^T (float64 library matmul);
    idx = first k of sorted by (score desc, id asc); torch.topk agrees
    wherever the k-th and (k+1)-th scores differ."""
    d = small_dims(T=64, E=16, k=4)
    inp = ms.make_custom(d, seed=5)
    r = _route(lib, d, inp.x, inp.router_w, inp.router_scale, inp.pes)
    lg = f64(r["normed"]) @ f64(inp.router_w).T
    assert np.allclose(r["logits"], lg, rtol=1e-12, atol=1e-15), "exact logits != library matmul"
    assert_nearest_bf16(r["scores"], lg, "router scores")
    s = f64(r["scores"])
    for t in range(d.T):
        want = sorted(range(d.E), key=lambda e: (-s[t, e], e))[: d.k]
        assert list(r["idx"][t]) == want, f"top-k order, token {t}"
        srt = np.sort(s[t])[::-1]
        if srt[d.k - 1] != srt[d.k]:
            tk = torch.topk(torch.from_numpy(s[t]), d.k).indices.numpy()
            assert set(tk.tolist()) == set(want), f"torch.topk disagrees, token {t}"


def check_router_weights(lib):
    """w ~ softmax(scores[idx]) * pes[idx] (exact math, two bf16 roundings);
    pes = 1 sums to 1 within k bf16 ulps; doubling pes doubles w exactly."""
    d = small_dims(T=64, E=16, k=4)
    inp = ms.make_custom(d, seed=6)
    r = _route(lib, d, inp.x, inp.router_w, inp.router_scale, inp.pes)
    s = np.take_along_axis(f64(r["scores"]), r["idx"].astype(np.int64), 1)
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    exact = p * f64(inp.pes)[r["idx"]]
    assert np.all(np.abs(f64(r["w"]) - exact) <= 2 * 2.0 ** -8 * exact), "routing weights"
    ones = np.full_like(inp.pes, 0x3F80)
    r1 = _route(lib, d, inp.x, inp.router_w, inp.router_scale, ones)
    assert np.all(np.abs(f64(r1["w"]).sum(1) - 1.0) <= d.k * 2.0 ** -8), "pes=1: sum of w"
    pes2 = ms.bf16_bits(ms.bits_to_f32(inp.pes) * 2.0)
    r2 = _route(lib, d, inp.x, inp.router_w, inp.router_scale, pes2)
    assert np.array_equal(r2["idx"], r["idx"])
    assert np.array_equal(f64(r2["w"]), 2.0 * f64(r["w"])), "pes*2 must give w*2 exactly"


# ---------------------------------------------------------- dispatch pins --
def check_dispatch(lib):
    rng = np.random.default_rng(7)
    for T, k, E in ((1, 1, 1), (16, 2, 8), (100, 8, 128), (37, 3, 11)):
        idx = rng.integers(0, max(1, E // 2 + 1), size=(T, k)).astype(np.int32)  # leaves experts empty
        idx[0, 0] = E - 1
        perm, off, inv = oracle.dispatch(T, k, E, idx, lib=lib)
        flat = idx.ravel()
        assert np.array_equal(perm, np.argsort(flat, kind="stable")), "perm != stable argsort"
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        assert np.array_equal(np.sort(perm), np.arange(T * k)), "perm is not a bijection"
        assert np.array_equal(inv[perm], np.arange(T * k)), "inv is not perm's inverse"
        assert np.all(flat[perm][:-1] <= flat[perm][1:])


# ----------------------------------------------------------- expert pins --
def check_experts_brute_force(lib):
    """z, m, y and out of every slot against a dense float64 computation of
    the same layer (library matmul, torch gelu tanh, torch bf16 rounding)."""
    d = small_dims(T=8, E=4, k=2)
    inp = ms.make_custom(d, seed=8)
    rt = oracle.route(d, inp.x, inp.router_w, inp.router_scale, inp.pes, lib=lib)
    out, z, m, y = oracle.experts(d, inp.x, rt["idx"], rt["w"], (inp.gu_w, inp.gu_s, inp.gu_b),
                                  (inp.dn_w, inp.dn_s, inp.dn_b), taps=True, lib=lib)
    I, H = d.inter, d.H
    x = f64(inp.x)
    for f in range(d.T * d.k):
        t, e = f // d.k, int(rt["idx"].ravel()[f])
        wgu = dense_dequant(inp.gu_w[e], inp.gu_s[e], inp.gu_b[e], H, d.group)
        wdn = dense_dequant(inp.dn_w[e], inp.dn_s[e], inp.dn_b[e], I, d.group)
        assert_nearest_bf16(z[f], wgu @ x[t], f"gate_up output, slot {f}")
        zz = f64(z[f])
        assert_nearest_bf16(m[f], geglu_exact(zz[:I], zz[I:]), f"GeGLU output, slot {f}")
        assert_nearest_bf16(y[f], wdn @ f64(m[f]), f"down output, slot {f}")
    prods = f64(torch_bf16_bits(ms.bits_to_f32(y) * ms.bits_to_f32(rt["w"]).reshape(-1, 1)))
    assert_nearest_bf16(out, prods.reshape(d.T, d.k, H).sum(1), "combine")


def _one_hot_layer(lib, xrows, gate_code, up_code, down_code, n0=37, K0=70, K1=201, h0=133):
    """Layer whose weights are all 0 (codes 8, S = 1, B = -8) except gate
    (n0, K0), up (I+n0, K1) and down (h0, n0), whose codes set multipliers
    code-8. k = 1, weight 1. Returns out [T, H] bits."""
    d = small_dims(T=len(xrows), E=1, k=1)
    I, H, g = d.inter, d.H, d.group
    gu_w = np.full((1, 2 * I, H // 8), 0x88888888, np.uint32)
    dn_w = np.full((1, H, I // 8), 0x88888888, np.uint32)
    gu_w[0, n0, K0 // 8] = np.uint32(0x88888888 ^ ((8 ^ gate_code) << (4 * (K0 % 8))))
    gu_w[0, I + n0, K1 // 8] = np.uint32(0x88888888 ^ ((8 ^ up_code) << (4 * (K1 % 8))))
    dn_w[0, h0, n0 // 8] = np.uint32(0x88888888 ^ ((8 ^ down_code) << (4 * (n0 % 8))))
    ones_g = lambda n, kk: np.full((1, n, kk // g), 0x3F80, np.uint16)
    m8_g = lambda n, kk: np.full((1, n, kk // g), 0xC100, np.uint16)  # -8.0
    x = np.zeros((d.T, H), np.uint16)
    x[:, K0] = xrows[:, 0]
    x[:, K1] = xrows[:, 1]
    idx = np.zeros((d.T, 1), np.int32)
    w = np.full((d.T, 1), 0x3F80, np.uint16)
    return oracle.experts(d, x, idx, w, (gu_w, ones_g(2 * I, H), m8_g(2 * I, H)),
                          (dn_w, ones_g(H, I), m8_g(H, I)), lib=lib or oracle.load()), h0


def check_experts_one_hot(lib):
    """Closed form: with gate multiplier 1, up 2 and down 3, out[t, h0] =
    bf16(3 m), m = bf16(gelu_tanh(x[t,K0]) * 2 x[t,K1]), and out is 0 elsewhere."""
    rng = np.random.default_rng(9)
    xr = ms.bf16_bits(rng.standard_normal((6, 2)) * 2)
    out, h0 = _one_hot_layer(lib, xr, 9, 10, 11)
    for t in range(len(xr)):
        gate, up = f64(xr[t, 0]), 2.0 * f64(xr[t, 1])
        mex = geglu_exact(np.array([gate]), np.array([up]))
        mbits = torch_bf16_bits(np.float32(mex))  # float32 first: exact enough away from ties
        assert_nearest_bf16(mbits, mex, "m")
        want = np.zeros(out.shape[1])
        want[h0] = f64(torch_bf16_bits(np.float32(3.0 * f64(mbits)[0])))[0]
        assert np.array_equal(f64(out[t]), want), f"one-hot layer, token {t}"


def check_geglu_ties(lib):
    """gelu_tanh(g) < g for g > 0, so where g*up is exactly halfway between two
    bf16 values, the exact product lies below the tie and rounds toward zero:
    g=5.5, up=2.0625: g*up = 11.34375 (between 11.3125 and 11.375) -> 11.3125;
    g=7.5, up=1.03125 (7.734375, between 7.71875 and 7.75) -> 7.71875, where
    double arithmetic can no longer tell the logistic factor from 1."""
    cases = [(5.5, 2.0625, 11.3125), (7.5, 1.03125, 7.71875), (-5.5, -2.0625, -0.0)]
    xr = ms.bf16_bits(np.array([[g, u] for g, u, _ in cases], np.float32))
    out, h0 = _one_hot_layer(lib, xr, 9, 9, 9)
    for t, (g, u, want) in enumerate(cases):
        got = f64(out[t, h0])
        if want == 0.0:
            assert abs(got) < 1e-6, f"g={g}: {got}"
        else:
            assert got == want, f"GeGLU tie g={g} up={u}: got {got}, want {want}"


def check_single_expert_identity(lib):
    """E = 1, k = 1, pes = 1: softmax of one score is 1, so w = 1 exactly and
    the layer is the dense 4-bit GeGLU MLP: out = y."""
    d = small_dims(T=8, E=1, k=1)
    inp = ms.make_custom(d, seed=10)
    pes = np.full(1, 0x3F80, np.uint16)
    rt = oracle.route(d, inp.x, inp.router_w, inp.router_scale, pes, lib=lib)
    assert np.all(rt["idx"] == 0) and np.all(rt["w"] == 0x3F80)
    out, z, m, y = oracle.experts(d, inp.x, rt["idx"], rt["w"], (inp.gu_w, inp.gu_s, inp.gu_b),
                                  (inp.dn_w, inp.dn_s, inp.dn_b), taps=True, lib=lib)
    assert np.array_equal(out, y), "single expert: out != y"


def check_expert_relabel(lib):
    """Renaming the experts (router rows, pes, weights permuted together)
    leaves the layer output unchanged on tokens without a score tie at the
    top-k boundary."""
    d = small_dims(T=32, E=8, k=2)
    inp = ms.make_custom(d, seed=11)
    out_a, idx_a, _ = oracle.forward(inp, lib=lib)
    pi = np.random.default_rng(12).permutation(d.E)
    perm_inp = dataclasses.replace(
        inp, router_w=inp.router_w[pi], pes=inp.pes[pi], gu_w=inp.gu_w[pi], gu_s=inp.gu_s[pi],
        gu_b=inp.gu_b[pi], dn_w=inp.dn_w[pi], dn_s=inp.dn_s[pi], dn_b=inp.dn_b[pi])
    out_b, idx_b, _ = oracle.forward(perm_inp, lib=lib)
    sc = f64(oracle.route(d, inp.x, inp.router_w, inp.router_scale, inp.pes, taps=True, lib=lib)["scores"])
    srt = -np.sort(-sc, 1)
    clean = srt[:, d.k - 1] != srt[:, d.k]
    assert clean.sum() > d.T // 2
    for t in np.flatnonzero(clean):
        assert set(pi[idx_b[t]].tolist()) == set(idx_a[t].tolist()), f"relabelled routing, token {t}"
    assert np.array_equal(out_a[clean], out_b[clean]), "relabelling experts changed the output"


def check_token_permutation(lib):
    """Tokens are independent: permuting them permutes the output rows."""
    d = small_dims(T=24, E=8, k=2)
    inp = ms.make_custom(d, seed=13)
    out_a, _, _ = oracle.forward(inp, lib=lib)
    pi = np.random.default_rng(14).permutation(d.T)
    out_b, _, _ = oracle.forward(dataclasses.replace(inp, x=inp.x[pi]), lib=lib)
    assert np.array_equal(out_b, out_a[pi]), "token permutation"


def check_rms_norm_exact_math(lib):
    """RMSNorm with a weight: out = x / sqrt(mean(x^2) + eps) * w within
    the error of its fp32 steps and one bf16 rounding (float64 reference)."""
    d = small_dims(T=32, H=512)
    x = ms.make_x(d, seed=20)
    w = ms.make_branch_norms(d, seed=20)[0]
    out = f64(oracle.rms_norm(x, w, d.eps, lib=lib))
    xf = f64(x)
    exact = xf / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + d.eps) * f64(w)
    tol = 2.0 ** -8 * np.abs(exact) + 1e-30
    assert np.all(np.abs(out - exact) <= tol), "rms_norm far from x / rms * w"


def check_rms_norm_invariances(lib):
    """eps = 0: RMSNorm(2x) == RMSNorm(x) bit for bit; doubling the weight
    doubles the output bit for bit (powers of two are exact)."""
    d = small_dims(T=16, H=256)
    x = ms.make_x(d, seed=21)
    w = ms.make_branch_norms(d, seed=21)[1]
    a = oracle.rms_norm(x, w, 0.0, lib=lib)
    b = oracle.rms_norm(ms.bf16_bits(ms.bits_to_f32(x) * 2.0), w, 0.0, lib=lib)
    assert np.array_equal(a, b), "rms_norm(2x) != rms_norm(x)"
    c = oracle.rms_norm(x, ms.bf16_bits(ms.bits_to_f32(w) * 2.0), 0.0, lib=lib)
    assert np.array_equal(f64(c), 2.0 * f64(a)), "rms_norm with 2w != 2 rms_norm"


def check_rms_norm_constant_row(lib):
    """A constant row c (eps = 0, weight 1) normalises to sign(c) exactly;
    weight w then gives w itself."""
    H = 384
    for c in (0x3F80, 0xC0A0, 0x3C23):  # 1, -5, ~0.00995
        x = np.full((2, H), c, np.uint16)
        ones = np.full(H, 0x3F80, np.uint16)
        want = 0xBF80 if c & 0x8000 else 0x3F80
        assert np.all(oracle.rms_norm(x, ones, 0.0, lib=lib) == want), f"constant row {c:#06x}"
        w = ms.make_branch_norms(small_dims(H=H), seed=22)[0]
        got = oracle.rms_norm(x, w, 0.0, lib=lib)
        sign = -1.0 if c & 0x8000 else 1.0
        assert np.array_equal(f64(got), sign * np.tile(f64(w), (2, 1))), f"constant row {c:#06x}, weight"



def check_rms_norm_rounding_golden(lib):
    """Hand-derived bits of bf16((x r) w) with x r kept in fp32 before the
    weight (golden: rms_norm_rounding.json); rounding x r to bf16 first
    gives different bits on this row."""
    g = load_golden("rms_norm_rounding.json")
    x = np.tile(_golden_row(g), (2, 1))
    w = np.full(g["H"], 0x3FC0, np.uint16)
    out = oracle.rms_norm(x, w, g["eps"], lib=lib)
    for h, want in g["out_bits"].items():
        assert np.all(out[:, int(h)] == int(want, 16)), f"rms_norm out[{h}] = {out[0, int(h)]:#06x}, golden {want}"

def check_moe_branch_wiring(lib):
    """The branch is route(residual), experts(RMSNorm(residual, pre)) and
    RMSNorm(., post) of their output, composed from the parts pinned above:
    the router reads the residual, not the normalised expert input."""
    d = small_dims(T=24, E=8, k=2)
    inp = ms.make_custom(d, seed=23)
    pre, post = ms.make_branch_norms(d, seed=23)
    out, idx, w, xe = oracle.moe_branch(inp, pre, post, taps=True, lib=lib)
    rt = oracle.route(d, inp.x, inp.router_w, inp.router_scale, inp.pes, lib=lib)
    assert np.array_equal(idx, rt["idx"]) and np.array_equal(w, rt["w"]), "branch routing != route(residual)"
    want_xe = oracle.rms_norm(inp.x, pre, d.eps, lib=lib)
    assert np.array_equal(xe, want_xe), "branch expert input != RMSNorm(residual, pre)"
    y = oracle.experts(d, want_xe, rt["idx"], rt["w"], (inp.gu_w, inp.gu_s, inp.gu_b),
                       (inp.dn_w, inp.dn_s, inp.dn_b), lib=lib)
    assert np.array_equal(out, oracle.rms_norm(y, post, d.eps, lib=lib)), "branch output != RMSNorm(experts, post)"


def check_route_q4(lib):
    """The 4-bit router equals the dense router on the dequantised weight
    bf16(S q + B), dequantised here independently (torch bf16 rounding of
    the unpacked codes), bit for bit on indices, weights and scores."""
    d = small_dims(T=32, H=256, E=16, k=4)
    inp = ms.make_custom(d, seed=24)
    rq = ms.make_router_q4(d, seed=24)
    dense = torch_bf16_bits(dense_dequant(rq[0][None], rq[1][None], rq[2][None], d.H, d.group)[0])
    a = oracle.route_q4(d, inp.x, rq, inp.router_scale, inp.pes, taps=True, lib=lib)
    b = oracle.route(d, inp.x, dense, inp.router_scale, inp.pes, taps=True, lib=lib)
    for key in ("idx", "w", "scores"):
        assert np.array_equal(a[key], b[key]), f"4-bit router != dense router on the dequantised weight: {key}"


def _dense_small(T=6, H=256, I=192, seed=25):
    return ms.make_dense(T, H=H, I=I, seed=seed)


def check_dense_mlp_brute_force(lib):
    """gate, up, m and out of every token against a dense float64 computation
    (library matmul, mpmath GeGLU, torch bf16 rounding of the dequantised
    weights): each is the nearest bf16 to its exact value."""
    dn = _dense_small()
    out, g, u, m = oracle.dense_mlp(dn.x, dn.gate, dn.up, dn.down, taps=True, lib=lib)
    wg = dense_dequant(dn.gate[0], dn.gate[1], dn.gate[2], dn.H, dn.group)
    wu = dense_dequant(dn.up[0], dn.up[1], dn.up[2], dn.H, dn.group)
    wd = dense_dequant(dn.down[0], dn.down[1], dn.down[2], dn.I, dn.group)
    x = f64(dn.x)
    assert_nearest_bf16(g, x @ wg.T, "dense gate_proj")
    assert_nearest_bf16(u, x @ wu.T, "dense up_proj")
    for t in range(dn.T):
        assert_nearest_bf16(m[t], geglu_exact(f64(g[t]), f64(u[t])), f"dense GeGLU, token {t}")
    assert_nearest_bf16(out, f64(m) @ wd.T, "dense down_proj")


def check_dense_mlp_is_single_expert(lib):
    """The dense MLP is the routed layer's one-expert, top-1 case with weight 1
    and the expert's gate_up rows = gate_proj rows then up_proj rows (the
    split at the intermediate size): bit for bit the same output."""
    dn = _dense_small(T=9, seed=26)
    d = small_dims(T=dn.T, H=dn.H, E=1, k=1, inter=dn.I)
    gu = tuple(np.concatenate([a, b])[None] for a, b in zip(dn.gate, dn.up))
    dw = tuple(a[None] for a in dn.down)
    idx = np.zeros((dn.T, 1), np.int32)
    w = np.full((dn.T, 1), 0x3F80, np.uint16)
    want = oracle.experts(d, dn.x, idx, w, gu, dw, lib=lib)
    assert np.array_equal(oracle.dense_mlp(dn.x, dn.gate, dn.up, dn.down, lib=lib), want), "dense MLP != one expert"


def check_dense_branch_wiring(lib):
    """The dense branch is RMSNorm(mlp(RMSNorm(h, pre)), post), composed
    from the parts pinned above (and not with the norms' weights exchanged)."""
    dn = _dense_small(T=7, seed=27)
    out = oracle.dense_branch(dn.x, dn.pre_w, dn.post_w, dn.gate, dn.up, dn.down, dn.eps, lib=lib)
    y = oracle.dense_mlp(oracle.rms_norm(dn.x, dn.pre_w, dn.eps, lib=lib), dn.gate, dn.up, dn.down, lib=lib)
    assert np.array_equal(out, oracle.rms_norm(y, dn.post_w, dn.eps, lib=lib)), "dense branch wiring"


def check_self_conditioning_exact_math(lib):
    """out = c / sqrt(mean(c^2) + eps) within its fp32 steps and one bf16
    rounding, for c = bf16(embeds + s) (torch's rounding of the exact sum)
    and s the pinned dense MLP of RMSNorm(signal, pre)."""
    dn = _dense_small(T=8, seed=28)
    out = f64(oracle.self_conditioning(dn.embeds, dn.x, dn.pre_w, dn.gate, dn.up, dn.down, dn.eps, lib=lib))
    s_ = oracle.dense_mlp(oracle.rms_norm(dn.x, dn.pre_w, dn.eps, lib=lib), dn.gate, dn.up, dn.down, lib=lib)
    exact_sum = f64(dn.embeds) + f64(s_)
    assert np.array_equal(exact_sum.astype(np.float32).astype(np.float64), exact_sum), "sum not exact in float32"
    c = f64(torch_bf16_bits(exact_sum.astype(np.float32)))
    exact = c / np.sqrt(np.mean(c * c, axis=1, keepdims=True) + dn.eps)
    assert np.all(np.abs(out - exact) <= 2.0 ** -8 * np.abs(exact) + 1e-30), "self-conditioning far from c / rms(c)"


def check_self_conditioning_zero_mlp(lib):
    """With an all-zero down_proj (codes, scales and biases 0) the MLP adds
    nothing, and RMSNormNoScale of a constant row c (eps = 0) is sign(c)."""
    dn = _dense_small(T=3, seed=29)
    zero = (np.zeros_like(dn.down[0]), np.zeros_like(dn.down[1]), np.zeros_like(dn.down[2]))
    emb = np.zeros((3, dn.H), np.uint16)
    for t, c in enumerate((0x3F80, 0xC0A0, 0x3C23)):  # 1, -5, ~0.00995
        emb[t] = c
    out = oracle.self_conditioning(emb, dn.x, dn.pre_w, dn.gate, dn.up, zero, 0.0, lib=lib)
    want = np.where(emb & 0x8000, 0xBF80, 0x3F80).astype(np.uint16)
    assert np.array_equal(out, want), "RMSNormNoScale of a constant row"


def check_lm_head_brute_force(lib):
    """The head's bf16 logits are the nearest bf16 to h . W^T (the table
    dequantised here, float64 matmul), and its output is cap * tanh(x / cap)
    of those logits within three fp32 ulps (three fp32 roundings; float64
    numpy tanh). h is scaled so the logits reach the softcap's saturation."""
    h, emb = ms.make_head(T=5, H=256, V=384, seed=50, h_scale=40.0)
    out, lg = oracle.lm_head(h, emb, cap=30.0, taps=True, lib=lib)
    w = dense_dequant(emb[0], emb[1], emb[2], 256, 64)
    assert_nearest_bf16(lg, f64(h) @ w.T, "head logits")
    x = f64(lg)
    assert np.abs(x).max() > 60.0, "test logits do not reach saturation"
    exact = 30.0 * np.tanh(x / 30.0)
    assert np.all(np.abs(out.astype(np.float64) - exact) <= 3 * 2.0 ** -24 * np.abs(exact) + 1e-30), \
        "head softcap far from cap * tanh(x / cap)"


def check_lm_head_symmetry_and_no_cap(lib):
    """Negating h negates the output bit for bit (every step is odd); the
    output stays within the cap; cap 0 returns the bf16 logits widened."""
    h, emb = ms.make_head(T=4, H=256, V=256, seed=51, h_scale=8.0)
    a = oracle.lm_head(h, emb, cap=30.0, lib=lib)
    b = oracle.lm_head(h ^ np.uint16(0x8000), emb, cap=30.0, lib=lib)
    assert np.array_equal(a, -b), "head(-h) != -head(h)"
    assert np.all(np.abs(a) <= 30.0), "softcapped logit beyond the cap"
    out, lg = oracle.lm_head(h, emb, cap=0.0, taps=True, lib=lib)
    assert np.array_equal(out, ms.bits_to_f32(lg)), "cap 0: output != float32(bf16 logits)"


ALL_CHECKS = [
    check_bf16_from_float, check_bf16_from_double,
    check_router_constant_row, check_router_norm_rounding_golden, check_router_zero_row, check_router_scale_invariance,
    check_router_exact_math, check_router_logits_topk, check_router_weights,
    check_dispatch,
    check_experts_brute_force, check_experts_one_hot, check_geglu_ties, check_single_expert_identity,
    check_expert_relabel, check_token_permutation,
    check_rms_norm_exact_math, check_rms_norm_invariances, check_rms_norm_constant_row, check_rms_norm_rounding_golden,
    check_moe_branch_wiring,
    check_route_q4,
    check_dense_mlp_brute_force, check_dense_mlp_is_single_expert, check_dense_branch_wiring,
    check_self_conditioning_exact_math, check_self_conditioning_zero_mlp,
    check_lm_head_brute_force, check_lm_head_symmetry_and_no_cap,
]
