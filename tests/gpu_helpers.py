"""Helpers for the GPU parity tests: run libmoe through its C ABI on seeded
inputs and compare with the CPU oracle.

Comparison rules (stated once here, used by every GPU test):
  * routing indices: the set of k experts per token is bit-exact, except on
    "near-tie" tokens where the oracle's exact k-th and (k+1)-th logits
    differ by less than 1e-3 relative; those tokens are counted and must
    still hold a valid top-k (one swap, between experts inside the band).
    The pages' top-k (argpartition) is an unordered set; the emitted order
    must be score descending with ties to the lower id, allowing a swap of
    neighbours whose oracle scores are one bf16 ulp apart;
  * routing weights: within 1 bf16 ulp, per (token, expert);
  * permutation, offsets, inverse: bit-exact;
  * layer output: |gpu - oracle| <= max(2e-2 * RMS(oracle), 1 bf16 ulp of
    the oracle value) per element, and RMS(gpu - oracle) <= 1e-3 * RMS.
    The bf16 output cannot resolve differences below its own ulp, and at
    |out| >= ~3 RMS one ulp already exceeds 2e-2 RMS, so a single rounding
    flip there (fp32 vs exact accumulation order) is allowed; the count of
    elements beyond the strict 2e-2 RMS bound is reported.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import bit_quantized_moe_layer_gb300 as moe
import moe_synth as ms
import oracle

NEAR_TIE_REL = 1e-3


def f64(bits) -> np.ndarray:
    return ms.bits_to_f32(bits).astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def dev16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).to(device)


def dev32(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32).copy()).to(device)


def host16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


@dataclasses.dataclass
class GpuLayer:
    d: moe.Dims
    x: torch.Tensor
    layer: moe.DeviceLayer


def upload(inp: ms.LayerInputs) -> GpuLayer:
    return GpuLayer(moe.dims_of(inp.dims), dev16(inp.x), moe.to_device_layer(inp))


def gpu_route(g: GpuLayer):
    T, k = g.d.T, g.d.k
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.int16, device="cuda")
    moe.moe_route(g.d, g.x, g.layer.router_w, g.layer.router_scale, g.layer.pes, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), host16(w)


def gpu_dispatch(d: moe.Dims, idx: np.ndarray):
    S = d.T * d.k
    idx_d = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda()
    perm = torch.full((max(S, 1),), -1, dtype=torch.int32, device="cuda")
    inv = torch.full((max(S, 1),), -1, dtype=torch.int32, device="cuda")
    off = torch.full((d.E + 1,), -1, dtype=torch.int32, device="cuda")
    moe.moe_dispatch(d, idx_d, perm, off, inv)
    torch.cuda.synchronize()
    return perm.cpu().numpy()[:S], off.cpu().numpy(), inv.cpu().numpy()[:S]


def gpu_experts(g: GpuLayer, idx: np.ndarray, w: np.ndarray, workspace=None):
    idx_d = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda()
    w_d = dev16(w)
    out = torch.empty((g.d.T, g.d.H), dtype=torch.int16, device="cuda")
    ws_bytes = 0 if workspace is None else workspace.numel()
    moe.moe_experts(g.d, g.x, idx_d, w_d, g.layer.gate_up, g.layer.down, out, workspace, ws_bytes)
    torch.cuda.synchronize()
    return host16(out)


def gpu_forward(g: GpuLayer, workspace=None):
    T, k = g.d.T, g.d.k
    out = torch.empty((T, g.d.H), dtype=torch.int16, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.int16, device="cuda")
    ws_bytes = 0 if workspace is None else workspace.numel()
    moe.moe_forward(g.d, g.x, g.layer.router_w, g.layer.router_scale, g.layer.pes, g.layer.gate_up,
                    g.layer.down, out, idx, w, workspace, ws_bytes)
    torch.cuda.synchronize()
    return host16(out), idx.cpu().numpy(), host16(w)


def near_tie_rows(logits: np.ndarray, scores: np.ndarray, k: int):
    """Tokens whose oracle k-th and (k+1)-th experts (in the canonical order)
    are a near tie. Returns two masks:
      band       the exact logits are within NEAR_TIE_REL of each other (the
                 stated exemption);
      score_tie  outside the band, but the two bf16 scores are equal: the
                 tie is decided by the lower id on both sides, so a GPU
                 difference there needs a GPU score that rounded the other
                 way, which check_routing only accepts next to a bf16
                 rounding midpoint (midpoint_logit)."""
    T, E = scores.shape
    if k >= E:
        z = np.zeros(T, bool)
        return z, z
    s = f64(scores)
    order = np.lexsort((np.broadcast_to(np.arange(E), (T, E)), -s), axis=1)
    lk = np.take_along_axis(logits, order[:, k - 1:k], 1)[:, 0]
    lk1 = np.take_along_axis(logits, order[:, k:k + 1], 1)[:, 0]
    sk = np.take_along_axis(s, order[:, k - 1:k], 1)[:, 0]
    sk1 = np.take_along_axis(s, order[:, k:k + 1], 1)[:, 0]
    band = np.abs(lk - lk1) <= NEAR_TIE_REL * np.maximum(np.abs(lk), np.abs(lk1))
    return band, (sk == sk1) & ~band


MIDPOINT_REL = 2.0 ** -20


def accum_steps(H: int) -> int:
    """fp32 accumulation bound of one GPU router logit, in units of 2^-24
    times the sum of |products|. The row router accumulates all H products in
    the tensor core's fp32 accumulator, 16 products a step: H/16 steps plus 16
    inside a step. The cluster router's bound is smaller (each of 8 CTAs
    accumulates H/8 products, then the 8 partials are added: H/128 + 24), so
    this one covers both kernels."""
    return H // 16 + 16


def midpoint_logit(v: float, abs_dot: float | None = None, steps: int = 64) -> bool:
    """Whether the exact logit v lies close enough to a bf16 rounding midpoint
    that an fp32-accumulated score may round the other way: within
    steps * 2^-24 * sum|products| (abs_dot) of it, or within MIDPOINT_REL of
    |v| when the products are not known."""
    u = float(bf16_ulp(np.array([v]))[0])
    mid = np.floor(abs(v) / u) * u + u / 2
    window = steps * 2.0 ** -24 * abs_dot if abs_dot is not None else MIDPOINT_REL * abs(v)
    return abs(abs(v) - mid) <= window


def softmax_near_midpoint(scores: np.ndarray) -> np.ndarray:
    """For the picked bf16 scores of one token: whether each fp32 softmax
    probability p lies within 4 fp32 ulps of a bf16 rounding midpoint. There
    the device's expf and the host's may round bf16(p) one ulp apart (each
    within its stated error), and w = bf16(bf16(p) * pes) then differs by up
    to two ulps (one ulp of p scaled by pes <= 1.5, and the final rounding)."""
    e = np.exp(scores - scores.max())
    p = e / e.sum()
    ulp = bf16_ulp(p)
    mid = np.floor(p / ulp) * ulp + ulp / 2
    return np.abs(p - mid) <= 4 * 2.0 ** -24 * np.abs(p)


def check_routing(d, ref, idx, w, router_w=None):
    """Compare GPU routing with the oracle's. The pages' top-k (argpartition)
    is an unordered set, so sets are compared per token and the weights per
    (token, expert); the emitted order must be descending in the oracle's
    scores except between experts whose exact logits are within the near-tie
    band. A token whose set differs must be a near tie (one swap, between its
    k-th and (k+1)-th experts): inside the band, or an equal-score tie whose
    two exact logits include one next to a bf16 rounding midpoint (the
    window is the GPU's fp32 accumulation bound when the router weight
    router_w [E,H] bf16 bits is given, with the oracle's normed input).
    Returns the counts {band, score_tie, differ, differ_score_tie}."""
    band, score_tie = near_tie_rows(ref["logits"], ref["scores"], d.k)
    T, k = idx.shape
    lg = ref["logits"]
    in_band = lambda a, b: abs(a - b) <= NEAR_TIE_REL * max(abs(a), abs(b)) + 1e-12
    differ = differ_score_tie = 0
    for t in range(T):
        gs, os_ = set(idx[t].tolist()), set(ref["idx"][t].tolist())
        assert len(gs) == k and all(0 <= e < d.E for e in gs), f"token {t}: invalid expert ids {idx[t]}"
        if gs != os_:
            differ += 1
            assert band[t] or score_tie[t], \
                f"routing differs on non-tie token {t}: gpu {sorted(gs)} oracle {sorted(os_)}"
            extra, missing = gs - os_, os_ - gs
            assert len(extra) == 1 and len(missing) == 1, f"near-tie token {t}: more than one swap"
            ex_, mi_ = extra.pop(), missing.pop()
            if in_band(lg[t, ex_], lg[t, mi_]):
                continue
            sc_ = f64(ref["scores"][t])
            assert sc_[ex_] == sc_[mi_], f"near-tie token {t}: swap outside the band"
            ad = [None, None]
            if router_w is not None and "normed" in ref:
                nt = np.abs(f64(ref["normed"][t]))
                ad = [float(nt @ np.abs(f64(router_w[e]))) for e in (ex_, mi_)]
            steps = accum_steps(d.H)
            assert midpoint_logit(lg[t, ex_], ad[0], steps) or midpoint_logit(lg[t, mi_], ad[1], steps), \
                (f"token {t}: equal-score swap ({ex_} for {mi_}) with neither exact logit near a bf16 "
                 f"rounding midpoint: {lg[t, ex_]!r}, {lg[t, mi_]!r}")
            differ_score_tie += 1
            continue
        sc = f64(ref["scores"][t])
        for j in range(k - 1):  # emitted order: score descending, ties to the lower id
            a, b = idx[t, j], idx[t, j + 1]
            ok = sc[a] > sc[b] or (sc[a] == sc[b] and a < b)
            # a one-ulp rounding flip of a GPU score may swap two neighbours
            ok = ok or abs(sc[a] - sc[b]) <= float(bf16_ulp(np.array([max(abs(sc[a]), abs(sc[b]))]))[0])
            assert ok, f"token {t}: order {idx[t]} vs oracle {ref['idx'][t]}"
        gw = dict(zip(idx[t].tolist(), f64(w[t]).tolist()))
        p_mid = softmax_near_midpoint(f64(ref["scores"][t][ref["idx"][t]]))
        for j, e in enumerate(ref["idx"][t].tolist()):
            o = float(f64(ref["w"][t, j]))
            ulps = 2 if p_mid[j] else 1
            assert abs(gw[e] - o) <= ulps * float(bf16_ulp(np.array([o]))[0]) + 1e-30, \
                f"token {t} expert {e}: weight {gw[e]} vs oracle {o}"
    return dict(band=int(band.sum()), score_tie=int(score_tie.sum()), differ=differ,
                differ_score_tie=differ_score_tie)


def workspace_dispatch(d, ws: torch.Tensor):
    """perm, offsets and inv that the last routed call left in the caller
    workspace `ws` (uint8 tensor), at the library's own workspace map."""
    m = moe.workspace_map(d)
    S = d.T * d.k
    host = ws.cpu().numpy()
    take = lambda off, n: host[off:off + 4 * n].view(np.int32).copy()
    return take(m.perm, S), take(m.offsets, d.E + 1), take(m.inv, S)


def bf16_round(v) -> np.ndarray:
    """float32-exact values -> nearest bf16 (torch's rounding), as float64."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def compare_out(gpu_bits: np.ndarray, ref_bits: np.ndarray, what: str = "out", explain=None) -> dict:
    """Layer output against the oracle's. Tier 1, per element:
    |gpu - oracle| <= max(2e-2 RMS, 1 bf16 ulp of the oracle value). An
    element beyond tier 1 must be explained by the accumulation order alone
    (tier 2): out = bf16(sum_j bf16(y_j w_j)), and each bf16 y_j that the GPU
    accumulates in fp32 may round one ulp away from the oracle's exactly
    rounded y_j, so |gpu - oracle| <= ulp(out) + sum_j (w_j ulp(y_j) +
    ulp(bf16(y_j w_j)) + |y_j| dw_j), dw_j the routing-weight difference.
    `explain(rows)` returns the oracle's y [rows, k, H], w [rows, k] and the
    weight differences dw [rows, k] of those token rows; without it tier 1
    is final. The RMS error stays <= 1e-3 RMS."""
    g, o = f64(gpu_bits), f64(ref_bits)
    rms = float(np.sqrt(np.mean(o * o)))
    err = np.abs(g - o)
    tol = np.maximum(2e-2 * rms, bf16_ulp(o))
    bad = np.argwhere(err > tol)
    stats = dict(rms=rms, max_err_over_rms=float(err.max() / rms) if err.size else 0.0,
                 rms_err_over_rms=float(np.sqrt(np.mean(err ** 2)) / rms) if err.size else 0.0,
                 n_strict=int((err > 2e-2 * rms).sum()), n_diff=int((err > 0).sum()), n=int(err.size),
                 n_tier2=int(len(bad)))
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    if len(bad):
        first = tuple(bad[0])
        msg = (f"{what}: {len(bad)} elements beyond max(2e-2 RMS, 1 ulp); first {first}: gpu {g[first]} "
               f"oracle {o[first]} (rms {rms}) {stats}")
        assert explain is not None, msg
        rows = np.unique(bad[:, 0])
        y, w, dw = explain(rows)
        at = {r: i for i, r in enumerate(rows)}
        for r, h in bad:
            i = at[r]
            yj, wj = y[i, :, h], w[i]
            p = bf16_round(yj * wj)
            bound = float(bf16_ulp(np.array([o[r, h]]))[0] + np.sum(wj * bf16_ulp(yj) + bf16_ulp(p) +
                                                                   np.abs(yj) * dw[i]))
            assert err[r, h] <= bound, f"{msg}; element ({r}, {h}) error {err[r, h]} > tier-2 bound {bound}"
    assert stats["rms_err_over_rms"] <= 1e-3, f"{what}: RMS error too large {stats}"
    return stats


def explainer(inp: ms.LayerInputs, idx: np.ndarray, w: np.ndarray, w_gpu: np.ndarray | None = None):
    """The oracle's per-slot expert outputs y and routing weights for given
    token rows (and the GPU's routing-weight differences), for compare_out's
    tier-2 check."""
    d = inp.dims

    def f(rows):
        sub = dataclasses.replace(d, T=len(rows))
        _, _, _, y = oracle.experts(sub, inp.x[rows], idx[rows], w[rows], (inp.gu_w, inp.gu_s, inp.gu_b),
                                    (inp.dn_w, inp.dn_s, inp.dn_b), taps=True)
        wf = f64(w[rows])
        dw = np.zeros_like(wf) if w_gpu is None else np.abs(f64(w_gpu[rows]) - wf)
        return f64(y).reshape(len(rows), d.k, d.H), wf, dw
    return f


def oracle_route(inp: ms.LayerInputs):
    d = inp.dims
    return oracle.route(d, inp.x, inp.router_w, inp.router_scale, inp.pes, taps=True)


def oracle_experts_rows(inp: ms.LayerInputs, idx: np.ndarray, w: np.ndarray, rows: np.ndarray | None = None):
    """Oracle experts output for the given token rows (all if None)."""
    d = inp.dims
    x = inp.x
    if rows is not None:
        d = dataclasses.replace(d, T=len(rows))
        x, idx, w = x[rows], idx[rows], w[rows]
    return oracle.experts(d, x, idx, w, (inp.gu_w, inp.gu_s, inp.gu_b), (inp.dn_w, inp.dn_s, inp.dn_b))


def compare_normed_out(got, want, c, w, eps, what, c_err=None):
    """Output of a post norm out = bf16((c * rs_t) [* w]), rs_t =
    rsqrt(mean(c^2) + eps), against the oracle's, for the oracle's input row
    c. A GPU input within c_err of c (default: the layer bound 2e-2 RMS(c)
    plus a one-ulp rounding difference of c) is carried by that scaling, and
    the output rounds once more: |out - ref| <= c_err rs_t |w[h]| + ulp(ref).
    The RMS error stays below 1e-3 of the RMS."""
    g, o, cc = f64(got), f64(want), f64(c)
    wv = np.ones((1, cc.shape[1])) if w is None else np.abs(f64(w))[None, :]
    rs = 1.0 / np.sqrt(np.mean(cc * cc, axis=1, keepdims=True) + eps)
    if c_err is None:
        c_err = 2e-2 * float(np.sqrt(np.mean(cc * cc))) + bf16_ulp(cc)
    err = np.abs(g - o)
    tol = c_err * rs * wv + bf16_ulp(o)
    bad = np.flatnonzero((err > tol).ravel())
    stats = dict(max_err_over_tol=float((err / tol).max()) if err.size else 0.0,
                 rms_err_over_rms=float(np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(o ** 2))) if err.size else 0.0)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    assert bad.size == 0, f"{what}: {bad.size} elements beyond tolerance {stats}"
    assert stats["rms_err_over_rms"] <= 1e-3, f"{what}: RMS error too large {stats}"
    return stats
