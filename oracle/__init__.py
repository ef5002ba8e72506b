"""CPU oracle for the routed 4-bit MoE layer -- TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check and bench.py's CPU-baseline / reference leg may
import this package. The CUDA library never links, loads or calls it, and
this package never touches the CUDA library.

`build()` compiles moe_oracle.c (plain C, OpenMP) into liboracle.so next to
it. The functions below marshal numpy arrays (bf16 carried as uint16 bit
patterns) into the C entry points and back.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("inter", ctypes.c_int32), ("group", ctypes.c_int32),
                ("bits", ctypes.c_int32), ("eps", ctypes.c_float)]


def compile_cmd(out: str = LIB_PATH, mutant: int = 0) -> list[str]:
    return ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
            f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", out, "-lm"]


def build(force: bool = False) -> str:
    """Compile the oracle if it is missing or older than its source."""
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(_SRC):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(compile_cmd(tmp), check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def load(path: str | None = None):
    """Load (building if needed) and return the oracle's ctypes handle."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _declare(lib):
    P = ctypes.c_void_p
    lib.oracle_bf16_from_float.argtypes = [ctypes.c_float]
    lib.oracle_bf16_from_float.restype = ctypes.c_uint16
    lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
    lib.oracle_bf16_from_double.restype = ctypes.c_uint16
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_route.argtypes = [ctypes.POINTER(_Dims)] + [P] * 9 + [ctypes.c_int]
    lib.oracle_route.restype = ctypes.c_int
    lib.oracle_dispatch.argtypes = [ctypes.c_int32] * 3 + [P] * 4
    lib.oracle_dispatch.restype = ctypes.c_int
    lib.oracle_experts.argtypes = [ctypes.POINTER(_Dims)] + [P] * 13 + [ctypes.c_int]
    lib.oracle_experts.restype = ctypes.c_int
    lib.oracle_forward.argtypes = [ctypes.POINTER(_Dims)] + [P] * 13 + [ctypes.c_int]
    lib.oracle_forward.restype = ctypes.c_int
    lib.oracle_route_q4.argtypes = [ctypes.POINTER(_Dims)] + [P] * 10 + [ctypes.c_int]
    lib.oracle_route_q4.restype = ctypes.c_int
    lib.oracle_rms_norm.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_float, P, P, P]
    lib.oracle_rms_norm.restype = ctypes.c_int
    lib.oracle_moe_branch.argtypes = [ctypes.POINTER(_Dims)] + [P] * 16 + [ctypes.c_int]
    lib.oracle_moe_branch.restype = ctypes.c_int
    Q = ctypes.POINTER(_QLinear)
    lib.oracle_dense_mlp.argtypes = [ctypes.c_int32] * 4 + [P, Q, Q, Q] + [P] * 4 + [ctypes.c_int]
    lib.oracle_dense_mlp.restype = ctypes.c_int
    lib.oracle_dense_branch.argtypes = [ctypes.c_int32] * 4 + [ctypes.c_float, P, P, P, Q, Q, Q, P, ctypes.c_int]
    lib.oracle_dense_branch.restype = ctypes.c_int
    lib.oracle_self_conditioning.argtypes = [ctypes.c_int32] * 4 + [ctypes.c_float, P, P, P, Q, Q, Q, P,
                                                                    ctypes.c_int]
    lib.oracle_self_conditioning.restype = ctypes.c_int
    lib.oracle_lm_head.argtypes = [ctypes.c_int32] * 4 + [ctypes.c_float, P, Q, P, P, ctypes.c_int]
    lib.oracle_lm_head.restype = ctypes.c_int
    return lib


class _QLinear(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("s", ctypes.c_void_p), ("b", ctypes.c_void_p)]


def _qlinear(q):
    """(w uint32 [N, K/8], scales [N, K/g], biases [N, K/g]) -> (struct, arrays kept alive)."""
    arrs = (_c(q[0], np.uint32), _c(q[1], np.uint16), _c(q[2], np.uint16))
    return _QLinear(*[a.ctypes.data for a in arrs]), arrs


def _dims(d) -> _Dims:
    return _Dims(d.T, d.H, d.E, d.k, d.inter, d.group, d.bits, d.eps)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def max_threads(lib=None) -> int:
    return (lib or load()).oracle_max_threads()


def bf16_from_float(f: float, lib=None) -> int:
    return int((lib or load()).oracle_bf16_from_float(f))


def bf16_from_double(d: float, lib=None) -> int:
    return int((lib or load()).oracle_bf16_from_double(d))


def route(d, x, router_w, router_scale, pes, taps: bool = False, nthreads: int = 0, lib=None):
    """DiffRouter.forward. Returns dict(idx [T,k] int32, w [T,k] bf16 bits
    [, normed [T,H], logits [T,E] float64, scores [T,E] bf16 bits])."""
    lib = lib or load()
    x = _c(x, np.uint16)
    idx = np.zeros((d.T, d.k), np.int32)
    w = np.zeros((d.T, d.k), np.uint16)
    normed = np.zeros((d.T, d.H), np.uint16) if taps else None
    logits = np.zeros((d.T, d.E), np.float64) if taps else None
    scores = np.zeros((d.T, d.E), np.uint16) if taps else None
    dims = _dims(d)
    args = [_c(router_w, np.uint16), _c(router_scale, np.uint16), _c(pes, np.uint16)]
    rc = lib.oracle_route(ctypes.byref(dims), _p(x), *[_p(a) for a in args], _p(idx), _p(w),
                          _p(normed), _p(logits), _p(scores), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_route rejected the sizes ({rc})")
    out = dict(idx=idx, w=w)
    if taps:
        out.update(normed=normed, logits=logits, scores=scores)
    return out


def dispatch(T: int, k: int, E: int, idx, lib=None):
    """Stable counting sort of the flat slots by expert: (perm, offsets, inv)."""
    lib = lib or load()
    idx = _c(idx, np.int32).reshape(-1)
    perm = np.zeros(T * k, np.int32)
    inv = np.zeros(T * k, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    rc = lib.oracle_dispatch(T, k, E, _p(idx), _p(perm), _p(offsets), _p(inv))
    if rc != 0:
        raise ValueError("oracle_dispatch: expert id out of range")
    return perm, offsets, inv


def experts(d, x, idx, w, gu, dn, taps: bool = False, nthreads: int = 0, lib=None):
    """DiffExperts.forward. gu/dn are (w uint32, scales, biases) triples.
    Returns out [T,H] bf16 bits, or (out, z, m, y) with per-slot taps."""
    lib = lib or load()
    S = d.T * d.k
    out = np.zeros((d.T, d.H), np.uint16)
    z = np.zeros((S, 2 * d.inter), np.uint16) if taps else None
    m = np.zeros((S, d.inter), np.uint16) if taps else None
    y = np.zeros((S, d.H), np.uint16) if taps else None
    dims = _dims(d)
    arrs = [_c(x, np.uint16), _c(idx, np.int32), _c(w, np.uint16),
            _c(gu[0], np.uint32), _c(gu[1], np.uint16), _c(gu[2], np.uint16),
            _c(dn[0], np.uint32), _c(dn[1], np.uint16), _c(dn[2], np.uint16)]
    rc = lib.oracle_experts(ctypes.byref(dims), *[_p(a) for a in arrs], _p(out), _p(z), _p(m),
                            _p(y), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_experts rejected the inputs ({rc})")
    return (out, z, m, y) if taps else out


def forward(inp, nthreads: int = 0, lib=None):
    """Router then experts on one x. `inp` is a moe_synth.LayerInputs."""
    lib = lib or load()
    d = inp.dims
    out = np.zeros((d.T, d.H), np.uint16)
    idx = np.zeros((d.T, d.k), np.int32)
    w = np.zeros((d.T, d.k), np.uint16)
    dims = _dims(d)
    arrs = [inp.x, inp.router_w, inp.router_scale, inp.pes, inp.gu_w, inp.gu_s, inp.gu_b,
            inp.dn_w, inp.dn_s, inp.dn_b]
    arrs = [np.ascontiguousarray(a) for a in arrs]
    rc = lib.oracle_forward(ctypes.byref(dims), *[_p(a) for a in arrs], _p(out), _p(idx), _p(w),
                            nthreads)
    if rc != 0:
        raise ValueError(f"oracle_forward rejected the inputs ({rc})")
    return out, idx, w


def rms_norm(x, weight, eps: float, lib=None):
    """RMSNorm with a weight (the decoder layer's plain nn.RMSNorm): x [T,H]
    and weight [H] bf16 bits -> [T,H] bf16 bits."""
    lib = lib or load()
    x = _c(x, np.uint16)
    T, H = x.shape
    out = np.zeros((T, H), np.uint16)
    rc = lib.oracle_rms_norm(T, H, ctypes.c_float(eps), _p(x), _p(_c(weight, np.uint16)), _p(out))
    if rc != 0:
        raise ValueError(f"oracle_rms_norm rejected the inputs ({rc})")
    return out


def moe_branch(inp, pre_norm_w, post_norm_w, taps: bool = False, nthreads: int = 0, lib=None):
    """The decoder layer's MoE branch: route on the residual (inp.x), experts
    on preFfNorm2(residual), postFfNorm2 of their combined output. Returns
    (out, idx, w[, expert input])."""
    lib = lib or load()
    d = inp.dims
    out = np.zeros((d.T, d.H), np.uint16)
    idx = np.zeros((d.T, d.k), np.int32)
    w = np.zeros((d.T, d.k), np.uint16)
    xe = np.zeros((d.T, d.H), np.uint16) if taps else None
    dims = _dims(d)
    arrs = [inp.x, inp.router_w, inp.router_scale, inp.pes, pre_norm_w, post_norm_w, inp.gu_w, inp.gu_s,
            inp.gu_b, inp.dn_w, inp.dn_s, inp.dn_b]
    arrs = [np.ascontiguousarray(a) for a in arrs]
    rc = lib.oracle_moe_branch(ctypes.byref(dims), *[_p(a) for a in arrs], _p(out), _p(idx), _p(w),
                               _p(xe) if taps else None, nthreads)
    if rc != 0:
        raise ValueError(f"oracle_moe_branch rejected the inputs ({rc})")
    return (out, idx, w, xe) if taps else (out, idx, w)


def route_q4(d, x, rq, router_scale, pes, taps: bool = False, nthreads: int = 0, lib=None):
    """DiffRouter.forward with the 4-bit group-64 projection: rq = (w uint32
    [E, H/8], scales [E, H/g], biases [E, H/g]). Returns dict(idx, w[, logits,
    scores])."""
    lib = lib or load()
    x = _c(x, np.uint16)
    idx = np.zeros((d.T, d.k), np.int32)
    w = np.zeros((d.T, d.k), np.uint16)
    logits = np.zeros((d.T, d.E), np.float64) if taps else None
    scores = np.zeros((d.T, d.E), np.uint16) if taps else None
    dims = _dims(d)
    args = [_c(rq[0], np.uint32), _c(rq[1], np.uint16), _c(rq[2], np.uint16), _c(router_scale, np.uint16),
            _c(pes, np.uint16)]
    rc = lib.oracle_route_q4(ctypes.byref(dims), _p(x), *[_p(a) for a in args], _p(idx), _p(w),
                             _p(logits) if taps else None, _p(scores) if taps else None, nthreads)
    if rc != 0:
        raise ValueError(f"oracle_route_q4 rejected the inputs ({rc})")
    out = dict(idx=idx, w=w)
    if taps:
        out.update(logits=logits, scores=scores)
    return out


def dense_mlp(x, gate, up, down, group: int = 64, taps: bool = False, nthreads: int = 0, lib=None):
    """The dense 4-bit GeGLU MLP (SelfConditioning's three QuantizedLinears and
    geglu; the decoder layer's GegluMLP). gate, up: (w [I, H/8], scales, biases),
    down: (w [H, I/8], ...). Returns out [T,H] bf16 bits, or (out, gate, up, m)
    with the per-token [T,I] taps."""
    lib = lib or load()
    x = _c(x, np.uint16)
    T, H = x.shape
    I = np.asarray(gate[0]).shape[0]
    out = np.zeros((T, H), np.uint16)
    tg, tu, tm = ((np.zeros((T, I), np.uint16) for _ in range(3)) if taps else (None, None, None))
    (qg, ag), (qu, au), (qd, ad) = _qlinear(gate), _qlinear(up), _qlinear(down)
    rc = lib.oracle_dense_mlp(T, H, I, group, _p(x), ctypes.byref(qg), ctypes.byref(qu), ctypes.byref(qd), _p(out),
                              _p(tg), _p(tu), _p(tm), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_dense_mlp rejected the inputs ({rc})")
    return (out, tg, tu, tm) if taps else out


def dense_branch(h, pre_norm_w, post_norm_w, gate, up, down, eps: float, group: int = 64, nthreads: int = 0,
                 lib=None):
    """The decoder layer's dense branch: postFfNorm1(mlp(preFfNorm(h)))."""
    lib = lib or load()
    h = _c(h, np.uint16)
    T, H = h.shape
    I = np.asarray(gate[0]).shape[0]
    out = np.zeros((T, H), np.uint16)
    (qg, ag), (qu, au), (qd, ad) = _qlinear(gate), _qlinear(up), _qlinear(down)
    pre, post = _c(pre_norm_w, np.uint16), _c(post_norm_w, np.uint16)
    rc = lib.oracle_dense_branch(T, H, I, group, ctypes.c_float(eps), _p(h), _p(pre), _p(post), ctypes.byref(qg),
                                 ctypes.byref(qu), ctypes.byref(qd), _p(out), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_dense_branch rejected the inputs ({rc})")
    return out


def self_conditioning(embeds, signal, pre_norm_w, gate, up, down, eps: float, group: int = 64, nthreads: int = 0,
                      lib=None):
    """SelfConditioning.forward: RMSNormNoScale(embeds + mlp(preNorm(signal)))."""
    lib = lib or load()
    embeds, signal = _c(embeds, np.uint16), _c(signal, np.uint16)
    T, H = signal.shape
    assert embeds.shape == (T, H)
    I = np.asarray(gate[0]).shape[0]
    out = np.zeros((T, H), np.uint16)
    (qg, ag), (qu, au), (qd, ad) = _qlinear(gate), _qlinear(up), _qlinear(down)
    pre = _c(pre_norm_w, np.uint16)
    rc = lib.oracle_self_conditioning(T, H, I, group, ctypes.c_float(eps), _p(embeds), _p(signal), _p(pre),
                                      ctypes.byref(qg), ctypes.byref(qu), ctypes.byref(qd), _p(out), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_self_conditioning rejected the inputs ({rc})")
    return out


def lm_head(h, embed, cap: float = 30.0, group: int = 64, taps: bool = False, nthreads: int = 0, lib=None):
    """The tied 4-bit head and its fp32 softcap: h [T,H] bf16 bits, embed =
    (w uint32 [V, H/8], scales [V, H/g], biases [V, H/g]). Returns out
    [T,V] float32, or (out, logits bf16 bits [T,V])."""
    lib = lib or load()
    h = _c(h, np.uint16)
    T, H = h.shape
    V = np.asarray(embed[0]).shape[0]
    out = np.zeros((T, V), np.float32)
    lg = np.zeros((T, V), np.uint16) if taps else None
    q, keep = _qlinear(embed)
    rc = lib.oracle_lm_head(T, H, V, group, ctypes.c_float(cap), _p(h), ctypes.byref(q), _p(out), _p(lg), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_lm_head rejected the inputs ({rc})")
    return (out, lg) if taps else out
