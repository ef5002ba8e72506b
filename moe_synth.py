"""Seeded synthetic inputs for the routed 4-bit MoE layer.

This module is the only code shared by the CPU oracle's tests and the CUDA
path's tests and benchmark. It draws random tensors and returns their raw
bit patterns (bf16 as uint16, packed 4-bit codes as uint32). It holds none of
the layer's arithmetic: no norm, no projection, no top-k, no dequantisation.

Workloads (the MoE layer of DiffusionGemma-26B-A4B, "diffusion-gemma/model.ts",
classes DiffRouter and DiffExperts):

  tiny     T=16,   H=256,  E=8,   k=2, I=128, g=64   (parity-sized layer)
  canvas   T=256,  H=2816, E=128, k=8, I=704, g=64   (decoder canvas pass)
  decode   T=8,    same layer as canvas              (drafter / decode step)
  prefill  T=4096, same layer as canvas              (encoder prompt prefill)
  skew     T=2048, same layer, Zipf(1.2)-biased routing

Distributions: x ~ N(0,1); router weight ~ N(0, 0.05^2); router scale and
per-expert scale ~ U(0.5, 1.5); 4-bit codes ~ U{0..15} packed 8 per uint32,
low nibble first; per-group scale ~ U(0.005, 0.02); bias = -8 * scale. Every
float is rounded to bf16 (round to nearest even) before use.

Each tensor comes from its own stream, keyed by (seed, tensor name, shape),
so the canvas, decode, prefill and skew workloads share the same layer
weights and differ only in the activations.
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np


@dataclasses.dataclass(frozen=True)
class Dims:
    """Shape of one MoE layer call. bits is fixed at 4."""
    T: int
    H: int
    E: int
    k: int
    inter: int
    group: int = 64
    bits: int = 4
    eps: float = 1e-6


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: Dims
    seed: int = 0
    # Skewed routing: x gets a mean offset `skew_mu` and router row e gets
    # `skew_kappa * b_e` added, with b_e = -zipf_s * ln(rank_e).
    skew_kappa: float = 0.0
    skew_mu: float = 0.0
    zipf_s: float = 1.2


_LAYER = dict(H=2816, E=128, k=8, inter=704, group=64)

# Skew strength, calibrated once with the oracle router by
# tests/golden/calibrate_skew.py: the 13 most-loaded experts (10%) take
# 60 +- 5% of the slots and at least three experts take none.
SKEW_KAPPA = 0.00054

WORKLOADS = {
    "tiny": Workload("tiny", Dims(T=16, H=256, E=8, k=2, inter=128, group=64)),
    "canvas": Workload("canvas", Dims(T=256, **_LAYER)),
    "decode": Workload("decode", Dims(T=8, **_LAYER)),
    "prefill": Workload("prefill", Dims(T=4096, **_LAYER)),
    "skew": Workload("skew", Dims(T=2048, **_LAYER), skew_kappa=SKEW_KAPPA, skew_mu=1.0),
}


def _rng(seed: int, name: str) -> np.random.Generator:
    key = zlib.crc32(name.encode())
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, key])))


def bf16_bits(a) -> np.ndarray:
    """float array -> bf16 bit patterns (uint16), round to nearest even.

    Input preparation only: the generator states its draws in bf16.
    """
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bits_to_f32(b) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def random_words(rng: np.random.Generator, n: int) -> np.ndarray:
    """n uniform uint32 words; each is 8 independent U{0..15} codes."""
    raw = rng.bit_generator.random_raw((n + 1) // 2)
    return np.ascontiguousarray(np.asarray(raw, dtype=np.uint64).view(np.uint32)[:n])


def make_x(d: Dims, seed: int = 0, mu: float = 0.0) -> np.ndarray:
    rng = _rng(seed, f"x:{d.T}x{d.H}")
    return bf16_bits(rng.standard_normal((d.T, d.H)) + mu)


def make_router(d: Dims, seed: int = 0, kappa: float = 0.0, zipf_s: float = 1.2):
    """router_w [E,H], router_scale [H], per_expert_scale [E] as bf16 bits."""
    rng = _rng(seed, f"router:{d.E}x{d.H}")
    wr = rng.normal(0.0, 0.05, (d.E, d.H))
    scale = rng.uniform(0.5, 1.5, d.H)
    pes = rng.uniform(0.5, 1.5, d.E)
    if kappa != 0.0:
        rank = _rng(seed, f"skew-rank:{d.E}").permutation(d.E) + 1
        b = -zipf_s * np.log(rank.astype(np.float64))
        wr = wr + kappa * b[:, None]
    return bf16_bits(wr), bf16_bits(scale), bf16_bits(pes)


def make_qweight(E: int, N: int, K: int, group: int, seed: int, tag: str):
    """4-bit affine weight for E experts of an N x K linear (out = x W^T).

    Returns (w uint32 [E,N,K/8], scales bf16 [E,N,K/g], biases bf16 [E,N,K/g]).
    """
    assert K % 8 == 0 and K % group == 0
    rng = _rng(seed, f"{tag}:w:{E}x{N}x{K}")
    w = random_words(rng, E * N * (K // 8)).reshape(E, N, K // 8)
    rs = _rng(seed, f"{tag}:s:{E}x{N}x{K // group}")
    s = bf16_bits(rs.uniform(0.005, 0.02, (E, N, K // group)))
    # -8 * s is exact in bf16 (power-of-two multiple, sign flip).
    b = bf16_bits(-8.0 * bits_to_f32(s))
    return w, s, b


@dataclasses.dataclass
class LayerInputs:
    dims: Dims
    x: np.ndarray            # uint16 [T,H]
    router_w: np.ndarray     # uint16 [E,H]
    router_scale: np.ndarray  # uint16 [H]
    pes: np.ndarray          # uint16 [E]
    gu_w: np.ndarray         # uint32 [E,2I,H/8]
    gu_s: np.ndarray         # uint16 [E,2I,H/g]
    gu_b: np.ndarray         # uint16 [E,2I,H/g]
    dn_w: np.ndarray         # uint32 [E,H,I/8]
    dn_s: np.ndarray         # uint16 [E,H,I/g]
    dn_b: np.ndarray         # uint16 [E,H,I/g]


def make_layer(wl, T: int | None = None, seed: int | None = None) -> LayerInputs:
    """All inputs of one workload (optionally another token count or seed)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    d = wl.dims if T is None else dataclasses.replace(wl.dims, T=T)
    sd = wl.seed if seed is None else seed
    x = make_x(d, sd, mu=wl.skew_mu)
    wr, sc, pes = make_router(d, sd, kappa=wl.skew_kappa, zipf_s=wl.zipf_s)
    gw, gs, gb = make_qweight(d.E, 2 * d.inter, d.H, d.group, sd, "gate_up")
    dw, ds, db = make_qweight(d.E, d.H, d.inter, d.group, sd, "down")
    return LayerInputs(d, x, wr, sc, pes, gw, gs, gb, dw, ds, db)


def make_router_q4(d: Dims, seed: int = 0):
    """The router projection as a 4-bit group-64 weight (the pages'
    QuantizedLinear): (w uint32 [E, H/8], scales [E, H/g], biases [E, H/g]),
    with the experts' code, scale and bias recipe."""
    w, s, b = make_qweight(1, d.E, d.H, d.group, seed, "router")
    return w[0], s[0], b[0]


def make_branch_norms(d: Dims, seed: int = 0):
    """Weights [H] of the MoE branch's two RMS norms (pre_feedforward_layernorm_2,
    post_feedforward_layernorm_2) as bf16 bits, U(0.5, 1.5) like the router
    scale (trained RMS-norm weights are O(1) and positive)."""
    rng = _rng(seed, f"branch-norms:{d.H}")
    return bf16_bits(rng.uniform(0.5, 1.5, d.H)), bf16_bits(rng.uniform(0.5, 1.5, d.H))


# The dense MLP's intermediate size is not on the pages; the decoder-sized
# dense workloads use 2112 (three times moe_intermediate, a multiple of 64).
DENSE_INTER = 2112


@dataclasses.dataclass
class DenseInputs:
    """Inputs of the dense 4-bit GeGLU MLP and the two calls built on it."""
    T: int
    H: int
    I: int
    group: int
    eps: float
    x: np.ndarray        # uint16 [T,H]: the MLP input, the dense branch's h, or the self-conditioning signal
    embeds: np.ndarray   # uint16 [T,H]: SelfConditioning's inputs_embeds
    gate: tuple          # (w uint32 [I,H/8], scales [I,H/g], biases [I,H/g])
    up: tuple            # same shapes as gate
    down: tuple          # (w uint32 [H,I/8], scales [H,I/g], biases [H,I/g])
    pre_w: np.ndarray    # uint16 [H]: preFfNorm / SelfConditioning.preNorm weight
    post_w: np.ndarray   # uint16 [H]: postFfNorm1 weight


def make_dense(T: int, H: int = 2816, I: int = DENSE_INTER, seed: int = 0, group: int = 64,
               eps: float = 1e-6) -> DenseInputs:
    """Dense-MLP inputs with the layer's distributions: activations and
    embeddings ~ N(0,1), the experts' 4-bit code, scale and bias recipe for the
    three linears, norm weights ~ U(0.5, 1.5)."""
    d = Dims(T=T, H=H, E=1, k=1, inter=I, group=group, eps=eps)
    x = make_x(d, seed)
    embeds = bf16_bits(_rng(seed, f"embeds:{T}x{H}").standard_normal((T, H)))
    tri = lambda a: (a[0][0], a[1][0], a[2][0])
    gate = tri(make_qweight(1, I, H, group, seed, "dense_gate"))
    up = tri(make_qweight(1, I, H, group, seed, "dense_up"))
    down = tri(make_qweight(1, H, I, group, seed, "dense_down"))
    rng = _rng(seed, f"dense-norms:{H}")
    pre_w, post_w = bf16_bits(rng.uniform(0.5, 1.5, H)), bf16_bits(rng.uniform(0.5, 1.5, H))
    return DenseInputs(T, H, I, group, eps, x, embeds, gate, up, down, pre_w, post_w)


# The vocabulary size is not on the pages; the image token id 258880 bounds
# it from below, and the head workloads take 2^18 = 262144.
VOCAB = 262144


def make_head(T: int, H: int = 2816, V: int = VOCAB, seed: int = 0, group: int = 64, h_scale: float = 1.0):
    """Inputs of the tied 4-bit head: h [T,H] bf16 bits ~ N(0, h_scale^2) (a
    final-normed hidden state), the embedding table [V,H] as a 4-bit group-g
    weight with the experts' code, scale and bias recipe."""
    h = bf16_bits(_rng(seed, f"head-h:{T}x{H}").standard_normal((T, H)) * h_scale)
    w, s, b = make_qweight(1, V, H, group, seed, "embed")
    return h, (w[0], s[0], b[0])


def make_custom(d: Dims, seed: int = 0, **skew) -> LayerInputs:
    """Inputs for an arbitrary layer shape with the standard distributions."""
    return make_layer(Workload("custom", d, seed=seed, **skew))
