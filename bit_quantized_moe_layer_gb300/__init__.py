"""Python binding of libmoe, the GB300 (sm_103a) routed 4-bit MoE layer.

Argument marshalling only: every function here checks tensor shapes and
dtypes, takes raw pointers and calls the same-named C entry point of
libmoe.so (include/moe.h). Every step of the layer runs in libmoe's CUDA
kernels; there is no Python or CPU fallback. If the library is missing the
calls raise.

bf16 tensors may be torch.bfloat16 or their uint16/int16 bit patterns.
The 4-bit weights of one SwitchLinear are a (w, scales, biases) triple:
w int32/uint32 [E, N, K/8], scales and biases bf16 [E, N, K/64].
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

STAGES = ("route", "dispatch", "gather", "gate_up", "down", "combine")
STATUS = {0: "ok", 1: "null pointer", 2: "bad shape", 3: "pointer not 16-byte aligned",
          4: "unsupported configuration", 5: "workspace too small", 6: "CUDA error",
          7: "kernel wait timed out", 8: "no usable GPU (needs compute capability 10.3, sm_103a)"}

# Every function the public header declares.
EXPORTS = ("moe_status_str", "moe_workspace_bytes", "moe_workspace_map_of", "moe_route", "moe_dispatch", "moe_experts",
           "moe_experts_noalloc", "moe_forward", "moe_forward_branch", "moe_forward_hostio", "moe_route_q4",
           "moe_forward_q4router", "moe_dense_mlp", "moe_dense_branch", "moe_self_conditioning", "moe_lm_head",
           "moe_set_small_t_path", "moe_set_router_path", "moe_timing_enable",
           "moe_timing_read",
           "moe_launches_per_forward", "moe_device_error")


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {STATUS.get(status, status)} (status {status})")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("inter", ctypes.c_int32), ("group", ctypes.c_int32),
                ("bits", ctypes.c_int32), ("eps", ctypes.c_float)]


class WorkspaceMap(ctypes.Structure):
    _fields_ = [("idx", ctypes.c_size_t), ("w", ctypes.c_size_t), ("perm", ctypes.c_size_t),
                ("inv", ctypes.c_size_t), ("offsets", ctypes.c_size_t)]


class QWeight(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libmoe.so (built by __graft_entry__.build()); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    D = ctypes.POINTER(Dims)
    Q = ctypes.POINTER(QWeight)
    lib.moe_status_str.argtypes = [I]
    lib.moe_status_str.restype = ctypes.c_char_p
    lib.moe_workspace_bytes.argtypes = [D]
    lib.moe_workspace_bytes.restype = Z
    lib.moe_workspace_map_of.argtypes = [D, ctypes.POINTER(WorkspaceMap)]
    lib.moe_workspace_map_of.restype = I
    lib.moe_route.argtypes = [D, P, P, P, P, P, P, P]
    lib.moe_dispatch.argtypes = [D, P, P, P, P, P]
    lib.moe_experts.argtypes = [D, P, P, P, Q, Q, P, P, Z, P]
    lib.moe_experts_noalloc.argtypes = [D, P, P, P, Q, Q, P, P]
    lib.moe_forward.argtypes = [D, P, P, P, P, Q, Q, P, P, P, P, Z, P]
    lib.moe_forward_hostio.argtypes = [D, P, P, P, P, Q, Q, P, P, Z, P]
    lib.moe_forward_branch.argtypes = [D, P, P, P, P, P, P, Q, Q, P, P, P, P, P, Z, P]
    lib.moe_route_q4.argtypes = [D, P, Q, P, P, P, P, P]
    lib.moe_forward_q4router.argtypes = [D, P, Q, P, P, Q, Q, P, P, P, P, Z, P]
    lib.moe_dense_mlp.argtypes = [D, P, Q, Q, P, P, Z, P]
    lib.moe_dense_branch.argtypes = [D, P, P, P, Q, Q, P, P, Z, P]
    lib.moe_self_conditioning.argtypes = [D, P, P, P, Q, Q, P, P, Z, P]
    lib.moe_lm_head.argtypes = [D, ctypes.c_int32, ctypes.c_float, P, Q, P, P, Z, P]
    lib.moe_set_small_t_path.argtypes = [I]
    lib.moe_set_small_t_path.restype = I
    lib.moe_set_router_path.argtypes = [I]
    lib.moe_set_router_path.restype = I
    lib.moe_timing_enable.argtypes = [I]
    lib.moe_timing_read.argtypes = [ctypes.POINTER(ctypes.c_float), I, ctypes.POINTER(I)]
    lib.moe_launches_per_forward.argtypes = [ctypes.c_void_p]
    lib.moe_device_error.argtypes = []
    for fn in ("moe_route", "moe_dispatch", "moe_experts", "moe_experts_noalloc", "moe_forward", "moe_forward_branch",
               "moe_forward_hostio", "moe_route_q4", "moe_forward_q4router", "moe_dense_mlp", "moe_dense_branch",
               "moe_self_conditioning", "moe_lm_head",
               "moe_timing_enable", "moe_timing_read", "moe_launches_per_forward", "moe_device_error"):
        getattr(lib, fn).restype = I
    _lib = lib
    return lib


def dims(T: int, H: int, E: int, k: int, inter: int, group: int = 64, bits: int = 4,
         eps: float = 1e-6) -> Dims:
    return Dims(T, H, E, k, inter, group, bits, eps)


def dims_of(d) -> Dims:
    """Dims from any object with T, H, E, k, inter (, group, bits, eps) attributes."""
    return Dims(d.T, d.H, d.E, d.k, d.inter, getattr(d, "group", 64), getattr(d, "bits", 4),
                getattr(d, "eps", 1e-6))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, rc: int):
    if rc != 0:
        raise MoeError(fn, rc)


def qweight(w, scales, biases) -> QWeight:
    return QWeight(_ptr(w), _ptr(scales), _ptr(biases))


def workspace_bytes(d: Dims) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(d)))


def workspace_map(d: Dims) -> WorkspaceMap:
    """Byte offsets of idx, w, perm, inv and offsets inside a caller workspace."""
    m = WorkspaceMap()
    _check("moe_workspace_map_of", load().moe_workspace_map_of(ctypes.byref(d), ctypes.byref(m)))
    return m


def moe_route(d: Dims, x, router_w, router_scale, per_expert_scale, idx_out, w_out, stream=None):
    _check("moe_route", load().moe_route(ctypes.byref(d), _ptr(x), _ptr(router_w), _ptr(router_scale),
                                         _ptr(per_expert_scale), _ptr(idx_out), _ptr(w_out), _stream(stream)))


def moe_dispatch(d: Dims, idx, perm, offsets, inv, stream=None):
    _check("moe_dispatch", load().moe_dispatch(ctypes.byref(d), _ptr(idx), _ptr(perm), _ptr(offsets),
                                               _ptr(inv), _stream(stream)))


def moe_experts(d: Dims, x, idx, w, gate_up: QWeight, down: QWeight, out, workspace=None,
                ws_bytes: int = 0, stream=None):
    _check("moe_experts", load().moe_experts(ctypes.byref(d), _ptr(x), _ptr(idx), _ptr(w),
                                             ctypes.byref(gate_up), ctypes.byref(down), _ptr(out),
                                             _ptr(workspace), ws_bytes, _stream(stream)))


def moe_experts_noalloc(d: Dims, x, idx, w, gate_up: QWeight, down: QWeight, out, stream=None):
    """moe_experts with the library's fixed scratch (no allocation)."""
    _check("moe_experts_noalloc", load().moe_experts_noalloc(ctypes.byref(d), _ptr(x), _ptr(idx), _ptr(w),
                                                             ctypes.byref(gate_up), ctypes.byref(down),
                                                             _ptr(out), _stream(stream)))


def moe_forward(d: Dims, x, router_w, router_scale, per_expert_scale, gate_up: QWeight, down: QWeight,
                out, idx_out=None, w_out=None, workspace=None, ws_bytes: int = 0, stream=None):
    _check("moe_forward", load().moe_forward(
        ctypes.byref(d), _ptr(x), _ptr(router_w), _ptr(router_scale), _ptr(per_expert_scale),
        ctypes.byref(gate_up), ctypes.byref(down), _ptr(out), _ptr(idx_out), _ptr(w_out),
        _ptr(workspace), ws_bytes, _stream(stream)))


def moe_route_q4(d: Dims, x, router_q: QWeight, router_scale, per_expert_scale, idx_out, w_out, stream=None):
    """moe_route with the 4-bit group-64 router projection."""
    _check("moe_route_q4", load().moe_route_q4(ctypes.byref(d), _ptr(x), ctypes.byref(router_q), _ptr(router_scale),
                                               _ptr(per_expert_scale), _ptr(idx_out), _ptr(w_out), _stream(stream)))


def moe_forward_q4router(d: Dims, x, router_q: QWeight, router_scale, per_expert_scale, gate_up: QWeight,
                         down: QWeight, out, idx_out=None, w_out=None, workspace=None, ws_bytes: int = 0,
                         stream=None):
    """moe_forward with the 4-bit group-64 router projection."""
    _check("moe_forward_q4router", load().moe_forward_q4router(
        ctypes.byref(d), _ptr(x), ctypes.byref(router_q), _ptr(router_scale), _ptr(per_expert_scale),
        ctypes.byref(gate_up), ctypes.byref(down), _ptr(out), _ptr(idx_out), _ptr(w_out), _ptr(workspace),
        ws_bytes, _stream(stream)))


def moe_forward_branch(d: Dims, residual, router_w, router_scale, per_expert_scale, pre_norm_w, post_norm_w,
                       gate_up: QWeight, down: QWeight, out, idx_out=None, w_out=None, expert_in_out=None,
                       workspace=None, ws_bytes: int = 0, stream=None):
    """The decoder layer's MoE branch: route on the residual, experts on
    RMSNorm(residual, pre_norm_w), RMSNorm(., post_norm_w) of their output."""
    _check("moe_forward_branch", load().moe_forward_branch(
        ctypes.byref(d), _ptr(residual), _ptr(router_w), _ptr(router_scale), _ptr(per_expert_scale),
        _ptr(pre_norm_w), _ptr(post_norm_w), ctypes.byref(gate_up), ctypes.byref(down), _ptr(out),
        _ptr(idx_out), _ptr(w_out), _ptr(expert_in_out), _ptr(workspace), ws_bytes, _stream(stream)))


def moe_dense_mlp(d: Dims, x, gate_up: QWeight, down: QWeight, out, workspace=None, ws_bytes: int = 0,
                  stream=None):
    """The dense 4-bit GeGLU MLP over all rows (d.E = d.k = 1, d.inter = its
    intermediate size); gate_up rows are gate_proj then up_proj."""
    _check("moe_dense_mlp", load().moe_dense_mlp(ctypes.byref(d), _ptr(x), ctypes.byref(gate_up),
                                                 ctypes.byref(down), _ptr(out), _ptr(workspace), ws_bytes,
                                                 _stream(stream)))


def moe_dense_branch(d: Dims, h, pre_norm_w, post_norm_w, gate_up: QWeight, down: QWeight, out, workspace=None,
                     ws_bytes: int = 0, stream=None):
    """The decoder layer's dense branch: RMSNorm(mlp(RMSNorm(h, pre)), post)."""
    _check("moe_dense_branch", load().moe_dense_branch(
        ctypes.byref(d), _ptr(h), _ptr(pre_norm_w), _ptr(post_norm_w), ctypes.byref(gate_up), ctypes.byref(down),
        _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)))


def moe_self_conditioning(d: Dims, inputs_embeds, signal, pre_norm_w, gate_up: QWeight, down: QWeight, out,
                          workspace=None, ws_bytes: int = 0, stream=None):
    """SelfConditioning.forward: RMSNormNoScale(inputs_embeds + mlp(RMSNorm(signal, pre)))."""
    _check("moe_self_conditioning", load().moe_self_conditioning(
        ctypes.byref(d), _ptr(inputs_embeds), _ptr(signal), _ptr(pre_norm_w), ctypes.byref(gate_up),
        ctypes.byref(down), _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)))


def moe_lm_head(d: Dims, vocab: int, softcap: float, h, embed: QWeight, logits, workspace=None, ws_bytes: int = 0,
                stream=None):
    """The tied 4-bit head: logits [T, vocab] float32 = softcap * tanh(bf16(h . W^T) / softcap)."""
    _check("moe_lm_head", load().moe_lm_head(ctypes.byref(d), vocab, ctypes.c_float(softcap), _ptr(h),
                                             ctypes.byref(embed), _ptr(logits), _ptr(workspace), ws_bytes,
                                             _stream(stream)))


def moe_forward_hostio(d: Dims, x_host, router_w, router_scale, per_expert_scale, gate_up: QWeight,
                       down: QWeight, out_host, workspace=None, ws_bytes: int = 0, stream=None):
    _check("moe_forward_hostio", load().moe_forward_hostio(
        ctypes.byref(d), _ptr(x_host), _ptr(router_w), _ptr(router_scale), _ptr(per_expert_scale),
        ctypes.byref(gate_up), ctypes.byref(down), _ptr(out_host), _ptr(workspace), ws_bytes,
        _stream(stream)))


def set_small_t_path(mode: int) -> int:
    """0: tcgen05 grouped GEMM for every call (default); 1: the dequant-GEMV
    for calls with T*k <= 2*E. Returns the previous mode."""
    rc = load().moe_set_small_t_path(int(mode))
    if rc < 0:
        raise MoeError("moe_set_small_t_path", -rc)
    return rc


def set_router_path(mode: int) -> int:
    """0 (default): the row router where it fits and the cluster router would
    walk two or more waves of tiles, else the cluster router; 1: always
    the cluster router; 2: the row router wherever it fits. Returns the
    previous mode."""
    rc = load().moe_set_router_path(int(mode))
    if rc < 0:
        raise MoeError("moe_set_router_path", -rc)
    return rc


def timing_enable(on: bool = True):
    _check("moe_timing_enable", load().moe_timing_enable(1 if on else 0))


def timing_read() -> tuple[dict, int]:
    """Summed milliseconds per stage since the last read, and the call count."""
    ms = (ctypes.c_float * len(STAGES))()
    calls = ctypes.c_int(0)
    n = load().moe_timing_read(ms, len(STAGES), ctypes.byref(calls))
    if n < 0:
        raise MoeError("moe_timing_read", -n)
    return {s: float(ms[i]) for i, s in enumerate(STAGES)}, calls.value


def launches_per_forward(d: "Dims") -> int:
    return int(load().moe_launches_per_forward(ctypes.byref(d)))


def device_error() -> int:
    return int(load().moe_device_error())


@dataclasses.dataclass
class DeviceLayer:
    """One MoE layer's parameters resident on the GPU (bit patterns)."""
    router_w: torch.Tensor
    router_scale: torch.Tensor
    pes: torch.Tensor
    gu: tuple
    dn: tuple

    @property
    def gate_up(self) -> QWeight:
        return qweight(*self.gu)

    @property
    def down(self) -> QWeight:
        return qweight(*self.dn)


def to_device_layer(inp, device="cuda") -> DeviceLayer:
    """Copy a moe_synth.LayerInputs' parameters to the GPU (int16 / int32 bit patterns)."""
    def t16(a):
        return torch.from_numpy(a.view("int16").copy()).to(device)

    def t32(a):
        return torch.from_numpy(a.view("int32").copy()).to(device)
    return DeviceLayer(t16(inp.router_w), t16(inp.router_scale), t16(inp.pes),
                       (t32(inp.gu_w), t16(inp.gu_s), t16(inp.gu_b)),
                       (t32(inp.dn_w), t16(inp.dn_s), t16(inp.dn_b)))
