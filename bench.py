"""Throughput of the routed 4-bit MoE layer on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload canvas] [--impl ours|reference]

One step = one whole layer call (router, dispatch, gather, gate_up + GeGLU,
down, combine) on one batch of synthetic tokens of the named workload
(default: the decoder canvas pass, T=256, H=2816, E=128, k=8, inter=704,
4-bit g64 weights). With N > 1 (torchrun) every rank runs its own replica on
its own batch (weak scaling, no collective on the data path).

Prints ONE JSON line (rank 0). `value` is tokens/s with the inputs resident
in HBM, timed with CUDA events around each layer call on its stream; L2 is
flushed between steps, outside the timed events (a 256 MB memset, then a
256 MB read so that no dirty line of the flush is written back inside the
timed region; --flush write keeps the memset alone). `workloads` times the
layer's other workloads (decode, prefill, skew, tiny) the same way. `e2e` is the
same metric through moe_forward_hostio (pinned host x in, host out, copies
inside the timed call). `roofline` is for the dominant kernel (gate_up),
timed with the library's own CUDA events on the launching stream.
`cpu_baseline` times the CPU oracle on a bounded sample of the workload.
`--impl reference` times the CPU oracle alone (the only reference there is).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import threading
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth as ms  # noqa: E402

METRIC = "MoE-layer tokens/s at T=256 canvas (H=2816,E=128,k=8); % of HBM/TC roofline"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return dict(hbm=j["hbm_gbs"], tc=j["bf16_tflops"], tc_sustained=j.get("bf16_tflops_sustained"),
                    source="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sustained=1700.0, source="fallback")


def layer_bytes(d: ms.Dims):
    """Algorithmic bytes of one expert's weights: (gate_up, down)."""
    g = d.group
    gu = 2 * d.inter * d.H // 2 + 2 * (2 * d.inter * d.H // g) * 2
    dn = d.H * d.inter // 2 + 2 * (d.H * d.inter // g) * 2
    return gu, dn


def roofline_model(d: ms.Dims, touched: int, peaks):
    gu, dn = layer_bytes(d)
    S = d.T * d.k
    bytes_alg = touched * (gu + dn) + d.E * d.H * 2 + d.H * 2 + d.E * 2 + 2 * d.T * d.H * 2
    flops = 2 * d.T * d.H * d.E + S * (2 * d.H * 2 * d.inter + 2 * d.inter * d.H)
    t_hbm = bytes_alg / (peaks["hbm"] * 1e9)
    t_tc = flops / (peaks["tc"] * 1e12)
    return dict(bytes=bytes_alg, flops=flops, t_roof_s=max(t_hbm, t_tc), bound="hbm" if t_hbm >= t_tc else "tensor")


def dense_model(dn):
    """Algorithmic bytes (packed weights, scales, biases, x in, out) and
    flops of one dense MLP call over T rows."""
    g = dn.group
    w = 3 * dn.I * dn.H // 2 + 3 * 2 * (dn.I * dn.H // g) * 2
    return dict(bytes=w + 2 * dn.T * dn.H * 2, flops=2 * dn.T * dn.H * 3 * dn.I,
                gate_up_flops=2 * dn.T * dn.H * 2 * dn.I)


def dense_report(dn, dense_ms, stage_ms, calls, peaks, world):
    m = dense_model(dn)
    t_hbm, t_tc = m["bytes"] / (peaks["hbm"] * 1e9), m["flops"] / (peaks["tc"] * 1e12)
    t_roof = max(t_hbm, t_tc)
    gu_ms = stage_ms["gate_up"] / max(1, calls)
    gu_tflops = m["gate_up_flops"] / (gu_ms * 1e-3) / 1e12
    return dict(
        workload=f"dense 4-bit GeGLU MLP: T={dn.T} H={dn.H} I={dn.I} group={dn.group} (I not on the pages)",
        ms_per_step={k: v for k, v in dense_ms.items()},
        value={k: whole_job_rate(dn.T, world, v * 1e-3) for k, v in dense_ms.items()}, unit="tokens/s",
        roofline=dict(bound="tensor" if t_tc >= t_hbm else "hbm", t_roof_us=t_roof * 1e6,
                      t_mlp_us=dense_ms["mlp"] * 1e3, frac=t_roof / (dense_ms["mlp"] * 1e-3), bytes=m["bytes"],
                      flops=m["flops"], peak_source=f"{peaks['source']} bf16_tflops and hbm_gbs"),
        gate_up_kernel=dict(ms_per_launch=gu_ms, achieved_tflops=gu_tflops, peak=peaks["tc"],
                            frac=gu_tflops / peaks["tc"]),
        stages_ms_per_call={k: v / max(1, calls) for k, v in stage_ms.items() if v > 0})


def head_report(T, H, V, head_ms, stage_ms, calls, peaks, world, group=64):
    """The tied head: algorithmic bytes = packed table + scales + biases +
    h in + fp32 logits out; flops = 2 T H V."""
    bytes_ = V * H // 2 + 2 * (V * H // group) * 2 + T * H * 2 + T * V * 4
    flops = 2 * T * H * V
    t_hbm, t_tc = bytes_ / (peaks["hbm"] * 1e9), flops / (peaks["tc"] * 1e12)
    gemm_ms = stage_ms["gate_up"] / max(1, calls)
    return dict(workload=f"tied 4-bit head + fp32 softcap 30: T={T} H={H} vocab={V} group={group} (vocab not on the "
                         f"pages)",
                ms_per_step=head_ms, value=whole_job_rate(T, world, head_ms * 1e-3), unit="tokens/s",
                roofline=dict(bound="tensor" if t_tc >= t_hbm else "hbm", t_roof_us=max(t_hbm, t_tc) * 1e6,
                              t_head_us=head_ms * 1e3, frac=max(t_hbm, t_tc) / (head_ms * 1e-3), bytes=bytes_,
                              flops=flops),
                gemm_kernel=dict(ms_per_launch=gemm_ms, achieved_tflops=flops / (gemm_ms * 1e-3) / 1e12,
                                 achieved_gbs=bytes_ / (gemm_ms * 1e-3) / 1e9),
                stages_ms_per_call={k: v / max(1, calls) for k, v in stage_ms.items() if v > 0})


class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU, read through NVML
    (ctypes, read-only queries) every 2 ms while the timed region runs, plus
    one reading at each end. Falls back to nothing when NVML is missing."""
    # nvmlClocksEventReason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, uuid: str | None = None, period_s: float = 0.002):
        self.index, self.uuid, self.period = index, uuid, period_s
        self.rows, self.nvml, self.handle = [], None, None
        self._stop = threading.Event()
        self._thread = None

    def _open(self):
        import ctypes
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                lib = None
        if lib is None or lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) == 0
        if not ok:
            return False
        self.nvml, self.handle, self.ct = lib, h, ctypes
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
        return True

    def _sample(self):
        ct, lib, h = self.ct, self.nvml, self.handle
        clk, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) != 0:
            return
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        reasons = rs.value if fn(h, ct.byref(rs)) == 0 else 0
        power = pw.value / 1e3 if lib.nvmlDeviceGetPowerUsage(h, ct.byref(pw)) == 0 else None
        self.rows.append((float(clk.value), power, int(reasons)))

    def _run(self):
        while not self._stop.wait(self.period):
            self._sample()

    def __enter__(self):
        try:
            if self._open():
                self._sample()
                self._thread = threading.Thread(target=self._run, daemon=True)
                self._thread.start()
        except (OSError, AttributeError):
            self.nvml = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            self._sample()

    def summary(self):
        if not self.rows:
            return None
        reasons = sorted({name for _, _, r in self.rows for bit, name in self.REASONS.items() if r & bit})
        powers = [p for _, p, _ in self.rows if p is not None]
        return dict(sm_mhz=statistics.median(c for c, _, _ in self.rows), sm_max_mhz=self.max_mhz,
                    power_w_max=max(powers) if powers else None, samples=len(self.rows), reasons=reasons,
                    source="NVML every 2 ms during the timed region")


class L2Flush:
    """Between timed steps (outside the CUDA events): write a 256 MB buffer,
    which evicts the 129 MB L2; with mode "write+read" (default) then read a
    second 256 MB buffer, so the L2 holds clean lines of that buffer and the
    flush's own dirty lines are written back before the timed region instead
    of inside it."""

    def __init__(self, mode: str = "write+read"):
        import torch
        self.mode = mode
        self.wbuf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.rbuf = torch.ones((256 << 20) // 8, dtype=torch.int64, device="cuda") if mode == "write+read" else None

    def __call__(self):
        self.wbuf.zero_()
        if self.rbuf is not None:
            self.rbuf.max()

    def describe(self) -> str:
        return ("flushed between steps outside the timed events: 256 MB memset"
                + (", then a 256 MB read (clean L2)" if self.rbuf is not None else ""))


def cores_available() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(wl: ms.Workload, target_s: float = 8.0, max_tokens: int | None = None):
    """Time the CPU oracle on a growing prefix of the workload's tokens until a
    call takes target_s (bounded). Returns (tokens/s, tokens, seconds, threads)."""
    import oracle
    oracle.build()
    full = ms.make_layer(wl)
    n = 8
    limit = max_tokens or full.dims.T
    while True:
        d = ms.Dims(**{**full.dims.__dict__, "T": n})
        inp = ms.LayerInputs(d, full.x[:n], full.router_w, full.router_scale, full.pes, full.gu_w, full.gu_s,
                             full.gu_b, full.dn_w, full.dn_s, full.dn_b)
        t0 = time.perf_counter()
        oracle.forward(inp)
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= limit:
            return n / dt, n, dt, oracle.max_threads()
        n = min(limit, n * 2 if dt < target_s / 3 else int(n * target_s / dt) + 1)


def run_reference(args, wl):
    """--impl reference: the CPU oracle on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    tps, n, dt, threads = oracle_sample(wl, target_s=min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    full = ms.make_layer(wl)
    d = ms.Dims(**{**full.dims.__dict__, "T": n})
    inp = ms.LayerInputs(d, full.x[:n], full.router_w, full.router_scale, full.pes, full.gu_w, full.gu_s,
                         full.gu_b, full.dn_w, full.dn_s, full.dn_b)
    for _ in range(args.warmup):
        oracle.forward(inp)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.forward(inp)
        times.append(time.perf_counter() - t0)
    value = n / statistics.mean(times)
    line = dict(metric=METRIC, value=value, unit="tokens/s", impl="reference", n_gpus=args.gpus,
                steps=args.steps, warmup=args.warmup, ms_per_step=1e3 * statistics.mean(times),
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16", data="synthetic",
                config=dict(workload=wl_desc(wl), sample_tokens=n),
                cpu_baseline=dict(value=value, unit="tokens/s", cores=threads, kind="oracle",
                                  sample=f"first {n} of {full.dims.T} tokens of the {wl.name} workload, "
                                         f"per step"),
                e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def wl_desc(wl):
    d = wl.dims
    return (f"{wl.name}: T={d.T} H={d.H} E={d.E} k={d.k} inter={d.inter} group={d.group} 4-bit affine, "
            f"bf16 activations" + (f", Zipf({wl.zipf_s}) skew" if wl.skew_kappa else ""))


def traffic_from_profile(name: str, src_hash: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        j = json.load(fh)
    e = j.get(name)
    if not e or e.get("source_sha1") != src_hash:
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- replicas --
# The layer shards by tokens with no exchange: N GPUs run N independent
# replicas (weak scaling), each on its own seeded batch of the same workload.
def replica_layer(wl, rank: int):
    """Rank r's batch: the workload's generator with seed + r."""
    return ms.make_layer(wl, seed=wl.seed + rank)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's time (all ranks block until every rank has it)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank: int, world: int, seconds: float) -> float:
    """Tokens/s of the whole job: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / seconds


def time_workload(wl, rank, world, layer, head_inp, args, flush, stream, peaks, local, uuid):
    """One moe_forward per step on workload `wl`, timed like the headline:
    L2 flushed between steps outside the events, CUDA events around each
    step on the launching stream, clocks sampled meanwhile. The expert
    weights of the headline layer are reused when the layer is the same
    (same sizes and seed: the generator gives the same bytes)."""
    import torch
    import bit_quantized_moe_layer_gb300 as moe
    seed = wl.seed + rank
    d0 = wl.dims
    same = all(getattr(d0, f) == getattr(head_inp.dims, f) for f in ("H", "E", "inter", "group"))
    if same:
        x_h = ms.make_x(d0, seed, mu=wl.skew_mu)
        wr, sc, pes = ms.make_router(d0, seed, kappa=wl.skew_kappa, zipf_s=wl.zipf_s)
        t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).cuda()
        lay = moe.DeviceLayer(t16(wr), t16(sc), t16(pes), layer.gu, layer.dn)
    else:
        full = ms.make_layer(wl, seed=seed)
        x_h, lay = full.x, moe.to_device_layer(full)
    d = moe.dims_of(d0)
    x = torch.from_numpy(x_h.view(np.int16).copy()).cuda()
    out = torch.empty((d.T, d.H), dtype=torch.int16, device="cuda")
    idx = torch.empty((d.T, d.k), dtype=torch.int32, device="cuda")
    wts = torch.empty((d.T, d.k), dtype=torch.int16, device="cuda")
    ws = torch.empty(moe.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    step = lambda: moe.moe_forward(d, x, lay.router_w, lay.router_scale, lay.pes, lay.gate_up, lay.down, out, idx,
                                   wts, ws, ws.numel(), stream)
    steps = max(20, min(args.steps, 100))
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    touched = int(np.unique(idx.cpu().numpy()).size)
    st = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with ClockSampler(local, uuid) as clk:
        for i in range(steps):
            flush()
            st[i].record(stream)
            step()
            en[i].record(stream)
        torch.cuda.synchronize()
    ms_step = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(st, en)), world, "cuda")
    moe.timing_enable(True)
    for _ in range(steps):
        flush()
        step()
    torch.cuda.synchronize()
    stage_ms, calls = moe.timing_read()
    moe.timing_enable(False)
    model = roofline_model(d0, touched, peaks)
    gu_bytes, _ = layer_bytes(d0)
    gu_ms = stage_ms["gate_up"] / max(1, calls)
    return dict(workload=wl_desc(wl), steps=steps, ms_per_step=ms_step, value=whole_job_rate(d.T, world, ms_step * 1e-3),
                unit="tokens/s", experts_touched=touched,
                layer_roofline=dict(bound=model["bound"], t_roof_us=model["t_roof_s"] * 1e6,
                                    frac=model["t_roof_s"] / (ms_step * 1e-3), bytes=model["bytes"],
                                    flops=model["flops"]),
                gate_up=dict(ms_per_launch=gu_ms, achieved_gbs=touched * gu_bytes / (gu_ms * 1e-3) / 1e9,
                             achieved_tflops=(d.T * d.k * 2 * d.H * 2 * d.inter) / (gu_ms * 1e-3) / 1e12),
                stages_ms_per_call={k: v / max(1, calls) for k, v in stage_ms.items()},
                clocks=clk.summary(), gpu_launches=moe.launches_per_forward(d) * steps)


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    import bit_quantized_moe_layer_gb300 as moe
    from bit_quantized_moe_layer_gb300 import build as lib_build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    lib_build.build()
    moe.load()
    peaks = load_peaks()

    inp = replica_layer(wl, rank)
    d = moe.dims_of(inp.dims)
    layer = moe.to_device_layer(inp)
    x = torch.from_numpy(inp.x.view(np.int16).copy()).cuda()
    out = torch.empty((d.T, d.H), dtype=torch.int16, device="cuda")
    idx = torch.empty((d.T, d.k), dtype=torch.int32, device="cuda")
    wts = torch.empty((d.T, d.k), dtype=torch.int16, device="cuda")
    ws = torch.empty(moe.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    flush = L2Flush(args.flush)
    stream = torch.cuda.current_stream()

    def step():
        moe.moe_forward(d, x, layer.router_w, layer.router_scale, layer.pes, layer.gate_up, layer.down, out,
                        idx, wts, ws, ws.numel(), stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    touched = int(np.unique(idx.cpu().numpy()).size)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except (AttributeError, RuntimeError):
        uuid = None
    # Timed region 1: whole steps, events only around each step (the
    # library's kernels run back to back with programmatic dependent launch).
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local, uuid) as clk:
        for i in range(args.steps):
            flush()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    # Timed region 2: the same steps with the library's per-kernel events on
    # (they sit between the kernels, so this pass is only for the breakdown
    # and the per-launch roofline of the dominant kernel).
    moe.timing_enable(True)
    for i in range(args.steps):
        flush()
        step()
    torch.cuda.synchronize()
    stage_ms, calls = moe.timing_read()
    moe.timing_enable(False)
    err = moe.device_error()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_step = max_over_ranks(statistics.mean(step_ms), world, "cuda")

    # end to end through the host-buffer call (x in, out back, copies inside)
    x_host = torch.from_numpy(inp.x.view(np.int16).copy()).pin_memory()
    out_host = torch.empty((d.T, d.H), dtype=torch.int16).pin_memory()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        moe.moe_forward_hostio(d, x_host, layer.router_w, layer.router_scale, layer.pes, layer.gate_up,
                               layer.down, out_host, ws, ws.numel(), stream)
        if i >= args.warmup:
            e2e_ms.append(1e3 * (time.perf_counter() - t0))
    e2e_step = max_over_ranks(statistics.mean(e2e_ms), world, "cuda")

    def timed(call):
        """Mean ms of `call` over the timed steps, like region 1 (L2 flushed
        between steps, events around each call on its stream)."""
        for _ in range(args.warmup):
            flush()
            call()
        st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush()
            st[i].record(stream)
            call()
            en[i].record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(st, en)), world, "cuda")

    # The other workloads of the layer, each timed like the headline (L2
    # flushed, events around each moe_forward on its stream, clocks sampled).
    workloads = {}
    if not args.no_workloads:
        for name in ("decode", "prefill", "skew", "tiny"):
            if name == wl.name:
                continue
            workloads[name] = time_workload(ms.WORKLOADS[name], rank, world, layer, inp, args, flush, stream,
                                            peaks, local, uuid)
        # the decode step through the small-token dequant-GEMV path instead
        # of the tensor-core grouped GEMM (moe_set_small_t_path(1))
        prev = moe.set_small_t_path(1)
        try:
            workloads["decode_gemv_path"] = time_workload(ms.WORKLOADS["decode"], rank, world, layer, inp, args,
                                                          flush, stream, peaks, local, uuid)
        finally:
            moe.set_small_t_path(prev)
        torch.cuda.synchronize()

    if args.layer_only:
        emit_line(args, wl, inp, d, world, rank, peaks, touched, ms_step, stage_ms, calls, clk, e2e_step, workloads,
                  err, flush, None)
        if world > 1:
            dist.destroy_process_group()
        return

    # The decoder layer's MoE branch (moe_forward_branch: the router on the
    # residual, the experts on preFfNorm2(residual), postFfNorm2 of their
    # output).
    pre_w, post_w = (torch.from_numpy(a.view(np.int16).copy()).cuda()
                     for a in ms.make_branch_norms(inp.dims, wl.seed))
    out_b = torch.empty_like(out)
    branch_ms = timed(lambda: moe.moe_forward_branch(
        d, x, layer.router_w, layer.router_scale, layer.pes, pre_w, post_w, layer.gate_up, layer.down, out_b, idx,
        wts, None, ws, ws.numel(), stream))

    # The layer with the 4-bit group-64 router projection (moe_forward_q4router).
    rq = [torch.from_numpy(a.view(np.int32 if a.dtype == np.uint32 else np.int16).copy()).cuda()
          for a in ms.make_router_q4(inp.dims, wl.seed)]
    q4_ms = timed(lambda: moe.moe_forward_q4router(
        d, x, moe.qweight(*rq), layer.router_scale, layer.pes, layer.gate_up, layer.down, out_b, idx, wts, ws,
        ws.numel(), stream))

    # The dense 4-bit GeGLU MLP at the same T (H as the layer, I = 2112):
    # moe_dense_mlp, the decoder layer's dense branch and SelfConditioning.
    dn = ms.make_dense(d.T, H=d.H, I=ms.DENSE_INTER, seed=wl.seed + rank)
    dd = moe.dims(dn.T, dn.H, 1, 1, dn.I, eps=dn.eps)
    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).cuda()
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int32).copy()).cuda()
    dgu = (t32(np.concatenate([dn.gate[0], dn.up[0]])), t16(np.concatenate([dn.gate[1], dn.up[1]])),
           t16(np.concatenate([dn.gate[2], dn.up[2]])))
    ddn = (t32(dn.down[0]), t16(dn.down[1]), t16(dn.down[2]))
    dx, demb, dpre, dpost = t16(dn.x), t16(dn.embeds), t16(dn.pre_w), t16(dn.post_w)
    dws = torch.empty(moe.workspace_bytes(dd), dtype=torch.uint8, device="cuda")
    dout = torch.empty((dn.T, dn.H), dtype=torch.int16, device="cuda")
    qg, qd = moe.qweight(*dgu), moe.qweight(*ddn)
    dense_calls = {
        "mlp": lambda: moe.moe_dense_mlp(dd, dx, qg, qd, dout, dws, dws.numel(), stream),
        "branch": lambda: moe.moe_dense_branch(dd, dx, dpre, dpost, qg, qd, dout, dws, dws.numel(), stream),
        "self_conditioning": lambda: moe.moe_self_conditioning(dd, demb, dx, dpre, qg, qd, dout, dws, dws.numel(),
                                                               stream),
    }
    dense_ms = {k_: timed(f_) for k_, f_ in dense_calls.items()}

    # The tied 4-bit head with the fp32 softcap at the same T, vocabulary 2^18.
    hh, hemb = ms.make_head(d.T, H=d.H, V=ms.VOCAB, seed=wl.seed + rank)
    hd = moe.dims(d.T, d.H, 1, 1, 64)
    h_h, h_emb = t16(hh), (t32(hemb[0]), t16(hemb[1]), t16(hemb[2]))
    h_out = torch.empty((d.T, ms.VOCAB), dtype=torch.float32, device="cuda")
    h_ws = torch.empty(moe.workspace_bytes(hd), dtype=torch.uint8, device="cuda")
    qh = moe.qweight(*h_emb)
    head_call = lambda: moe.moe_lm_head(hd, ms.VOCAB, 30.0, h_h, qh, h_out, h_ws, h_ws.numel(), stream)
    head_ms = timed(head_call)
    moe.timing_enable(True)
    for _ in range(args.steps):
        flush()
        head_call()
    torch.cuda.synchronize()
    head_stage_ms, head_calls_n = moe.timing_read()
    moe.timing_enable(False)
    del h_out, h_emb, qh
    moe.timing_enable(True)
    for _ in range(args.steps):
        flush()
        dense_calls["mlp"]()
    torch.cuda.synchronize()
    dense_stage_ms, dense_calls_n = moe.timing_read()
    moe.timing_enable(False)
    err |= moe.device_error()

    extras = dict(
        branch=dict(call="moe_forward_branch (router on the residual, experts on preFfNorm2, postFfNorm2)",
                    ms_per_step=branch_ms, value=whole_job_rate(d.T, world, branch_ms * 1e-3), unit="tokens/s"),
        q4router=dict(call="moe_forward_q4router (the layer with the 4-bit group-64 router projection)",
                      ms_per_step=q4_ms, value=whole_job_rate(d.T, world, q4_ms * 1e-3), unit="tokens/s"),
        dense=dense_report(dn, dense_ms, dense_stage_ms, dense_calls_n, peaks, world),
        lm_head=head_report(d.T, d.H, ms.VOCAB, head_ms, head_stage_ms, head_calls_n, peaks, world))
    emit_line(args, wl, inp, d, world, rank, peaks, touched, ms_step, stage_ms, calls, clk, e2e_step, workloads,
              err, flush, extras)
    if world > 1:
        dist.destroy_process_group()


def emit_line(args, wl, inp, d, world, rank, peaks, touched, ms_step, stage_ms, calls, clk, e2e_step, workloads,
              err, flush, extras):
    """Rank 0 prints the one JSON line."""
    import bit_quantized_moe_layer_gb300 as moe
    if rank != 0:
        return
    gu_bytes, dn_bytes = layer_bytes(inp.dims)
    gu_ms = stage_ms["gate_up"] / max(1, calls)
    achieved = touched * gu_bytes / (gu_ms * 1e-3) / 1e9
    with open(os.path.join(ROOT, "bit_quantized_moe_layer_gb300", "csrc", "grouped_gemm.cu"), "rb") as fh:
        src_hash = hashlib.sha1(fh.read()).hexdigest()
    model = roofline_model(inp.dims, touched, peaks)
    value = whole_job_rate(d.T, world, ms_step * 1e-3)

    cpu = None
    if not args.no_cpu_baseline:
        tps, n, dt, threads = oracle_sample(wl, target_s=args.cpu_seconds)
        cpu = dict(value=tps, unit="tokens/s", cores=threads, kind="oracle",
                   sample=f"first {n} of {d.T} tokens of the {wl.name} workload, one oracle call ({dt:.1f} s)")
    line = dict(
        metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=args.steps, warmup=args.warmup,
        ms_per_step=ms_step, higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16",
        data="synthetic (seeded; no checkpoint on the pages)",
        config=dict(workload=wl_desc(wl), global_batch=world * d.T, tokens_per_gpu=d.T, parallelism=f"replicas x{world}",
                    l2=flush.describe(),
                    experts_touched=touched),
        roofline=dict(bound="hbm", achieved=achieved, peak=peaks["hbm"], unit="GB/s", frac=achieved / peaks["hbm"],
                      traffic=traffic_from_profile(f"gate_up:{wl.name}", src_hash), kernel="grouped_gemm gate_up",
                      bytes_per_launch=touched * gu_bytes, ms_per_launch=gu_ms,
                      peak_source=f"{peaks['source']} hbm_gbs (copy)",
                      timed="per-launch CUDA events in timed region 2 (same steps, library timing on)"),
        layer_roofline=dict(bound=model["bound"], t_roof_us=model["t_roof_s"] * 1e6, t_step_us=ms_step * 1e3,
                            frac=model["t_roof_s"] / (ms_step * 1e-3), bytes=model["bytes"], flops=model["flops"]),
        stages_ms_per_call={k: v / max(1, calls) for k, v in stage_ms.items()},
        cpu_baseline=cpu,
        e2e=dict(value=whole_job_rate(d.T, world, e2e_step * 1e-3), unit="tokens/s", h2d_bytes_per_step=d.T * d.H * 2,
                 d2h_bytes_per_step=d.T * d.H * 2, ms_per_step=e2e_step),
        gpu_launches=moe.launches_per_forward(d) * args.steps,
        **(extras or {}),
        clocks=clk.summary(),
        workloads=workloads,
        device_error=err,
    )
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="canvas", choices=sorted(ms.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--flush", default="write+read", choices=["write+read", "write"])
    ap.add_argument("--no-workloads", action="store_true", help="skip the other workloads' lines")
    ap.add_argument("--layer-only", action="store_true",
                    help="time the layer alone (no MoE branch, 4-bit router, dense MLP or head lines)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = ms.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
