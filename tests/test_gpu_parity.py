"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every workload of the layer runs at full size on the GPU and the oracle
checks every token of every workload (the two largest take the oracle ~20 s
each on 16 host cores, once per session): routing, the dispatch the forward
itself runs (read back from the caller workspace, bit for bit), the experts
path and the whole layer. Comparison rules: tests/gpu_helpers.py.
"""
import dataclasses

import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle
import gpu_helpers as gh

pytestmark = pytest.mark.gpu

ALL = ("tiny", "decode", "canvas", "prefill", "skew")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_moe_layer_gb300 import build
    build.build()
    oracle.build()


_cache = {}


def layer(name):
    if name not in _cache:
        inp = ms.make_layer(name)
        ref = gh.oracle_route(inp)
        _cache[name] = (inp, gh.upload(inp), ref)
    return _cache[name]


_oracle_out = {}


def oracle_out(name):
    """The oracle's layer output for every token, on its own routing."""
    if name not in _oracle_out:
        inp, g, ref = layer(name)
        _oracle_out[name] = gh.oracle_experts_rows(inp, ref["idx"], ref["w"])
    return _oracle_out[name]


def gpu_weights_in_oracle_order(idx, w, ref_idx, rows):
    """The GPU's routing weights rearranged into the oracle's expert order,
    for tokens whose expert sets agree (all others zero)."""
    out = np.zeros(ref_idx.shape, np.uint16)
    for t in rows:
        pos = {e: j for j, e in enumerate(idx[t].tolist())}
        out[t] = [w[t, pos[e]] for e in ref_idx[t].tolist()]
    return out


def sub_explainer(explain, rows):
    """An explainer for a comparison restricted to `rows` (indices into it)."""
    return lambda r: explain(rows[r])


def sample_rows(T, n=48, seed=0):
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    return np.sort(np.concatenate([[0, T - 1], rng.choice(np.arange(1, T - 1), n - 2, replace=False)]))


@pytest.mark.parametrize("name", ALL)
def test_route(name):
    inp, g, ref = layer(name)
    idx, w = gh.gpu_route(g)
    c = gh.check_routing(inp.dims, ref, idx, w, inp.router_w)
    print(f"{name}: routing {c} of {inp.dims.T} tokens")


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("name", ALL)
def test_route_each_kernel(name, mode):
    """Both router kernels against the oracle on every workload, whichever
    the default picks there: the cluster router (moe_set_router_path(1)),
    which the 4-bit projection and small T use, and the row router
    (moe_set_router_path(2)), which large T uses. The two sum the scores in
    different fp32 orders, so each is held to the oracle (check_routing), not
    to the other."""
    import bit_quantized_moe_layer_gb300 as moe
    inp, g, ref = layer(name)
    prev = moe.set_router_path(mode)
    try:
        idx, w = gh.gpu_route(g)
    finally:
        moe.set_router_path(prev)
    c = gh.check_routing(inp.dims, ref, idx, w, inp.router_w)
    print(f"{name}: {'cluster' if mode == 1 else 'row'} router {c} of {inp.dims.T} tokens")


@pytest.mark.parametrize("T", [1, 15, 17, 100, 257])
def test_row_router_ragged(T):
    """The row router on token counts that leave a partial 16-token tile."""
    import bit_quantized_moe_layer_gb300 as moe
    inp = ms.make_layer("canvas", T=T, seed=5)
    g = gh.upload(inp)
    ref = gh.oracle_route(inp)
    prev = moe.set_router_path(2)
    try:
        idx, w = gh.gpu_route(g)
    finally:
        moe.set_router_path(prev)
    gh.check_routing(inp.dims, ref, idx, w, inp.router_w)


def test_router_path_switch():
    import bit_quantized_moe_layer_gb300 as moe
    assert moe.set_router_path(0) == 0
    assert moe.set_router_path(1) == 0
    assert moe.set_router_path(2) == 1
    assert moe.set_router_path(0) == 2
    with pytest.raises(moe.MoeError):
        moe.set_router_path(3)


@pytest.mark.parametrize("name", ALL)
def test_dispatch(name):
    inp, g, ref = layer(name)
    d = inp.dims
    perm, off, inv = gh.gpu_dispatch(g.d, ref["idx"])
    operm, ooff, oinv = oracle.dispatch(d.T, d.k, d.E, ref["idx"])
    assert np.array_equal(off, ooff)
    assert np.array_equal(perm, operm)
    assert np.array_equal(inv, oinv)


@pytest.mark.parametrize("case", ["T1", "one_expert", "empty_experts", "k1"])
def test_dispatch_edges(case):
    rng = np.random.default_rng(5)
    if case == "T1":
        d = ms.Dims(T=1, H=256, E=8, k=2, inter=128)
        idx = np.array([[7, 0]], np.int32)
    elif case == "one_expert":
        d = ms.Dims(T=4000, H=256, E=8, k=1, inter=128)
        idx = np.full((d.T, 1), 3, np.int32)
    elif case == "empty_experts":
        d = ms.Dims(T=700, H=2816, E=128, k=8, inter=704)
        idx = np.stack([rng.permutation(8)[:8] for _ in range(d.T)]).astype(np.int32)
    else:
        d = ms.Dims(T=4096, H=2816, E=128, k=1, inter=704)
        idx = rng.integers(0, 128, (d.T, 1)).astype(np.int32)
    import bit_quantized_moe_layer_gb300 as moe
    perm, off, inv = gh.gpu_dispatch(moe.dims_of(d), idx)
    operm, ooff, oinv = oracle.dispatch(d.T, d.k, d.E, idx)
    assert np.array_equal(off, ooff) and np.array_equal(perm, operm) and np.array_equal(inv, oinv)


@pytest.mark.parametrize("name", ALL)
def test_experts(name):
    """The experts path alone, fed the oracle's routing; every token."""
    inp, g, ref = layer(name)
    out = gh.gpu_experts(g, ref["idx"], ref["w"])
    stats = gh.compare_out(out, oracle_out(name), f"{name} experts", gh.explainer(inp, ref["idx"], ref["w"]))
    print(f"{name} experts: {stats}")


@pytest.mark.parametrize("name", ALL)
def test_forward(name):
    """The whole layer on every token; tokens whose routing legitimately
    differs (near ties) are excluded from the output comparison."""
    inp, g, ref = layer(name)
    out, idx, w = gh.gpu_forward(g)
    c = gh.check_routing(inp.dims, ref, idx, w, inp.router_w)
    same = np.array([set(idx[t]) == set(ref["idx"][t]) for t in range(inp.dims.T)])
    rows = np.flatnonzero(same)
    w_gpu = gpu_weights_in_oracle_order(idx, w, ref["idx"], rows)
    stats = gh.compare_out(out[rows], oracle_out(name)[rows], f"{name} forward",
                           sub_explainer(gh.explainer(inp, ref["idx"], ref["w"], w_gpu), rows))
    print(f"{name} forward: routing {c}, output {stats}")


@pytest.mark.parametrize("name", ALL)
def test_forward_dispatch_bit_exact(name):
    """The dispatch the forward itself runs (the fused dispatch + gather
    kernel up to 8192 slots, the three-kernel sort above), read back from the
    caller workspace: perm, offsets and inv equal the oracle's stable sort of
    the routing the same call produced, bit for bit."""
    import bit_quantized_moe_layer_gb300 as moe
    inp, g, ref = layer(name)
    d = inp.dims
    ws = torch.full((moe.workspace_bytes(g.d),), 0xA5, dtype=torch.uint8, device="cuda")
    out, idx, w = gh.gpu_forward(g, workspace=ws)
    perm, off, inv = gh.workspace_dispatch(g.d, ws)
    operm, ooff, oinv = oracle.dispatch(d.T, d.k, d.E, idx)
    assert np.array_equal(off, ooff), "offsets"
    assert np.array_equal(perm, operm), "perm"
    assert np.array_equal(inv, oinv), "inv"


@pytest.mark.parametrize("case", ["empty_experts", "one_expert", "T1"])
def test_experts_dispatch_edges_bit_exact(case):
    """The in-call dispatch of moe_experts on edge routings (most experts
    empty; every slot on one expert, several token tiles; one token), read
    back from the caller workspace and compared bit for bit; the output is
    checked against the oracle."""
    import bit_quantized_moe_layer_gb300 as moe
    rng = np.random.default_rng(8)
    if case == "empty_experts":
        inp = ms.make_layer("canvas", T=96, seed=9)
        idx = np.stack([rng.permutation(8)[:8] + 40 for _ in range(96)]).astype(np.int32)
    elif case == "one_expert":
        inp = ms.make_layer("canvas", T=200, seed=10)
        idx = np.stack([np.concatenate([[77], rng.choice(np.r_[0:77, 78:128], 7, replace=False)])
                        for _ in range(200)]).astype(np.int32)
    else:
        inp = ms.make_layer("canvas", T=1, seed=11)
        idx = np.array([[127, 0, 64, 3, 100, 1, 2, 50]], np.int32)
    d = inp.dims
    w = ms.bf16_bits(rng.uniform(0.05, 0.3, idx.shape))
    g = gh.upload(inp)
    ws = torch.full((moe.workspace_bytes(g.d),), 0x5A, dtype=torch.uint8, device="cuda")
    out = gh.gpu_experts(g, idx, w, workspace=ws)
    perm, off, inv = gh.workspace_dispatch(g.d, ws)
    operm, ooff, oinv = oracle.dispatch(d.T, d.k, d.E, idx)
    assert np.array_equal(off, ooff) and np.array_equal(perm, operm) and np.array_equal(inv, oinv)
    rows = sample_rows(d.T, 64, seed=3)
    gh.compare_out(out[rows], gh.oracle_experts_rows(inp, idx, w, rows), f"edge {case}",
                   sub_explainer(gh.explainer(inp, idx, w), rows))


@pytest.mark.parametrize("T", [1, 17, 33, 130])
def test_ragged_token_counts(T):
    """Token counts that leave partial router tiles and partial MMA tiles."""
    inp = ms.make_layer("canvas", T=T, seed=3)
    g = gh.upload(inp)
    ref = gh.oracle_route(inp)
    out, idx, w = gh.gpu_forward(g)
    gh.check_routing(inp.dims, ref, idx, w, inp.router_w)
    same = np.array([set(idx[t]) == set(ref["idx"][t]) for t in range(T)])
    rows = np.flatnonzero(same)
    want = gh.oracle_experts_rows(inp, ref["idx"], ref["w"], rows)
    w_gpu = gpu_weights_in_oracle_order(idx, w, ref["idx"], rows)
    gh.compare_out(out[rows], want, f"T={T}", sub_explainer(gh.explainer(inp, ref["idx"], ref["w"], w_gpu), rows))


def test_tiny_layer_ragged():
    inp = ms.make_layer("tiny", T=37, seed=4)
    g = gh.upload(inp)
    ref = gh.oracle_route(inp)
    out = gh.gpu_experts(g, ref["idx"], ref["w"])
    gh.compare_out(out, gh.oracle_experts_rows(inp, ref["idx"], ref["w"]), "tiny T=37",
                   gh.explainer(inp, ref["idx"], ref["w"]))


def test_many_rows_one_expert():
    """One expert receives more rows than a token tile holds (several tiles),
    most experts receive none."""
    inp = ms.make_layer("canvas", T=300, seed=6)
    g = gh.upload(inp)
    rng = np.random.default_rng(6)
    idx = np.stack([np.concatenate([[5], rng.choice(np.r_[0:5, 6:12], 7, replace=False)])
                    for _ in range(300)]).astype(np.int32)
    w = ms.bf16_bits(rng.uniform(0.05, 0.3, (300, 8)))
    out = gh.gpu_experts(g, idx, w)
    rows = sample_rows(300, 40, seed=2)
    gh.compare_out(out[rows], gh.oracle_experts_rows(inp, idx, w, rows), "many rows one expert",
                   sub_explainer(gh.explainer(inp, idx, w), rows))


def test_ragged_tiles_many_rows():
    """~100 rows an expert (the 128-row token tiles): experts with 1, 16,
    127..130, 255..257 and 513 rows, one with 600 (several full tiles and a
    tail), the rest ~89 rows each. The sampled tokens include each special
    expert's rows at the tile boundaries."""
    T = 1600
    inp = ms.make_layer("canvas", T=T, seed=12)
    d = inp.dims
    special = {0: 600, 1: 257, 2: 129, 3: 128, 4: 1, 5: 255, 6: 256, 7: 513, 8: 16, 9: 130, 10: 127}
    rest = [e for e in range(d.E) if e not in special]
    left = T * d.k - sum(special.values())
    counts = dict(special)
    for i, e in enumerate(rest):
        counts[e] = left // len(rest) + (1 if i < left % len(rest) else 0)
    assert sum(counts.values()) == T * d.k and max(counts.values()) <= T
    # Expert e fills a run of consecutive positions of the column-major
    # [k, T] slot grid, so no token meets an expert twice.
    order = np.repeat(np.arange(d.E), [counts[e] for e in range(d.E)])
    rng = np.random.default_rng(12)
    order = np.concatenate([order[order == e] for e in rng.permutation(d.E)])
    idx = order.reshape(d.k, T).T.astype(np.int32).copy()
    assert all(len(set(r)) == d.k for r in idx.tolist())
    w = ms.bf16_bits(rng.uniform(0.05, 0.3, idx.shape))
    g = gh.upload(inp)
    out = gh.gpu_experts(g, idx, w)
    pick = set(sample_rows(T, 32, seed=5).tolist())
    for e, c in special.items():
        toks = np.flatnonzero((idx == e).any(axis=1))  # the expert's rows in sorted order
        for r in (0, 126, 127, 128, 129, 254, 255, 256, 257, 383, 384, 511, 512, 513, c - 1):
            if 0 <= r < c:
                pick.add(int(toks[r]))
    rows = np.array(sorted(pick))
    gh.compare_out(out[rows], gh.oracle_experts_rows(inp, idx, w, rows), "ragged tiles",
                   sub_explainer(gh.explainer(inp, idx, w), rows))


def test_single_expert_identity():
    """E = 1, k = 1, per_expert_scale = 1: the layer is one dense 4-bit GeGLU MLP."""
    d = ms.Dims(T=40, H=256, E=1, k=1, inter=128)
    inp = dataclasses.replace(ms.make_custom(d, seed=7), pes=np.full(1, 0x3F80, np.uint16))
    g = gh.upload(inp)
    out, idx, w = gh.gpu_forward(g)
    assert np.all(idx == 0) and np.all(w == 0x3F80)
    ref = gh.oracle_route(inp)
    gh.compare_out(out, gh.oracle_experts_rows(inp, ref["idx"], ref["w"]), "identity")


def test_deterministic_and_workspace_forms():
    inp, g, ref = layer("canvas")
    a, _, _ = gh.gpu_forward(g)
    b, _, _ = gh.gpu_forward(g)
    assert np.array_equal(a, b), "two runs differ"
    import bit_quantized_moe_layer_gb300 as moe
    ws = torch.empty(moe.workspace_bytes(g.d), dtype=torch.uint8, device="cuda")
    c, _, _ = gh.gpu_forward(g, workspace=ws)
    assert np.array_equal(a, c), "caller workspace differs from library workspace"


@pytest.mark.parametrize("pinned", [True, False])
def test_hostio_matches_device_call(pinned):
    """Pinned host buffers (used through their device mapping: a copy kernel
    reads x, the combine writes out) and pageable ones (copied through the
    copy engines) give the device call's output bit for bit."""
    import bit_quantized_moe_layer_gb300 as moe
    inp, g, ref = layer("canvas")
    a, _, _ = gh.gpu_forward(g)
    x_host = torch.from_numpy(inp.x.view(np.int16).copy())
    out_host = torch.full((g.d.T, g.d.H), 0x7FC0, dtype=torch.int16)
    if pinned:
        x_host, out_host = x_host.pin_memory(), out_host.pin_memory()
    moe.moe_forward_hostio(g.d, x_host, g.layer.router_w, g.layer.router_scale, g.layer.pes,
                           g.layer.gate_up, g.layer.down, out_host)
    assert np.array_equal(out_host.numpy().view(np.uint16), a)


def test_timing_and_error_word():
    import bit_quantized_moe_layer_gb300 as moe
    inp, g, ref = layer("canvas")
    moe.timing_enable(True)
    for _ in range(3):
        gh.gpu_forward(g)
    ms_per_stage, calls = moe.timing_read()
    moe.timing_enable(False)
    assert calls == 3
    assert all(v > 0 for v in ms_per_stage.values()), ms_per_stage
    assert moe.device_error() == 0


def test_bad_expert_id_is_flagged_not_faulted():
    """An out-of-range expert id is dropped by the dispatch kernel (bounds
    checked): its slot gets inv = -1 and no row, and the device error word
    reports it."""
    import bit_quantized_moe_layer_gb300 as moe
    d = moe.dims(4, 256, 8, 2, 128)
    idx = np.array([[0, 1], [2, 8], [3, 4], [5, -3]], np.int32)
    moe.device_error()
    perm, off, inv = gh.gpu_dispatch(d, idx)
    assert off[-1] == 6 and inv[3] == -1 and inv[7] == -1
    assert sorted(perm[:6].tolist()) == [0, 1, 2, 4, 5, 6]
    assert moe.device_error() & 2


@pytest.mark.parametrize("T", [16, 1200])
def test_bad_expert_id_in_experts_call(T):
    """A slot with an out-of-range expert id adds nothing to its token's
    output: the result equals the call with that slot moved to a valid
    expert with weight 0, bit for bit, and the error word is raised. The
    caller workspace is filled with garbage first, so a stale inverse index
    would read outside it. T = 1200 runs the three-kernel dispatch."""
    import bit_quantized_moe_layer_gb300 as moe
    inp = ms.make_layer("canvas", T=T, seed=12)
    g = gh.upload(inp)
    rng = np.random.default_rng(12)
    idx = np.stack([rng.choice(128, 8, replace=False) for _ in range(T)]).astype(np.int32)
    w = ms.bf16_bits(rng.uniform(0.05, 0.3, (T, 8)))
    bad_idx, zero_w = idx.copy(), w.copy()
    bad_idx[T // 2, 3] = 128
    bad_idx[T - 1, 0] = -1
    for t, j in ((T // 2, 3), (T - 1, 0)):
        zero_w[t, j] = 0
    ws = torch.full((moe.workspace_bytes(g.d),), 0x7F, dtype=torch.uint8, device="cuda")
    moe.device_error()
    got = gh.gpu_experts(g, bad_idx, w, workspace=ws)
    assert moe.device_error() & 2
    want = gh.gpu_experts(g, idx, zero_w)
    assert np.all(np.isfinite(gh.f64(got)))
    assert np.array_equal(got, want)


def test_geglu_ties_and_tails_exact():
    """Exact bf16 ties of gate*up (large gates) and the far negative tail go
    through the CUDA GeGLU epilogue exactly as through the oracle."""
    import oracle_checks as oc
    rng = np.random.default_rng(11)
    gates = [5.5, 7.5, -5.5, 9.0, -7.0625, -12.0, 3.0, 0.0]
    ups = [2.0625, 1.03125, -2.0625, 1.5, -1.3671875, 4.0, 2.0, 1.0]
    xr = np.concatenate([ms.bf16_bits(np.array(list(zip(gates, ups)), np.float32)),
                         ms.bf16_bits(rng.standard_normal((24, 2)) * 3)])
    want, h0 = oc._one_hot_layer(None, xr, 9, 9, 9)
    d = ms.Dims(T=len(xr), H=256, E=1, k=1, inter=128)
    I, H = d.inter, d.H
    # the same one-hot layer on the GPU
    gu_w = np.full((1, 2 * I, H // 8), 0x88888888, np.uint32)
    dn_w = np.full((1, H, I // 8), 0x88888888, np.uint32)
    n0, K0, K1 = 37, 70, 201
    gu_w[0, n0, K0 // 8] = np.uint32(0x88888888 ^ (1 << (4 * (K0 % 8))))
    gu_w[0, I + n0, K1 // 8] = np.uint32(0x88888888 ^ (1 << (4 * (K1 % 8))))
    dn_w[0, h0, n0 // 8] = np.uint32(0x88888888 ^ (1 << (4 * (n0 % 8))))
    ones = lambda n, kk: np.full((1, n, kk // 64), 0x3F80, np.uint16)
    m8 = lambda n, kk: np.full((1, n, kk // 64), 0xC100, np.uint16)
    x = np.zeros((d.T, H), np.uint16)
    x[:, K0], x[:, K1] = xr[:, 0], xr[:, 1]
    inp = ms.LayerInputs(d, x, np.zeros((1, H), np.uint16), np.full(H, 0x3F80, np.uint16),
                         np.full(1, 0x3F80, np.uint16), gu_w, ones(2 * I, H), m8(2 * I, H),
                         dn_w, ones(H, I), m8(H, I))
    g = gh.upload(inp)
    out = gh.gpu_experts(g, np.zeros((d.T, 1), np.int32), np.full((d.T, 1), 0x3F80, np.uint16))
    assert np.array_equal(out, want), np.flatnonzero((out != want).any(1))
