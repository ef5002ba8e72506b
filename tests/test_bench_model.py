"""bench.py's roofline arithmetic (CPU): the algorithmic bytes and flops it
divides by, against values worked out by hand for the canvas layer, the
dense MLP and the tied head."""
import bench
import moe_synth as ms

PEAKS = dict(hbm=6775.6, tc=1879.3, tc_sustained=1697.1, source="measured")


def test_expert_weight_bytes_canvas():
    # gate_up: 1408 x 2816 nibbles = 1,982,464 B + (1408 x 44 groups) x 2 (scale, bias) x 2 B = 247,808 B
    # down:    2816 x 704 nibbles  =   991,232 B + (2816 x 11 groups) x 2 x 2 B               = 123,904 B
    assert bench.layer_bytes(ms.WORKLOADS["canvas"].dims) == (2_230_272, 1_115_136)


def test_layer_roofline_canvas_is_hbm_bound():
    d = ms.WORKLOADS["canvas"].dims
    m = bench.roofline_model(d, 128, PEAKS)
    # weights of 128 experts + router weight [128, 2816] + scale [2816] + pes [128] + x and out [256, 2816], bf16
    want_bytes = 128 * (2_230_272 + 1_115_136) + 128 * 2816 * 2 + 2816 * 2 + 128 * 2 + 2 * 256 * 2816 * 2
    assert m["bytes"] == want_bytes == 431_822_592
    # router 2 T H E, experts per slot 2 H (2 I) + 2 I H
    assert m["flops"] == 2 * 256 * 2816 * 128 + 2048 * (2 * 2816 * 1408 + 2 * 704 * 2816)
    assert m["bound"] == "hbm"
    assert abs(m["t_roof_s"] * 1e6 - 63.73) < 0.01


def test_layer_roofline_prefill_is_tensor_bound():
    m = bench.roofline_model(ms.WORKLOADS["prefill"].dims, 128, PEAKS)
    assert m["bound"] == "tensor"
    assert abs(m["t_roof_s"] * 1e6 - 209.0) < 0.1


def test_dense_mlp_model():
    dn = ms.make_dense(256, H=2816, I=2112, seed=0)
    m = bench.dense_model(dn)
    # three linears of 2112 x 2816: 3 x 2,973,696 B packed + 3 x (2112 x 44) x 2 x 2 B; x and out [256, 2816] bf16
    assert m["bytes"] == 3 * 2112 * 2816 // 2 + 3 * 2112 * 44 * 4 + 2 * 256 * 2816 * 2 == 12_919_808
    assert m["flops"] == 2 * 256 * 2816 * 3 * 2112 == 9_135_194_112
    assert m["gate_up_flops"] == 2 * 256 * 2816 * 2 * 2112


def test_head_report():
    r = bench.head_report(256, 2816, 262144, 0.3, {"gate_up": 3.0, "gather": 0.2}, 10, PEAKS, 1)
    # table 262144 x 2816 nibbles + (262144 x 44) x 2 x 2 B; h in bf16; fp32 logits out
    want = 262144 * 2816 // 2 + 262144 * 44 * 4 + 256 * 2816 * 2 + 256 * 262144 * 4
    assert r["roofline"]["bytes"] == want == 685_113_344
    assert r["roofline"]["flops"] == 2 * 256 * 2816 * 262144
    assert r["roofline"]["bound"] == "tensor"
    assert abs(r["roofline"]["t_roof_us"] - 201.1) < 0.1
    assert abs(r["gemm_kernel"]["ms_per_launch"] - 0.3) < 1e-12  # 3.0 ms over 10 calls
    assert abs(r["value"] - 256 / 0.3e-3) < 1e-6
