"""Host-side arithmetic of bench.py on CPU: the algorithmic bytes and FLOPs behind
the roofline, the kernel count per step, the lookup of profiled DRAM traffic (and
its voiding when the kernel source changes), and the size of the L2 hint that the
library's decode-size router launch issues.  Expected values are worked out by
hand from the shapes in the comments, not by calling the functions under test.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from top_routing_grouped_gating_gb300 import workloads as W  # noqa: E402

MB = 1 << 20


def test_gemm_weight_and_implementation_bytes_30b_decode():
    cfg = W.CONFIGS["qwen3_30b_a3b_decode"]
    # 112 active experts x (w13 2048x1536 + down 768x2048) bf16 = 112 x 9,437,184 B
    assert bench.gemm_weight_bytes(cfg, 112) == 112 * 9_437_184 == 1_056_964_608
    # P = 256 pairs: x rows 256x2048 bf16 in (1 MiB), h 256x768 out and in (2 x 384 KiB),
    # y2 256x2048 out (1 MiB); reported apart, not credited
    assert bench.gemm_implementation_bytes(cfg) == 1_048_576 + 2 * 393_216 + 1_048_576 == 2_883_584


def test_layer_algorithmic_bytes_30b_decode():
    cfg = W.CONFIGS["qwen3_30b_a3b_decode"]
    # weights 1,056,964,608 + W_g 2048x128 fp32 (1 MiB) + x and out 32x2048 bf16 (128 KiB each)
    # + top-k ids and weights 256 x (4 + 4) B
    assert bench.layer_algorithmic_bytes(cfg, 112) == 1_056_964_608 + 1_048_576 + 2 * 131_072 + 2048


def test_layer_algorithmic_bytes_mxfp8_prefill():
    cfg = W.CONFIGS["mxfp8_prefill"]
    # e4m3 codes + one E8M0 byte per 32: 3*4096*1536 = 18,874,368 elements per expert x 33/32
    weights = 128 * 19_464_192
    wg = 4096 * 128 * 4
    # x and r in, out and residual_out written: four 4096x4096 bf16 tensors; norm weight 4096 bf16
    acts = 4 * 33_554_432 + 8192
    ids = 32768 * 8
    assert bench.layer_algorithmic_bytes(cfg, 128) == weights + wg + acts + ids


def test_gemm_bytes_mxfp8_and_w4a8():
    mx = W.CONFIGS["mxfp8_decode"]
    per_expert = 3 * 4096 * 1536 * 33 // 32
    assert bench.gemm_weight_bytes(mx, 100) == 100 * per_expert
    P = 64 * 8
    assert bench.gemm_implementation_bytes(mx) == P * 4096 * 33 // 32 + 2 * P * 1536 * 33 // 32 + P * 4096 * 2
    w4 = W.CONFIGS["w4a8_decode"]
    # e2m1: half a byte per code, plus the same scale bytes: 17/32 of a byte per element
    assert bench.gemm_weight_bytes(w4, 100) == 100 * (3 * 4096 * 1536 * 17 // 32)


def test_implementation_bytes_count_only_routed_pairs():
    cfg = W.CONFIGS["zero_experts_decode"]
    full = bench.gemm_implementation_bytes(cfg)
    fewer = bench.gemm_implementation_bytes(cfg, pairs=200)
    # 56 pairs fewer, each H*2 in + 2*I*2 for h + H*2 out = 4096 + 3072 + 4096 bytes
    assert full - fewer == 56 * (4096 + 3072 + 4096)


def test_hbm_roofline_nets_out_the_l2_hint():
    # 1.0e9 weight bytes of which 0.2e9 were asked into L2 by the router launch, a 0.1 ms
    # GEMM: 0.8e9 B / 1e-4 s = 8000 GB/s; 1.2e9 layer bytes in a 0.2 ms step: 6000 GB/s
    r = bench.hbm_roofline(1_000_000_000, 1_200_000_000, 200_000_000, 0.1, 0.2, 8000.0)
    assert r["achieved"] == pytest.approx(8000.0)
    assert r["frac"] == pytest.approx(1.0)
    assert r["step_achieved"] == pytest.approx(6000.0)
    assert r["step_frac"] == pytest.approx(0.75)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"


def test_tensor_roofline():
    # 2.0e12 FLOP in a 1 ms GEMM inside a 1.25 ms step against a 2500 TFLOP/s peak
    r = bench.tensor_roofline(2.0e12, 1.0, 1.25, 2500.0)
    assert r["achieved"] == pytest.approx(2000.0)
    assert r["frac"] == pytest.approx(0.8)
    assert r["step_frac"] == pytest.approx(0.64)


def test_oracle_sample_is_the_same_in_both_arms():
    # decode: the whole batch per oracle call; prefill: 64 consecutive tokens, wrapping
    assert bench.oracle_sample_tokens(W.CONFIGS["qwen3_30b_a3b_decode"]) == 32
    assert bench.oracle_sample_tokens(W.CONFIGS["qwen3_235b_a22b_decode"]) == 64
    pre = W.CONFIGS["qwen3_235b_a22b_prefill"]
    assert bench.oracle_sample_tokens(pre) == 64
    assert bench.oracle_sample_rows(pre, 0) == list(range(64))
    assert bench.oracle_sample_rows(pre, 1) == list(range(64, 128))
    assert bench.oracle_sample_rows(pre, 128) == list(range(64))          # 128 x 64 = 8192 wraps to 0
    assert bench.oracle_sample_rows(W.CONFIGS["qwen3_30b_a3b_decode"], 3) == list(range(32))


def test_suite_ends_with_the_largest_workload():
    sizes = [W.CONFIGS[n].T * W.CONFIGS[n].H * W.CONFIGS[n].I for n in bench.SUITE]
    assert bench.HEADLINE == "qwen3_235b_a22b_prefill" == bench.SUITE[-1]
    assert sizes[-1] == max(sizes)


def test_gemm_flops():
    # Zipf prefill: 2 * T*k * 3 * H * I = 2 * 32768 * 3 * 2048 * 768
    assert bench.gemm_flops(W.CONFIGS["qwen3_30b_a3b_prefill_zipf"]) == 309_237_645_312.0
    # 235B prefill: 2 * 65536 * 3 * 4096 * 1536
    assert bench.gemm_flops(W.CONFIGS["qwen3_235b_a22b_prefill"]) == 2_473_901_162_496.0


@pytest.mark.parametrize("name,router,expect", [
    ("qwen3_30b_a3b_decode", True, 5),          # router, gating+routing, gather, GEMM, finalize
    ("qwen3_30b_a3b_decode", False, 4),         # logits given: no router launch
    ("qwen3_30b_a3b_prefill_zipf", True, 9),    # split/pack + TC GEMM router, 3 routing kernels
    ("mxfp8_prefill", True, 10),                # norm/quant (+ the router's split), pack +
                                                # TC GEMM router, gating, 3 routing, expand,
                                                # GEMM, finalize
    ("qwen3_30b_a3b_decode_prenorm", True, 6),  # + fused add+RMSNorm+cast
])
def test_launches_per_step(name, router, expect):
    assert bench.launches_per_step(W.CONFIGS[name], router=router) == expect


def test_l2_hint_bytes():
    sms, l2 = 152, 126 * MB
    # bf16, H = 2048: 5/8 of 152 x 128 rows x 4096 B = 49,807,360 B (below 5/8 of L2)
    assert bench.l2_hint_bytes(W.CONFIGS["qwen3_30b_a3b_decode"], sms, l2) == 49_807_360
    # bf16, H = 4096: the first wave (99.6 MB x 5/8 of 159 MB) is capped at 5/8 of L2
    assert bench.l2_hint_bytes(W.CONFIGS["qwen3_235b_a22b_decode"], sms, l2) == 126 * MB * 5 // 8
    # e4m3 rows are H bytes, packed e2m1 rows H / 2
    assert bench.l2_hint_bytes(W.CONFIGS["mxfp8_decode"], sms, l2) == 152 * 128 * 4096 * 5 // 8
    assert bench.l2_hint_bytes(W.CONFIGS["w4a8_decode"], sms, l2) == 152 * 128 * 2048 * 5 // 8
    # capped by w13 itself: 8 experts x 256 rows x 512 B = 1 MB
    tiny = W.with_shape(W.CONFIGS["tiny"], E=8, H=256, I=128)
    assert bench.l2_hint_bytes(tiny, sms, l2) == 8 * 256 * 512
    # prefill sizes (T > 64) use the tensor-core router, which issues no hint
    assert bench.l2_hint_bytes(W.CONFIGS["qwen3_30b_a3b_prefill_zipf"], sms, l2) == 0


def test_profiled_traffic_lookup_and_voiding(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "top_routing_grouped_gating_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "gmm.cu").write_text("// kernel v1\n")
    (src / "gmm_mx.cu").write_text("// mx kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.file_sha(str(src / "gmm.cu"))
    (tmp_path / "profiles" / "grouped_gemm_qwen3_30b_a3b_decode.md").write_text(
        f"kernel_source_sha256_16: {sha}\ntraffic_bytes_per_launch: 1062940744\n")
    assert bench.profiled_traffic("qwen3_30b_a3b_decode") == 1062940744.0
    assert bench.profiled_traffic("qwen3_235b_a22b_decode") is None          # no summary
    (src / "gmm.cu").write_text("// kernel v2\n")                             # kernel changed
    assert bench.profiled_traffic("qwen3_30b_a3b_decode") is None
    # block-scaled workloads are checked against the block-scaled kernel's source
    mx_sha = bench.file_sha(str(src / "gmm_mx.cu"))
    (tmp_path / "profiles" / "grouped_gemm_mxfp8_prefill.md").write_text(
        f"kernel_source_sha256_16: {mx_sha}\ntraffic_bytes_per_launch: 2.5e9\n")
    assert bench.profiled_traffic("mxfp8_prefill") == 2.5e9


def test_parse_shape():
    assert bench.parse_shape("E=32,T=2048") == {"E": 32, "T": 2048}
    assert bench.parse_shape("") == {}
    with pytest.raises(SystemExit):
        bench.parse_shape("Z=3")
    with pytest.raises(SystemExit):
        bench.parse_shape("E=x")


def test_clock_samples_keep_the_loaded_ones():
    # index, sm, max sm, power, active mask, hw, hw thermal, sw thermal, sw power cap, idle
    text = "\n".join([
        "0, 2070, 2070, 180.5, 0x0000000000000001, Not Active, Not Active, Not Active, Not Active, Active",
        "0, 1830, 2070, 1210.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active, Not Active",
        "0, 1800, 2070, 1390.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active, Not Active",
        "0, 1860, 2070, 1250.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 175.0, 0x0000000000000001, Not Active, Not Active, Not Active, Not Active, Active",
    ])
    c = bench.parse_clock_samples(text)
    assert c["samples"] == 5 and c["samples_under_load"] == 3
    assert c["sm_mhz"] == 1830.0                    # median of 1830, 1800, 1860
    assert c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    # no loaded sample: all samples, and the count says so
    idle = bench.parse_clock_samples(text.splitlines()[0] + "\n" + text.splitlines()[4])
    assert idle["samples_under_load"] == 0 and idle["sm_mhz"] == 2070.0
    assert bench.parse_clock_samples("") is None


def test_sustained_peak_is_read_when_present(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.sustained_bf16_peak() is None                    # no file
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6800, "bf16_tflops": 1900}')
    assert bench.sustained_bf16_peak() is None                    # no sustained figure
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        '{"hbm_gbs": 6800, "bf16_tflops": 1900, "bf16_tflops_sustained": 1700.5}')
    assert bench.sustained_bf16_peak() == 1700.5
