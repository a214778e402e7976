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


def test_algorithmic_bytes_30b_decode():
    cfg = W.CONFIGS["qwen3_30b_a3b_decode"]
    # 112 active experts x (w13 2048x1536 + down 768x2048) bf16 = 112 x 9,437,184 B
    weights = 112 * 9_437_184
    # P = 256 pairs: x rows 256x2048 bf16 in, h 256x768 out and in, y2 256x2048 out
    acts = 1_048_576 + 2 * 393_216 + 1_048_576
    assert bench.algorithmic_gemm_bytes(cfg, 112) == weights + acts == 1_059_848_192


def test_algorithmic_bytes_mxfp8_and_w4a8():
    mx = W.CONFIGS["mxfp8_decode"]
    # e4m3 codes + one E8M0 byte per 32: 3*4096*1536 elements per expert x 33/32
    per_expert = 3 * 4096 * 1536 * 33 // 32
    P = 64 * 8
    acts = P * 4096 * 33 // 32 + 2 * P * 1536 * 33 // 32 + P * 4096 * 2
    assert bench.algorithmic_gemm_bytes(mx, 100) == 100 * per_expert + acts
    w4 = W.CONFIGS["w4a8_decode"]
    # e2m1: half a byte per code, plus the same scale bytes: 17/32 of a byte per element
    assert bench.algorithmic_gemm_bytes(w4, 100) == 100 * (3 * 4096 * 1536 * 17 // 32) + acts


def test_algorithmic_bytes_count_only_routed_pairs():
    cfg = W.CONFIGS["zero_experts_decode"]
    full = bench.algorithmic_gemm_bytes(cfg, 100)
    fewer = bench.algorithmic_gemm_bytes(cfg, 100, pairs=200)
    # 56 pairs fewer, each H*2 in + 2*I*2 for h + H*2 out = 4096 + 3072 + 4096 bytes
    assert full - fewer == 56 * (4096 + 3072 + 4096)


def test_gemm_flops():
    # Zipf prefill: 2 * T*k * 3 * H * I = 2 * 32768 * 3 * 2048 * 768
    assert bench.gemm_flops(W.CONFIGS["qwen3_30b_a3b_prefill_zipf"]) == 309_237_645_312.0
    # 235B prefill: 2 * 65536 * 3 * 4096 * 1536
    assert bench.gemm_flops(W.CONFIGS["qwen3_235b_a22b_prefill"]) == 2_473_901_162_496.0


@pytest.mark.parametrize("name,router,expect", [
    ("qwen3_30b_a3b_decode", True, 5),          # router, gating+routing, gather, GEMM, finalize
    ("qwen3_30b_a3b_decode", False, 4),         # logits given: no router launch
    ("qwen3_30b_a3b_prefill_zipf", True, 9),    # split/pack + TC GEMM router, 3 routing kernels
    ("mxfp8_prefill", True, 11),                # norm/quant, 3 router, gating, 3 routing,
                                                # expand, GEMM, finalize
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
