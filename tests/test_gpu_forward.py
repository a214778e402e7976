"""End-to-end parity of moe_forward (one C-ABI call for the whole layer) against the
CPU oracle on the seeded workloads, at their full sizes.

Routing is checked bit-exactly by feeding both sides the oracle's fp32 logits
(logits_override), so the comparison of outputs cannot be masked by near-tie
routing flips of the fp32 router.  Every configuration, the two prefill layers
(4096 and 8192 tokens) included, is compared on every token, so every active
expert and every expert's last token block is checked; the oracle's per-expert
loop runs on a host thread pool there.  A separate test runs the GPU router and
compares the tokens whose routing margin is larger than the router's error bound.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import top_routing_grouped_gating_gb300 as moe
from oracle import moe_oracle as O
from tests._helpers import (LazyExperts, assert_close_layer, expert_coverage, forced_topk_logits,
                           oracle_threads, routing_margin_ok, to_np)
from top_routing_grouped_gating_gb300 import workloads as W

pytestmark = pytest.mark.gpu

FULL_ORACLE_MAX_T = 64


@pytest.fixture(scope="module")
def layers(cuda_dev):
    cache = {}

    def get(name, **kw):
        key = (name, tuple(sorted(kw.items())))
        if key not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            cfg = W.with_shape(W.CONFIGS[name], **kw) if kw else W.CONFIGS[name]
            inp = W.make_inputs(cfg, device="cuda")
            layer = moe.MoELayer(inp["Wg"], inp["w13"], inp["down"], cfg.k)
            cache[key] = (cfg, inp, layer)
        return cache[key]
    return get


def _check_forward(cfg, inp, layer, sample=None, threads=1):
    x, Wg = inp["x"], inp["Wg"]
    xn = to_np(x)
    lg32 = O.router_logits_f32(xn, to_np(Wg))
    out, ids, w = layer(x, logits_override=torch.from_numpy(lg32).to(x.device))
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    r_ids, r_w = O.gating_topk_softmax(lg32, cfg.k)
    np.testing.assert_array_equal(to_np(ids), r_ids)
    np.testing.assert_allclose(to_np(w), r_w, rtol=2e-6, atol=1e-7)
    rows = np.arange(cfg.T) if sample is None else sample
    with ThreadPoolExecutor(threads) as pool:
        ref = O.moe_forward(xn[rows], None, LazyExperts(inp["w13"]), LazyExperts(inp["down"]), cfg.k,
                            logits32=lg32[rows], keep_intermediates=False,
                            expert_map=pool.map if threads > 1 else map)
    hit, active = expert_coverage(r_ids, rows, cfg.E)
    print(f"{cfg.name}: {len(rows)}/{cfg.T} tokens compared, {hit}/{active} active experts covered")
    return assert_close_layer(to_np(out)[rows], ref["out"], what=cfg.name)


@pytest.mark.parametrize("name", ["tiny", "qwen3_30b_a3b_decode", "qwen3_235b_a22b_decode"])
def test_forward_full_oracle(layers, name):
    cfg, inp, layer = layers(name)
    _check_forward(cfg, inp, layer)


@pytest.mark.parametrize("name", ["qwen3_30b_a3b_prefill_zipf", "qwen3_235b_a22b_prefill"])
def test_forward_prefill_full_oracle(layers, name):
    """The prefill layers at full size (4096 tokens, Zipf-skewed loads; 8192 tokens,
    uniform) against the oracle on every token: every active expert, every token
    block of the CTA-pair GEMM and every expert's last, partial block."""
    cfg, inp, layer = layers(name)
    _check_forward(cfg, inp, layer, threads=oracle_threads())


@pytest.mark.parametrize("T", [1, 3, 17, 100])
def test_forward_ragged_token_counts(layers, T):
    cfg, inp, layer = layers("qwen3_30b_a3b_decode", T=T)
    _check_forward(cfg, inp, layer)


def test_forward_single_expert_is_dense_mlp(layers):
    cfg, inp, layer = layers("tiny", E=1, k=1, T=40)
    _check_forward(cfg, inp, layer)


@pytest.mark.parametrize("T,E,k", [(40, 256, 32),    # the largest expert count and top-k
                                   (33, 4, 4),       # k = E: every token visits every expert
                                   (700, 256, 8)])   # 256 experts, multi-CTA routing (P > 4096)
def test_forward_limits(layers, T, E, k):
    cfg, inp, layer = layers("tiny", T=T, E=E, k=k, H=256, I=128)
    _check_forward(cfg, inp, layer)


@pytest.mark.parametrize("counts,light", [
    ([256, 257, 255, 512, 513, 33, 40, 254], 0),  # no expert of <= 32 rows: 256-row blocks
    ([224, 225, 223, 448, 449, 1, 0, 32], 1),     # 1 and 32 rows run light: 224-row heavy blocks
    ([224, 225, 223, 448, 449, 1, 0, 32], 2),     # the same experts all on the one pipeline
    ([1, 16, 17, 33, 255, 256, 480, 990], 1),     # light 1-17; heavy halves of 17 to 112 rows
    ([1, 16, 17, 33, 255, 256, 480, 990], 0),     # the kernel's own choice
])
def test_forward_token_block_boundaries(layers, counts, light):
    """Expert loads forced through designed logits onto both sides of the token
    blocks of the CTA-pair GEMM: 256-row blocks when every expert runs on one
    pipeline, 224-row heavy blocks next to the light pipeline's experts (up to 32
    rows, one with a single row, one with none; the light pipeline forced on), and
    the thin boxes of units whose half block has at most 16 rows."""
    k = 2
    T = sum(counts) // k
    cfg, inp, layer = layers("tiny", T=T, E=len(counts), k=k)
    lg = forced_topk_logits(counts, k, seed=7)
    x = inp["x"]
    moe.debug_set_pair_light(light)
    try:
        out, ids, w = layer(x, logits_override=torch.from_numpy(lg).to(x.device))
        torch.cuda.synchronize()
    finally:
        moe.debug_set_pair_light(0)
    assert moe.get_device_status() == 0
    r_ids, r_w = O.gating_topk_softmax(lg, k)
    np.testing.assert_array_equal(np.bincount(r_ids.ravel(), minlength=cfg.E), counts)
    np.testing.assert_array_equal(to_np(ids), r_ids)
    ref = O.moe_forward(to_np(x), None, LazyExperts(inp["w13"]), LazyExperts(inp["down"]), k,
                        logits32=lg, keep_intermediates=False)
    assert_close_layer(to_np(out), ref["out"], what="token-block boundaries")


def test_forward_prefill_one_cta_tiles(layers):
    """Prefill-size token blocks with a hidden size (384) that does not split into
    256-row weight blocks: both projections run on the one-CTA wide-tile kernel
    instead of the CTA-pair kernel."""
    cfg, inp, layer = layers("tiny", T=300, E=8, k=4, H=384, I=128)
    assert cfg.T * cfg.k > 16 * cfg.E and cfg.H % 256 != 0
    _check_forward(cfg, inp, layer)


@pytest.mark.parametrize("T", [64, 300])
def test_forward_with_gpu_router(layers, T):
    cfg, inp, layer = layers("qwen3_30b_a3b_decode", T=T)
    x, Wg = inp["x"], inp["Wg"]
    out, ids, w = layer(x)
    torch.cuda.synchronize()
    xn = to_np(x).astype(np.float64)
    Wn = to_np(Wg).astype(np.float64)
    lg = O.router_logits_f32(xn, Wn)
    tol = 1e-5 * (np.abs(xn) @ np.abs(Wn)).max(axis=1)
    safe = routing_margin_ok(lg, cfg.k, tol)
    assert safe.sum() >= cfg.T * 0.9
    r_ids, _ = O.gating_topk_softmax(lg, cfg.k)
    np.testing.assert_array_equal(to_np(ids)[safe], r_ids[safe])
    rows = np.nonzero(safe)[0]
    ref = O.moe_forward(to_np(x)[rows], None, LazyExperts(inp["w13"]), LazyExperts(inp["down"]), cfg.k,
                        logits32=lg[rows], keep_intermediates=False)
    assert_close_layer(to_np(out)[rows], ref["out"])


def test_forward_is_deterministic(layers):
    cfg, inp, layer = layers("qwen3_30b_a3b_prefill_zipf")
    a = layer(inp["x"])[0].clone()
    b = layer(inp["x"])[0]
    assert torch.equal(a, b)
    assert moe.get_device_status() == 0


def test_graphed_layer_matches_direct_calls(layers):
    cfg, inp, layer = layers("qwen3_30b_a3b_decode")
    g = layer.capture(cfg.T)
    x = inp["x"]
    ref = layer(x)[0].clone()
    out = g(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    x2 = torch.flip(x, dims=[0]).contiguous()
    out2 = g(x2).clone()
    torch.cuda.synchronize()
    assert torch.equal(out2, layer(x2)[0])
    assert moe.get_device_status() == 0
