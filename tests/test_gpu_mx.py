"""MXFP8 path on the GPU against the CPU oracle (via the C ABI).

Bit-exact where both sides quantise identical inputs (the standalone quantiser on
seeded fp32 data, the weight pre-quantisation of bf16 weights).  Where the GPU
quantises its own fp32 RMSNorm output, the codes are compared through their
dequantised values, since the oracle's fp64 normalisation can sit on the other
side of a rounding boundary.  The layer output must stay within relative
Frobenius error 4e-2 of the oracle run on dequantised inputs.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import top_routing_grouped_gating_gb300 as moe
from oracle import moe_oracle as O
from tests._helpers import (REL_FRO_MX, LazyExperts, expert_coverage, forced_topk_logits, oracle_threads,
                           rel_fro, to_np)
from top_routing_grouped_gating_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def tricky_fp32(rows, n, seed):
    """Seeded fp32 data with MX edge cases: zero blocks, powers of two, e4m3
    rounding midpoints, saturating values, tiny and negative-zero entries."""
    rng = np.random.default_rng(seed)
    y = rng.standard_normal((rows, n)) * np.exp2(rng.integers(-30, 30, size=(rows, 1)))
    yb = y.reshape(rows, n // 32, 32)
    yb[0, 0] = 0.0
    yb[0, 1] = -0.0
    yb[1, 0] = np.exp2(np.arange(32) - 16.0)
    codes = np.arange(1, 126)
    mids = (O.e4m3_decode(codes) + O.e4m3_decode(codes + 1)) / 2
    yb[2, :, :] = rng.choice(mids, size=yb[2].shape) * rng.choice([-1, 1], size=yb[2].shape)
    yb[2, :, 0] = 448.0 * 1.1           # block max: saturating neighbours
    yb[3, 0, :] = 500.0                 # whole block saturates
    yb[3, 1, :] = 1e-42                 # fp32 subnormals
    yb[3, 1, 3] = -0.0
    return y.reshape(rows, n).astype(np.float32)


def test_mx_quantize_bit_exact(cuda_dev):
    y = tricky_fp32(64, 512, seed=1)
    q, sc = moe.mx_quantize(torch.from_numpy(y).to(cuda_dev))
    rq, rsc = O.mx_quantize(y.astype(np.float64))
    np.testing.assert_array_equal(to_np(sc), rsc)
    np.testing.assert_array_equal(to_np(q), rq)


def test_add_rmsnorm_mxquant(cuda_dev):
    cfg = W.with_shape(W.CONFIGS["mxfp8_prefill"], T=64)
    inp = W.make_inputs(cfg, weights=True, device="cpu")
    x, r, w = inp["x"], inp["r"], inp["norm_w"]
    res, y32, q, sc = moe.add_rmsnorm_mxquant(x.to(cuda_dev), r.to(cuda_dev), w.to(cuda_dev), cfg.eps)
    s, y = O.add_rmsnorm(to_np(x), to_np(r), to_np(w), cfg.eps)
    ref_res = torch.from_numpy(s).to(torch.bfloat16)
    assert torch.equal(res.cpu().view(torch.int16), ref_res.view(torch.int16))
    # fp32 normalisation: a few roundings (sum of squares over H, rsqrt, two products)
    np.testing.assert_allclose(to_np(y32), y, rtol=2e-5, atol=1e-6)
    rq, rsc = O.mx_quantize(y)
    deq = O.mx_dequantize(to_np(q).astype(np.uint8), to_np(sc).astype(np.uint8))
    rdeq = O.mx_dequantize(rq, rsc)
    diff = deq != rdeq
    assert diff.mean() < 2e-3
    # any disagreement is one e4m3 step of that block (a rounding-boundary straddle)
    step = np.exp2(np.repeat(to_np(sc).astype(np.float64), 32, axis=1) - 127) * 2.0 ** -2
    assert np.all(np.abs(deq - rdeq)[diff] <= np.maximum(np.abs(rdeq[diff]) * 2.0 ** -3, step[diff]))
    # residual-free variant
    _, y0, _, _ = moe.add_rmsnorm_mxquant(x.to(cuda_dev), None, w.to(cuda_dev), cfg.eps)
    _, y0r = O.add_rmsnorm(to_np(x), None, to_np(w), cfg.eps)
    np.testing.assert_allclose(to_np(y0), y0r, rtol=2e-5, atol=1e-6)


def _unpack_w13(q, sf, E, H, I):
    """Packed MX w13 -> per expert (codes (H, 2I) logical, scales (H/32, 2I))."""
    q = q.reshape(E, 2 * I, H)
    sf = sf.reshape(E, 2 * I // 128, H // 128, 512)
    r = np.arange(2 * I)
    # packed row 32q + i of 128-row block b: gate feature 64b + 16q + i (i < 16), else
    # the up feature 64b + 16q + i - 16 (logical column I + that feature)
    blk, quarter, i = r // 128, (r % 128) // 32, r % 32
    col = blk * 64 + quarter * 16 + i % 16 + np.where(i < 16, 0, I)
    codes = np.empty((E, H, 2 * I), np.uint8)
    scales = np.empty((E, H // 32, 2 * I), np.uint8)
    b = np.arange(H // 32)
    for e in range(E):
        codes[e][:, col] = q[e].T
        off = (r[:, None] % 32) * 16 + ((r[:, None] % 128) // 32) * 4 + (b[None, :] % 4)
        scales[e][:, col] = sf[e][r[:, None] // 128, b[None, :] // 4, off].T
    return codes, scales


def test_pack_weights_mx_bit_exact(cuda_dev):
    E, H, I = 4, 256, 128
    g = torch.Generator().manual_seed(7)
    w13 = (torch.randn(E, H, 2 * I, generator=g) * 0.05).to(torch.bfloat16)
    down = (torch.randn(E, I, H, generator=g) * 0.05).to(torch.bfloat16)
    w13[0, :32, 5] = 0                       # an all-zero block
    w13_q, w13_sf, down_q, down_sf = moe.pack_weights_mx(w13.to(cuda_dev), down.to(cuda_dev))
    codes, scales = _unpack_w13(to_np(w13_q), to_np(w13_sf), E, H, I)
    for e in range(E):
        rq, rsc = O.mx_quantize(to_np(w13[e]).astype(np.float64).T)   # along H, per column
        np.testing.assert_array_equal(codes[e].T, rq)
        np.testing.assert_array_equal(scales[e].T, rsc)
    dq = to_np(down_q).reshape(E, H, I)
    dsf = to_np(down_sf).reshape(E, H // 128, I // 128, 512)
    n = np.arange(H)[:, None]
    b = np.arange(I // 32)[None, :]
    for e in range(E):
        rq, rsc = O.mx_quantize(to_np(down[e]).astype(np.float64).T)  # along I, per column n
        np.testing.assert_array_equal(dq[e], rq)
        got_sc = dsf[e][n // 128, b // 4, (n % 32) * 16 + ((n % 128) // 32) * 4 + b % 4]
        np.testing.assert_array_equal(got_sc, rsc)


def _mx_layer(cfg, device="cuda"):
    inp = W.make_inputs(cfg, device=device)
    layer = moe.MoELayerMX(inp["Wg"], inp["w13"], inp["down"], inp["norm_w"], cfg.k, cfg.eps)
    return inp, layer


def _check_mx_forward(cfg, inp, layer, sample=None, threads=1):
    x, r = inp["x"], inp["r"]
    xn, rn, wn = to_np(x), to_np(r), to_np(inp["norm_w"])
    _, y = O.add_rmsnorm(xn, rn, wn, cfg.eps)
    lg32 = O.router_logits_f32(y, to_np(inp["Wg"]))
    out, res, ids, w = layer(x, r, logits_override=torch.from_numpy(lg32).to(x.device))
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    r_ids, r_w = O.gating_topk_softmax(lg32, cfg.k)
    np.testing.assert_array_equal(to_np(ids), r_ids)
    rows = np.arange(cfg.T) if sample is None else sample
    with ThreadPoolExecutor(threads) as pool:
        ref = O.moe_forward_mx(xn[rows], rn[rows], wn, cfg.eps, None, LazyExperts(inp["w13"]),
                               LazyExperts(inp["down"]), cfg.k, logits32=lg32[rows],
                               expert_map=pool.map if threads > 1 else map)
    hit, active = expert_coverage(r_ids, rows, cfg.E)
    print(f"{cfg.name}: {len(rows)}/{cfg.T} tokens compared, {hit}/{active} active experts covered")
    got = to_np(out)[rows]
    assert np.all(np.isfinite(got))
    rf = rel_fro(got, ref["out"])
    assert rf <= REL_FRO_MX, f"relative Frobenius error {rf:.3e}"
    return rf


# (600, 4, 2): about 300 rows per expert, i.e. a full 256-row token block plus a short
# one, each block over 128 rows taking two scale atoms
@pytest.mark.parametrize("T,E,k,H,I", [(64, 8, 2, 256, 128), (300, 4, 2, 256, 256), (1, 8, 8, 512, 128),
                                       (600, 4, 2, 256, 128)])
def test_forward_mx_small(cuda_dev, T, E, k, H, I):
    cfg = W.with_shape(W.CONFIGS["mxfp8_prefill"], T=T, E=E, k=k, H=H, I=I)
    inp, layer = _mx_layer(cfg)
    _check_mx_forward(cfg, inp, layer)


@pytest.mark.parametrize("counts", [
    [128, 160, 161, 288, 289, 1, 0, 1021],   # one-CTA blocks: 128 rows, the last absorbing 32
    [256, 257, 272, 288, 289, 544, 545, 17],  # CTA-pair units: 256 rows, the last absorbing 32
])
def test_forward_mx_token_block_boundaries(cuda_dev, counts):
    """Expert loads on both sides of the block-scaled GEMM's token blocks, forced
    through designed logits: the CTA-pair kernel's 256-row units (an expert's last
    unit takes up to 32 more rows through a second MMA of N = 32), and the 128-row
    blocks of the one-CTA layout."""
    k = 2
    cfg = W.with_shape(W.CONFIGS["mxfp8_prefill"], T=sum(counts) // k, E=len(counts), k=k, H=256,
                       I=128)
    inp, layer = _mx_layer(cfg)
    lg = forced_topk_logits(counts, k, seed=11)
    x, r = inp["x"], inp["r"]
    out, res, ids, w = layer(x, r, logits_override=torch.from_numpy(lg).to(x.device))
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    r_ids, _ = O.gating_topk_softmax(lg, k)
    np.testing.assert_array_equal(np.bincount(r_ids.ravel(), minlength=cfg.E), counts)
    np.testing.assert_array_equal(to_np(ids), r_ids)
    ref = O.moe_forward_mx(to_np(x), to_np(r), to_np(inp["norm_w"]), cfg.eps, None,
                           LazyExperts(inp["w13"]), LazyExperts(inp["down"]), k, logits32=lg)
    got = to_np(out)
    assert np.all(np.isfinite(got))
    rf = rel_fro(got, ref["out"])
    assert rf <= REL_FRO_MX, f"relative Frobenius error {rf:.3e}"


@pytest.mark.parametrize("T,E,k", [(40, 256, 32), (700, 256, 8)])
def test_forward_mx_limits(cuda_dev, T, E, k):
    """256 experts (the routing tables' size) with the largest top-k, and with enough
    pairs for the multi-CTA routing and the wide block-scaled tiles."""
    cfg = W.with_shape(W.CONFIGS["mxfp8_prefill"], T=T, E=E, k=k, H=256, I=128)
    inp, layer = _mx_layer(cfg)
    _check_mx_forward(cfg, inp, layer)


def test_forward_mx_decode_tiles_skewed(cuda_dev):
    """Few pairs per expert on average (the narrow-tile shape) but Zipf-skewed, so the
    busiest expert spans several 32-token tiles and every 32-row group of a scale atom."""
    cfg = W.with_shape(W.CONFIGS["mxfp8_prefill"], T=256, E=16, k=1, H=256, I=128, router="zipf",
                       zipf_s=2.0)
    inp, layer = _mx_layer(cfg)
    assert cfg.T * cfg.k <= 16 * cfg.E
    _check_mx_forward(cfg, inp, layer)
    _, y = O.add_rmsnorm(to_np(inp["x"]), to_np(inp["r"]), to_np(inp["norm_w"]), cfg.eps)
    ids, _ = O.gating_topk_softmax(O.router_logits_f32(y, to_np(inp["Wg"])), cfg.k)
    assert np.bincount(ids.ravel(), minlength=cfg.E).max() > 128   # two atoms, all groups


def test_forward_mx_full_size(cuda_dev):
    """The MXFP8 prefill layer at full size (4096 tokens, 128 experts, H = 4096,
    I = 1536) against the oracle on every token, so every expert and every token
    block of the block-scaled GEMM is compared."""
    cfg = W.CONFIGS["mxfp8_prefill"]
    inp, layer = _mx_layer(cfg)
    _check_mx_forward(cfg, inp, layer, threads=oracle_threads())
    a = layer(inp["x"], inp["r"])[0].clone()
    b = layer(inp["x"], inp["r"])[0]
    assert torch.equal(a, b)


def test_forward_mx_with_gpu_router(cuda_dev):
    from tests._helpers import routing_margin_ok
    cfg = W.with_shape(W.CONFIGS["mxfp8_prefill"], T=300, E=16, k=4, H=512, I=128)
    inp, layer = _mx_layer(cfg)
    out, res, ids, w = layer(inp["x"], inp["r"])
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    _, y = O.add_rmsnorm(to_np(inp["x"]), to_np(inp["r"]), to_np(inp["norm_w"]), cfg.eps)
    Wn = to_np(inp["Wg"]).astype(np.float64)
    lg = O.router_logits_f32(y, Wn)
    # router error: fp32 RMSNorm output (~1e-6 relative) plus fp32 accumulation
    tol = 1e-5 * (np.abs(y) @ np.abs(Wn)).max(axis=1)
    safe = routing_margin_ok(lg, cfg.k, tol)
    assert safe.sum() >= 0.9 * cfg.T
    r_ids, _ = O.gating_topk_softmax(lg, cfg.k)
    np.testing.assert_array_equal(to_np(ids)[safe], r_ids[safe])
    rows = np.nonzero(safe)[0][:24]
    ref = O.moe_forward_mx(to_np(inp["x"])[rows], to_np(inp["r"])[rows], to_np(inp["norm_w"]), cfg.eps, None,
                           LazyExperts(inp["w13"]), LazyExperts(inp["down"]), cfg.k, logits32=lg[rows])
    assert rel_fro(to_np(out)[rows], ref["out"]) <= REL_FRO_MX


@pytest.mark.parametrize("T,E,k,H,I,fmt", [
    (64, 8, 2, 256, 128, 0),      # P <= 16E: narrow tiles, 32-row padding
    (64, 8, 2, 256, 128, 1),
    (300, 4, 2, 256, 256, 0),     # wide tiles, 128-row padding, experts over 128 rows
    (300, 4, 2, 512, 128, 1),
    (600, 4, 2, 256, 128, 0),     # a 256-row block and a short one per expert
])
def test_grouped_gemms_mx_match_oracle(cuda_dev, T, E, k, H, I, fmt):
    """Standalone block-scaled GEMMs on expert-sorted MX rows.  The activations are
    MX-quantised by the oracle from seeded fp32 data; expected values are the oracle's
    fp64 products of the dequantised operands (h then MX-quantised along I)."""
    rng = np.random.default_rng(T + E + fmt)
    ids = W.make_topk_ids(T, E, k, seed=T + 3)
    rt = O.init_routing(to_np(ids), E)
    P = T * k
    A = rng.standard_normal((P, H)).astype(np.float32)
    Aq, Asc = O.mx_quantize(A.astype(np.float64))
    Adq = O.mx_dequantize(Aq, Asc)
    g = torch.Generator().manual_seed(T + 11)
    w13 = (torch.randn(E, H, 2 * I, generator=g) * 0.05).to(torch.bfloat16)
    down = (torch.randn(E, I, H, generator=g) * 0.05).to(torch.bfloat16)
    pack = moe.pack_weights_mx4 if fmt else moe.pack_weights_mx
    rt_w = O.mx4_roundtrip if fmt else O.mx_roundtrip
    w13_q, w13_sf, down_q, down_sf = pack(w13.to(cuda_dev), down.to(cuda_dev))
    off = torch.from_numpy(rt["offsets"].astype(np.int32)).to(cuda_dev)
    Aq_d = torch.from_numpy(Aq).to(cuda_dev)
    Asc_d = torch.from_numpy(Asc).to(cuda_dev)
    h_q, h_sc = moe.grouped_matmul_swiglu_mx(Aq_d, Asc_d, w13_q, w13_sf, off, E, I, weight_format=fmt)
    # down projection on its own seeded MX rows (no GPU output feeds the oracle)
    A2 = rng.standard_normal((P, I)).astype(np.float32)
    A2q, A2sc = O.mx_quantize(A2.astype(np.float64))
    y = moe.grouped_matmul_mx(torch.from_numpy(A2q).to(cuda_dev), torch.from_numpy(A2sc).to(cuda_dev),
                              down_q, down_sf, off, E, H, weight_format=fmt)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    offs = rt["offsets"]
    h_ref = np.zeros((P, I))
    y_ref = np.zeros((P, H))
    A2dq = O.mx_dequantize(A2q, A2sc)
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        h_ref[lo:hi] = O.swiglu(Adq[lo:hi] @ rt_w(to_np(w13[e]).astype(np.float64), axis=0))
        y_ref[lo:hi] = A2dq[lo:hi] @ rt_w(to_np(down[e]).astype(np.float64), axis=0)
    # y: one bf16 rounding after fp32 accumulation of exactly representable products
    assert rel_fro(to_np(y).astype(np.float64), y_ref) <= 5e-3
    # h: the GPU quantises its fp32 h; codes and scales match the oracle's quantisation
    # of the fp64 h except where the two sit on opposite sides of a rounding boundary
    rq, rsc = O.mx_quantize(h_ref)
    got = O.mx_dequantize(to_np(h_q).astype(np.uint8), to_np(h_sc).astype(np.uint8))
    ref = O.mx_dequantize(rq, rsc)
    diff = got != ref
    assert diff.mean() < 2e-3, diff.mean()
    step = np.exp2(np.repeat(rsc.astype(np.float64), 32, axis=1) - 127) * 2.0 ** -2
    assert np.all(np.abs(got - ref)[diff] <= np.maximum(np.abs(ref[diff]) * 2.0 ** -3, step[diff]))
    assert (to_np(h_sc) != rsc).mean() < 2e-3
