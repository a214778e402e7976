"""W4A8 layer (MXFP4 expert weights, MXFP8 activations) on the GPU against the CPU
oracle, through the C ABI.

The weight pre-quantisation is compared bit for bit: both sides quantise the same
bf16 weights, and the e2m1 codes, their nibble packing and the E8M0 scale atoms
must match exactly.  The layer output is held to the MXFP8 layer's relative
Frobenius bound against ``moe_forward_w4a8`` run on the same dequantised values.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import top_routing_grouped_gating_gb300 as moe
from oracle import moe_oracle as O
from tests._helpers import REL_FRO_MX, LazyExperts, expert_coverage, oracle_threads, rel_fro, to_np
from tests.test_gpu_mx import _unpack_w13
from top_routing_grouped_gating_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# e2m1 magnitudes and the midpoints between neighbours (ties go to the even code)
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_MIDS = (_E2M1[1:] + _E2M1[:-1]) / 2


def _unnibble(q):
    """Bytes holding two e2m1 codes (element 2j in the low nibble) -> one code per byte."""
    q = np.asarray(q, np.uint8)
    out = np.empty(q.shape[:-1] + (2 * q.shape[-1],), np.uint8)
    out[..., 0::2] = q & 15
    out[..., 1::2] = q >> 4
    return out


def _untile(q, E, rows, K):
    """Tile-major packed codes (tiles of 128 rows x 128 K-elements, 64 bytes a row)
    -> row-major (E, rows, K/2) bytes."""
    t = np.asarray(q, np.uint8).reshape(E, rows // 128, K // 128, 128, 64)
    return t.transpose(0, 1, 3, 2, 4).reshape(E, rows, K // 2)


def _tricky_weights(E, H, I, seed):
    """Seeded bf16 weights with MXFP4 edge cases along the reduction axis: an
    all-zero block, a block of exact e2m1 midpoints (round-half-even), a block
    whose maximum saturates (scaled 7.5 -> 6), and negative zeros."""
    g = torch.Generator().manual_seed(seed)
    w13 = torch.randn(E, H, 2 * I, generator=g) * 0.05
    down = torch.randn(E, I, H, generator=g) * 0.05
    rng = np.random.default_rng(seed)
    w13[0, :32, 3] = 0.0
    # block max 6 * 2^-5 -> X = -5; the rest are midpoints times 2^-5
    mids = rng.choice(_MIDS, size=31) * rng.choice([-1.0, 1.0], size=31)
    w13[0, 32:64, 7] = torch.from_numpy(np.concatenate([[6.0], mids]) * 2.0 ** -5).float()
    # block max 7.5 * 2^-6: X = floor(log2(0.117)) - 2 = -6, scaled 7.5 saturates to 6
    w13[1, 64:96, 9] = torch.from_numpy(np.concatenate([[7.5], rng.choice(_E2M1, 31)]) * 2.0 ** -6).float()
    down[0, :32, 5] = -0.0
    down[0, 32:64, 6] = torch.from_numpy(np.concatenate([[-6.0], mids]) * 2.0 ** -3).float()
    return w13.to(torch.bfloat16), down.to(torch.bfloat16)


def test_pack_weights_mx4_bit_exact(cuda_dev):
    E, H, I = 4, 512, 256          # several K steps and row blocks per expert
    w13, down = _tricky_weights(E, H, I, seed=11)
    w13_q, w13_sf, down_q, down_sf = moe.pack_weights_mx4(w13.to(cuda_dev), down.to(cuda_dev))
    assert w13_q.numel() == E * 2 * I * H // 2 and down_q.numel() == E * H * I // 2
    codes, scales = _unpack_w13(_unnibble(_untile(to_np(w13_q), E, 2 * I, H)).reshape(-1), to_np(w13_sf),
                                E, H, I)
    for e in range(E):
        rq, rsc = O.mx4_quantize(to_np(w13[e]).astype(np.float64).T)   # along H, per column
        np.testing.assert_array_equal(codes[e].T, rq)
        np.testing.assert_array_equal(scales[e].T, rsc)
    dq = _unnibble(_untile(to_np(down_q), E, H, I))
    dsf = to_np(down_sf).reshape(E, H // 128, I // 128, 512)
    n = np.arange(H)[:, None]
    b = np.arange(I // 32)[None, :]
    for e in range(E):
        rq, rsc = O.mx4_quantize(to_np(down[e]).astype(np.float64).T)  # along I, per output column
        np.testing.assert_array_equal(dq[e], rq)
        got_sc = dsf[e][n // 128, b // 4, (n % 32) * 16 + ((n % 128) // 32) * 4 + b % 4]
        np.testing.assert_array_equal(got_sc, rsc)


def _w4_layer(cfg, device="cuda"):
    inp = W.make_inputs(cfg, device=device)
    layer = moe.MoELayerW4A8(inp["Wg"], inp["w13"], inp["down"], inp["norm_w"], cfg.k, cfg.eps)
    return inp, layer


def _check_w4_forward(cfg, inp, layer, sample=None, threads=1):
    x, r = inp["x"], inp["r"]
    xn, rn, wn = to_np(x), to_np(r), to_np(inp["norm_w"])
    _, y = O.add_rmsnorm(xn, rn, wn, cfg.eps)
    lg32 = O.router_logits_f32(y, to_np(inp["Wg"]))
    out, res, ids, w = layer(x, r, logits_override=torch.from_numpy(lg32).to(x.device))
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    r_ids, _ = O.gating_topk_softmax(lg32, cfg.k)
    np.testing.assert_array_equal(to_np(ids), r_ids)
    rows = np.arange(cfg.T) if sample is None else sample
    with ThreadPoolExecutor(threads) as pool:
        ref = O.moe_forward_w4a8(xn[rows], rn[rows], wn, cfg.eps, None, LazyExperts(inp["w13"]),
                                 LazyExperts(inp["down"]), cfg.k, logits32=lg32[rows],
                                 expert_map=pool.map if threads > 1 else map)
    hit, active = expert_coverage(r_ids, rows, cfg.E)
    print(f"{cfg.name}: {len(rows)}/{cfg.T} tokens compared, {hit}/{active} active experts covered")
    got = to_np(out)[rows]
    assert np.all(np.isfinite(got))
    rf = rel_fro(got, ref["out"])
    assert rf <= REL_FRO_MX, f"relative Frobenius error {rf:.3e}"
    return rf


@pytest.mark.parametrize("T,E,k,H,I", [(64, 8, 2, 256, 128), (300, 4, 2, 256, 256), (1, 8, 8, 512, 128),
                                       (200, 16, 4, 512, 384),
                                       (64, 16, 2, 256, 128), (600, 4, 2, 256, 128)])
def test_forward_w4a8_small(cuda_dev, T, E, k, H, I):
    cfg = W.with_shape(W.CONFIGS["w4a8_prefill"], T=T, E=E, k=k, H=H, I=I)
    inp, layer = _w4_layer(cfg)
    _check_w4_forward(cfg, inp, layer)


def test_forward_w4a8_token_block_boundaries(cuda_dev):
    """MXFP4 weights through the CTA-pair kernel with expert loads on both sides of its
    256-row units and of the 32 absorbed rows, forced through designed logits."""
    from tests._helpers import forced_topk_logits
    counts = [256, 257, 288, 289, 31, 0, 545, 130]
    k = 2
    cfg = W.with_shape(W.CONFIGS["w4a8_prefill"], T=sum(counts) // k, E=len(counts), k=k, H=256, I=128)
    inp, layer = _w4_layer(cfg)
    lg = forced_topk_logits(counts, k, seed=13)
    x, r = inp["x"], inp["r"]
    out, res, ids, w = layer(x, r, logits_override=torch.from_numpy(lg).to(x.device))
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    r_ids, _ = O.gating_topk_softmax(lg, k)
    np.testing.assert_array_equal(np.bincount(r_ids.ravel(), minlength=cfg.E), counts)
    np.testing.assert_array_equal(to_np(ids), r_ids)
    ref = O.moe_forward_w4a8(to_np(x), to_np(r), to_np(inp["norm_w"]), cfg.eps, None,
                             LazyExperts(inp["w13"]), LazyExperts(inp["down"]), k, logits32=lg)
    got = to_np(out)
    assert np.all(np.isfinite(got))
    rf = rel_fro(got, ref["out"])
    assert rf <= REL_FRO_MX, f"relative Frobenius error {rf:.3e}"


def test_forward_w4a8_decode_tiles_skewed(cuda_dev):
    """Narrow-tile shape with a Zipf-skewed router: one expert spans several 32-token
    tiles, so all four 32-row groups of the activation scale atoms are used."""
    cfg = W.with_shape(W.CONFIGS["w4a8_decode"], T=256, E=16, k=1, H=256, I=128, router="zipf",
                       zipf_s=2.0)
    inp, layer = _w4_layer(cfg)
    assert cfg.T * cfg.k <= 16 * cfg.E
    _check_w4_forward(cfg, inp, layer)
    _, y = O.add_rmsnorm(to_np(inp["x"]), to_np(inp["r"]), to_np(inp["norm_w"]), cfg.eps)
    ids, _ = O.gating_topk_softmax(O.router_logits_f32(y, to_np(inp["Wg"])), cfg.k)
    assert np.bincount(ids.ravel(), minlength=cfg.E).max() > 128   # two atoms, all groups


def test_forward_w4a8_few_pairs_skewed(cuda_dev):
    """At most 8 pairs per expert on average with a Zipf-skewed router, so one expert
    spans several narrow token blocks while most have one or two tokens."""
    cfg = W.with_shape(W.CONFIGS["w4a8_decode"], T=128, E=16, k=1, H=256, I=128, router="zipf",
                       zipf_s=2.0)
    inp, layer = _w4_layer(cfg)
    assert cfg.T * cfg.k <= 8 * cfg.E
    _check_w4_forward(cfg, inp, layer)
    _, y = O.add_rmsnorm(to_np(inp["x"]), to_np(inp["r"]), to_np(inp["norm_w"]), cfg.eps)
    ids, _ = O.gating_topk_softmax(O.router_logits_f32(y, to_np(inp["Wg"])), cfg.k)
    assert np.bincount(ids.ravel(), minlength=cfg.E).max() > 48


def test_w4a8_differs_from_mxfp8(cuda_dev):
    """The 4-bit weights are really used: the W4A8 output is farther from the MXFP8
    oracle than from the W4A8 one (MXFP4 error ~ 2^-3 relative, MXFP8 ~ 2^-5)."""
    cfg = W.with_shape(W.CONFIGS["w4a8_prefill"], T=64, E=8, k=2, H=256, I=128)
    inp, layer = _w4_layer(cfg)
    xn, rn, wn = to_np(inp["x"]), to_np(inp["r"]), to_np(inp["norm_w"])
    lg32 = O.router_logits_f32(O.add_rmsnorm(xn, rn, wn, cfg.eps)[1], to_np(inp["Wg"]))
    out = to_np(layer(inp["x"], inp["r"], logits_override=torch.from_numpy(lg32).cuda())[0])
    args = (xn, rn, wn, cfg.eps, None, LazyExperts(inp["w13"]), LazyExperts(inp["down"]), cfg.k)
    e4 = rel_fro(out, O.moe_forward_w4a8(*args, logits32=lg32)["out"])
    e8 = rel_fro(out, O.moe_forward_mx(*args, logits32=lg32)["out"])
    assert e4 < 0.5 * e8


def test_forward_w4a8_full_size(cuda_dev):
    """The W4A8 prefill layer at full size against the oracle on every token."""
    cfg = W.CONFIGS["w4a8_prefill"]
    inp, layer = _w4_layer(cfg)
    _check_w4_forward(cfg, inp, layer, threads=oracle_threads())
    a = layer(inp["x"], inp["r"])[0].clone()
    b = layer(inp["x"], inp["r"])[0]
    assert torch.equal(a, b)


def test_forward_w4a8_decode_full_size(cuda_dev):
    cfg = W.CONFIGS["w4a8_decode"]
    inp, layer = _w4_layer(cfg)
    _check_w4_forward(cfg, inp, layer, threads=oracle_threads())


def test_w4a8_rejects_unaligned_codes(cuda_dev):
    cfg = W.with_shape(W.CONFIGS["w4a8_prefill"], T=8, E=4, k=2, H=256, I=128)
    inp, layer = _w4_layer(cfg)
    buf = torch.empty(layer.w13_q.numel() + 16, dtype=torch.uint8, device=layer.w13_q.device)
    layer.w13_q = buf[16:]                   # 16-byte but not 32-byte aligned
    with pytest.raises(moe.MoEError):
        layer(inp["x"], inp["r"])
