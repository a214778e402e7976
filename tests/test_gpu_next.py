"""GPU parity of the rows after the core path: fused add+RMSNorm+cast, expert-range
routing (init_routing_v2), re-routing, finalize with zero-computation experts, and
the layer with pre-norm and/or zero-computation experts (moe_forward_v2)."""
import numpy as np
import pytest
import torch

import top_routing_grouped_gating_gb300 as moe
from oracle import moe_oracle as O
from tests._helpers import LazyExperts, assert_close_layer, routing_margin_ok, to_np
from top_routing_grouped_gating_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_add_rmsnorm_cast(cuda_dev):
    cfg = W.with_shape(W.CONFIGS["qwen3_30b_a3b_decode_prenorm"], T=48, E=8, I=128)
    inp = W.make_inputs(cfg)
    x, r, w = inp["x"], inp["r"], inp["norm_w"]
    res, y32, ybf = moe.add_rmsnorm_cast(x.to(cuda_dev), r.to(cuda_dev), w.to(cuda_dev), cfg.eps)
    s, y, yb = O.add_rmsnorm_cast(to_np(x), to_np(r), to_np(w), cfg.eps)
    assert torch.equal(res.cpu().view(torch.int16), torch.from_numpy(s).to(torch.bfloat16).view(torch.int16))
    np.testing.assert_allclose(to_np(y32), y, rtol=2e-5, atol=1e-6)
    got = to_np(ybf).astype(np.float64)
    # bf16 of the fp32 value: equal except where the two fp32 values straddle a bf16
    # rounding boundary, then one bf16 ulp apart
    diff = got != yb
    assert diff.mean() < 1e-3
    assert np.all(np.abs(got - yb)[diff] <= np.abs(yb[diff]) * 2.0 ** -7)
    _, y0, _ = moe.add_rmsnorm_cast(x.to(cuda_dev), None, w.to(cuda_dev), cfg.eps)
    np.testing.assert_allclose(to_np(y0), O.add_rmsnorm(to_np(x), None, to_np(w), cfg.eps)[1], rtol=2e-5,
                               atol=1e-6)


@pytest.mark.parametrize("T,E_total,k,begin,end", [(300, 64, 8, 16, 40), (40, 128, 8, 0, 128),
                                                   (1000, 192, 8, 0, 128), (3, 16, 2, 15, 16),
                                                   (2500, 256, 4, 128, 256)])
def test_init_routing_v2_bit_exact(cuda_dev, T, E_total, k, begin, end):
    ids = W.make_topk_ids(T, E_total, k, seed=T + begin)
    x = torch.randn(T, 128, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    moe.clear_device_status()
    got = moe.init_routing_v2(ids.to(cuda_dev), E_total, begin, end, x=x.to(cuda_dev))
    assert moe.get_device_status() == 0          # skipped ids are not errors
    ref = O.init_routing_v2(ids.numpy(), E_total, begin, end)
    n = int(ref["offsets"][-1])
    np.testing.assert_array_equal(to_np(got["expanded_row_idx"]), ref["expanded_row_idx"])
    np.testing.assert_array_equal(to_np(got["counts"]), ref["counts"])
    np.testing.assert_array_equal(to_np(got["expert_offsets"]), ref["offsets"])
    np.testing.assert_array_equal(to_np(got["sorted_row_idx"])[:n], ref["sorted_row_idx"][:n])
    xe = got["expanded_x"][:n].cpu()
    assert torch.equal(xe.view(torch.int16), x[torch.from_numpy(ref["sorted_row_idx"][:n] // k).long()].view(
        torch.int16))


def test_init_routing_v2_flags_only_invalid_ids(cuda_dev):
    ids = W.make_topk_ids(20, 32, 2, seed=2)
    ids[4, 0] = 40
    moe.clear_device_status()
    moe.init_routing_v2(ids.to(cuda_dev), 32, 0, 16)
    st = moe.get_device_status()
    moe.clear_device_status()
    assert st & moe.DEV_BAD_EXPERT_ID


@pytest.mark.parametrize("R,El,H", [(4, 8, 256), (2, 32, 64), (8, 1, 128)])
def test_re_routing_bit_exact(cuda_dev, R, El, H):
    g = torch.Generator().manual_seed(R * El)
    cnt = torch.randint(0, 9, (R, El), generator=g, dtype=torch.int32)
    cnt[0, 0] = 0
    N = int(cnt.sum())
    xr = torch.randn(N, H, generator=g).to(torch.bfloat16)
    xo, perm, off = moe.re_routing(cnt.to(cuda_dev), xr.to(cuda_dev), N)
    rperm, roff = O.re_routing(cnt.numpy())
    np.testing.assert_array_equal(to_np(perm), rperm)
    np.testing.assert_array_equal(to_np(off), roff)
    ref = torch.empty_like(xr)
    ref[torch.from_numpy(rperm).long()] = xr
    assert torch.equal(xo.cpu().view(torch.int16), ref.view(torch.int16))


def _v2_layer(name, **kw):
    cfg = W.with_shape(W.CONFIGS[name], **kw) if kw else W.CONFIGS[name]
    inp = W.make_inputs(cfg, device="cuda")
    layer = moe.MoELayerV2(inp["Wg"], inp["w13"], inp["down"], cfg.k, Z=cfg.Z,
                           norm_w=inp.get("norm_w") if cfg.prenorm else None, eps=cfg.eps)
    return cfg, inp, layer


def _oracle_v2(cfg, inp, lg32, rows):
    xn = to_np(inp["x"])
    rn = to_np(inp["r"])[rows] if cfg.prenorm else None
    nw = to_np(inp["norm_w"]) if cfg.prenorm else None
    return O.moe_forward_v2(xn[rows], rn, nw, cfg.eps, None, LazyExperts(inp["w13"]), LazyExperts(inp["down"]),
                            cfg.k, num_zero_experts=cfg.Z, logits32=lg32[rows])


def _router_input(cfg, inp):
    if cfg.prenorm:
        return O.add_rmsnorm(to_np(inp["x"]), to_np(inp["r"]), to_np(inp["norm_w"]), cfg.eps)[1]
    return to_np(inp["x"]).astype(np.float64)


@pytest.mark.parametrize("name,kw", [("qwen3_30b_a3b_decode_prenorm", {}), ("zero_experts_decode", {}),
                                     ("zero_experts_decode", dict(T=700)),
                                     ("qwen3_30b_a3b_decode_prenorm", dict(T=300, Z=16))])
def test_forward_v2_matches_oracle(cuda_dev, name, kw):
    cfg, inp, layer = _v2_layer(name, **kw)
    lg32 = O.router_logits_f32(_router_input(cfg, inp), to_np(inp["Wg"]))
    out, res, ids, w = layer(inp["x"], inp.get("r") if cfg.prenorm else None,
                             logits_override=torch.from_numpy(lg32).to(cuda_dev))
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    r_ids, r_w = O.gating_topk_softmax(lg32, cfg.k)
    np.testing.assert_array_equal(to_np(ids), r_ids)
    if cfg.Z:
        assert (r_ids >= cfg.E).any()            # some pairs land on identity experts
    rows = np.arange(cfg.T) if cfg.T <= 64 else np.unique(np.r_[0, np.arange(5, cfg.T, cfg.T // 40), cfg.T - 1])
    ref = _oracle_v2(cfg, inp, lg32, rows)
    assert_close_layer(to_np(out)[rows], ref["out"], what=name)


@pytest.mark.parametrize("T", [32, 300])
def test_forward_v2_prenorm_gpu_router(cuda_dev, T):
    cfg, inp, layer = _v2_layer("qwen3_30b_a3b_decode_prenorm", T=T, Z=8)
    out, res, ids, w = layer(inp["x"], inp["r"])
    torch.cuda.synchronize()
    y = _router_input(cfg, inp)
    Wn = to_np(inp["Wg"]).astype(np.float64)
    lg = O.router_logits_f32(y, Wn)
    tol = 1e-5 * (np.abs(y) @ np.abs(Wn)).max(axis=1)
    safe = routing_margin_ok(lg, cfg.k, tol)
    assert safe.sum() >= 0.9 * cfg.T
    r_ids, _ = O.gating_topk_softmax(lg, cfg.k)
    np.testing.assert_array_equal(to_np(ids)[safe], r_ids[safe])
    rows = np.nonzero(safe)[0][:32]
    ref = _oracle_v2(cfg, inp, lg, rows)
    assert_close_layer(to_np(out)[rows], ref["out"])
    _, y2_ref = O.add_rmsnorm(to_np(inp["x"]), to_np(inp["r"]), to_np(inp["norm_w"]), cfg.eps)
    s = to_np(inp["x"]).astype(np.float64) + to_np(inp["r"])
    assert torch.equal(res.cpu().view(torch.int16), torch.from_numpy(s).to(torch.bfloat16).view(torch.int16))
