"""Per-operator parity of the CUDA kernels against the CPU oracle (GPU, via the C ABI).

Integer results (top-k ids, routing permutation, counts, offsets, gathered rows)
must match bit for bit; floating-point results within tolerances stated per test.
"""
import numpy as np
import pytest
import torch

import top_routing_grouped_gating_gb300 as moe
from oracle import moe_oracle as O
from tests._helpers import LazyExperts, assert_close_layer, rel_fro, to_np
from top_routing_grouped_gating_gb300 import workloads as W

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ gating --

@pytest.mark.parametrize("T,E,k,ties", [
    (1, 8, 2, False), (33, 8, 2, True), (64, 128, 8, False), (257, 128, 8, True),
    (100, 256, 8, False), (17, 64, 1, True), (9, 1, 1, False), (40, 32, 32, True), (5, 200, 16, True),
])
def test_gating_matches_oracle(cuda_dev, T, E, k, ties):
    lg = W.make_logits(T, E, seed=T * 7 + E + k, ties=ties)
    ids, w = moe.gating_topk_softmax(lg.to(cuda_dev), k)
    r_ids, r_w = O.gating_topk_softmax(lg.numpy(), k)
    np.testing.assert_array_equal(to_np(ids), r_ids)
    # fp32 softmax over k values: a few roundings of 2^-24 each
    np.testing.assert_allclose(to_np(w), r_w, rtol=2e-6, atol=1e-7)


def test_gating_without_renormalisation(cuda_dev):
    lg = W.make_logits(50, 64, seed=3)
    ids, w = moe.gating_topk_softmax(lg.to(cuda_dev), 6, renormalize=False)
    r_ids, r_w = O.gating_topk_softmax(lg.numpy(), 6, renormalize=False)
    np.testing.assert_array_equal(to_np(ids), r_ids)
    np.testing.assert_allclose(to_np(w), r_w, rtol=5e-6, atol=1e-7)


# ------------------------------------------------------------------ router --

@pytest.mark.parametrize("name,T", [("tiny", 16), ("qwen3_30b_a3b_decode", 32), ("qwen3_30b_a3b_decode", 300),
                                    ("qwen3_235b_a22b_decode", 64), ("qwen3_30b_a3b_prefill_zipf", 4096),
                                    ("qwen3_235b_a22b_prefill", 1000), ("tiny", 200)])
def test_router_logits(cuda_dev, name, T):
    cfg = W.with_shape(W.CONFIGS[name], T=T)
    inp = W.make_inputs(cfg, weights=False)
    got = to_np(moe.router_logits(inp["x"].to(cuda_dev), inp["Wg"].to(cuda_dev)))
    x, Wg = to_np(inp["x"]).astype(np.float64), inp["Wg"].numpy().astype(np.float64)
    ref = O.router_logits(x, Wg)
    # fp32 FMA accumulation over H terms: |err| <= ~H * 2^-24 * sum|x*w| (bound used: 1e-5 * sum)
    scale = np.abs(x) @ np.abs(Wg)
    assert np.all(np.abs(got - ref) <= 1e-5 * scale + 1e-30)


# ----------------------------------------------------------------- routing --

@pytest.mark.parametrize("T,E,k,skew", [
    (1, 8, 8, None), (3, 8, 2, None), (32, 128, 8, None), (511, 128, 8, 1.2), (4096, 128, 8, 1.2),
    (8192, 128, 8, None), (700, 256, 4, None), (2000, 1, 1, None), (100, 16, 16, None),
])
def test_init_routing_bit_exact(cuda_dev, T, E, k, skew):
    ids = W.make_topk_ids(T, E, k, seed=T + 3 * E, skew=skew)
    H = 256
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
    got = moe.init_routing(ids.to(cuda_dev), E, x=x.to(cuda_dev))
    ref = O.init_routing(ids.numpy(), E)
    for key in ("expanded_row_idx", "sorted_row_idx", "counts"):
        np.testing.assert_array_equal(to_np(got[key]), ref[key], err_msg=key)
    np.testing.assert_array_equal(to_np(got["expert_offsets"]), ref["offsets"])
    xe_ref = x[torch.from_numpy(ref["sorted_row_idx"].astype(np.int64) // k)]
    assert torch.equal(got["expanded_x"].cpu().view(torch.int16), xe_ref.view(torch.int16))
    cnt, off = moe.compute_expert_tokens(ids.to(cuda_dev), E)
    np.testing.assert_array_equal(to_np(cnt), ref["counts"])
    np.testing.assert_array_equal(to_np(off), ref["offsets"])


def test_routing_flags_bad_ids(cuda_dev):
    ids = W.make_topk_ids(40, 16, 2, seed=1)
    ids[3, 1] = 16
    ids[7, 0] = -1
    moe.clear_device_status()
    got = moe.init_routing(ids.to(cuda_dev), 16)
    st = moe.get_device_status()
    moe.clear_device_status()
    assert st & moe.DEV_BAD_EXPERT_ID
    eri = to_np(got["expanded_row_idx"])
    assert eri[3 * 2 + 1] == -1 and eri[7 * 2 + 0] == -1
    valid = np.ones(80, bool)
    valid[[7, 14]] = False
    flat = ids.numpy().reshape(-1)
    assert to_np(got["expert_offsets"])[-1] == 78
    # the valid pairs are sorted stably among themselves
    order = np.argsort(np.where(valid, flat, 99), kind="stable")[:78]
    np.testing.assert_array_equal(to_np(got["sorted_row_idx"])[:78], order)


# ---------------------------------------------------------------- finalize --

@pytest.mark.parametrize("T,k,H", [(1, 1, 256), (16, 2, 256), (33, 8, 2048), (300, 8, 4096)])
def test_finalize_matches_oracle(cuda_dev, T, k, H):
    g = torch.Generator().manual_seed(T + k)
    y2 = torch.randn(T * k, H, generator=g).to(torch.bfloat16)
    w = torch.rand(T, k, generator=g)
    eri = torch.randperm(T * k, generator=g).to(torch.int32)
    got = moe.finalize_routing(y2.to(cuda_dev), w.to(cuda_dev), eri.to(cuda_dev))
    ref = O.finalize_routing(to_np(y2), w.numpy().astype(np.float64), eri.numpy(), k)
    # fp32 sum of k terms then one bf16 rounding
    np.testing.assert_allclose(to_np(got), ref, rtol=2 ** -8, atol=1e-6 * np.abs(ref).max())
    again = moe.finalize_routing(y2.to(cuda_dev), w.to(cuda_dev), eri.to(cuda_dev))
    assert torch.equal(got, again)  # deterministic


# ------------------------------------------------------------ grouped GEMMs --

def _gemm_case(cuda_dev, T, E, k, H, I, skew, seed):
    ids = W.make_topk_ids(T, E, k, seed=seed, skew=skew)
    rt = O.init_routing(ids.numpy(), E)
    P = T * k
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(P, H, generator=g).to(torch.bfloat16)
    w13 = (torch.randn(E, H, 2 * I, generator=g) * 0.05).to(torch.bfloat16)
    down = (torch.randn(E, I, H, generator=g) * 0.05).to(torch.bfloat16)
    w13p, downp = moe.pack_weights(w13.to(cuda_dev), down.to(cuda_dev))
    off = torch.from_numpy(rt["offsets"]).to(cuda_dev)
    return rt, A, w13, down, w13p, downp, off


@pytest.mark.parametrize("T,E,k,H,I,skew", [
    (16, 8, 2, 256, 128, None),        # tiny config shape
    (32, 128, 8, 2048, 768, None),     # decode: thin token tiles
    (1, 8, 8, 256, 128, None),         # 8 pairs, one per expert
    (600, 16, 4, 256, 192, 1.0),       # wide tiles, ragged, hot experts > 256 rows
    (300, 64, 8, 512, 64, 1.5),        # some empty experts, I = 64
    (600, 16, 4, 256, 128, 1.5),       # CTA pairs, one projection a launch, light and heavy experts
    (1024, 8, 2, 512, 256, None),      # CTA pairs without light experts (256-row token blocks)
])
def test_grouped_gemms_match_oracle(cuda_dev, T, E, k, H, I, skew):
    rt, A, w13, down, w13p, downp, off = _gemm_case(cuda_dev, T, E, k, H, I, skew, seed=T + E + I)
    h = moe.grouped_matmul_swiglu(A.to(cuda_dev), w13p, off, E, I)
    An = to_np(A).astype(np.float64)
    h_ref = np.zeros((T * k, I))
    offs = rt["offsets"]
    for e in range(E):
        lo, hi = offs[e], offs[e + 1]
        if hi > lo:
            _, h_ref[lo:hi] = O.expert_mlp(An[lo:hi], to_np(w13[e]), to_np(down[e]), return_h=True)
    assert_close_layer(to_np(h), h_ref, rel=5e-3, max_abs_frac=1e-2, what="h")
    # down projection on its own seeded bf16 input (no GPU output feeds the oracle)
    A2 = torch.randn(T * k, I, generator=torch.Generator().manual_seed(T + 1)).to(torch.bfloat16)
    y = moe.grouped_matmul(A2.to(cuda_dev), downp, off, E, H)
    hn = to_np(A2).astype(np.float64)
    y_ref = np.zeros((T * k, H))
    for e in range(E):
        lo, hi = offs[e], offs[e + 1]
        if hi > lo:
            y_ref[lo:hi] = hn[lo:hi] @ to_np(down[e]).astype(np.float64)
    assert_close_layer(to_np(y), y_ref, rel=5e-3, max_abs_frac=1e-2, what="y")


def test_grouped_gemm_is_deterministic(cuda_dev):
    rt, A, w13, down, w13p, downp, off = _gemm_case(cuda_dev, 200, 32, 4, 512, 128, 1.0, seed=5)
    A = A.to(cuda_dev)
    h1 = moe.grouped_matmul_swiglu(A, w13p, off, 32, 128)
    h2 = moe.grouped_matmul_swiglu(A, w13p, off, 32, 128)
    assert torch.equal(h1, h2)
    assert moe.get_device_status() == 0
