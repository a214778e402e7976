"""Pins for the CPU oracle (no GPU).

Each check ties the oracle to something other than itself: hand-derived fixtures
in tests/golden/, closed forms, library routines on special cases (scipy softmax,
numpy stable argsort, torch fp64 SiLU / rms_norm, torch float8_e4m3fn), brute
force on tiny inputs, and invariants.  The ``test_mutation_*`` tests plant a
plausible mistake in a copy of an oracle function and check that a pin catches it.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe_oracle as O
from top_routing_grouped_gating_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def f32(t):
    return t.float().numpy()


def tiny_layer(T=12, H=32, E=6, k=2, I=16, seed=3, scale=0.3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    Wg = rng.standard_normal((H, E)) * scale
    w13 = [rng.standard_normal((H, 2 * I)) * scale for _ in range(E)]
    down = [rng.standard_normal((I, H)) * scale for _ in range(E)]
    return x, Wg, w13, down, k


# ------------------------------------------------------------------ router --


def test_router_logits_exact_on_integers():
    rng = np.random.default_rng(0)
    x = rng.integers(-4, 5, size=(5, 7)).astype(np.float64)
    Wg = rng.integers(-3, 4, size=(7, 4)).astype(np.float64)
    lg = O.router_logits(x, Wg)
    for t in range(5):
        for e in range(4):
            assert lg[t, e] == sum(int(x[t, h]) * int(Wg[h, e]) for h in range(7))


def test_router_logits_f32_is_one_rounding_of_exact_sum():
    cfg = W.with_shape(W.CONFIGS["tiny"], T=4, H=64, E=8)
    inp = W.make_inputs(cfg, weights=False)
    x, Wg = f32(inp["x"]), inp["Wg"].numpy()
    got = O.router_logits_f32(x, Wg)
    for t in range(4):
        for e in range(8):
            exact = sum(Fraction(float(x[t, h])) * Fraction(float(Wg[h, e])) for h in range(64))
            assert got[t, e] == np.float32(float(exact))


# ------------------------------------------------------------------ gating --


def test_gating_golden(golden):
    for c in golden("gating.json")["cases"]:
        lg = np.array([c["logits"]], np.float32)
        ids, w = O.gating_topk_softmax(lg, c["k"])
        assert ids[0].tolist() == c["ids"], c["derivation"]
        np.testing.assert_allclose(w[0], c["weights"], rtol=1e-6, err_msg=c["derivation"])


def test_gating_weights_sum_to_one():
    lg = W.make_logits(64, 128, seed=1).numpy()
    _, w = O.gating_topk_softmax(lg, 8)
    assert np.all(np.abs(w.sum(1) - 1.0) < 1e-12)
    assert np.all(w > 0)
    assert np.all(np.diff(w, axis=1) <= 0)   # slots in descending weight


def test_gating_k_equals_E_is_full_softmax():
    lg = W.make_logits(16, 8, seed=2).numpy()
    ids, w = O.gating_topk_softmax(lg, 8)
    ref_ids = np.argsort(-lg.astype(np.float64), axis=1, kind="stable")
    np.testing.assert_array_equal(ids, ref_ids)
    p = scipy.special.softmax(lg.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(p, ref_ids, 1), rtol=1e-13)


def test_gating_equals_softmax_topk_renormalise():
    # the spec reading (softmax over all E, top-k, renormalise) vs the
    # oracle's (top-k, softmax over the chosen k): equal up to rounding.
    lg = W.make_logits(32, 64, seed=5).numpy()
    ids, w = O.gating_topk_softmax(lg, 6)
    p = scipy.special.softmax(lg.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, ids.astype(np.int64), 1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-12)
    _, w_nr = O.gating_topk_softmax(lg, 6, renormalize=False)
    np.testing.assert_allclose(w_nr, sel, rtol=1e-12)


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (7, 4), (7, 7)])
def test_gating_brute_force_with_ties(E, k):
    lg = W.make_logits(40, E, seed=E * 10 + k, ties=True).numpy()
    ids, _ = O.gating_topk_softmax(lg, k)
    for t in range(lg.shape[0]):
        assert ids[t].tolist() == O.brute_force_topk(lg[t], k).tolist()


# ----------------------------------------------------------------- routing --


def test_routing_golden(golden):
    for c in golden("routing.json")["cases"]:
        rt = O.init_routing(np.array(c["topk_ids"], np.int32), c["E"])
        for key in ("counts", "offsets", "expanded_row_idx", "sorted_row_idx"):
            assert rt[key].tolist() == c[key], (key, c["derivation"])


@pytest.mark.parametrize("T,E,k,skew", [(37, 8, 2, None), (300, 64, 8, None), (257, 128, 8, 1.2),
                                        (5, 1, 1, None), (1, 16, 16, None)])
def test_routing_is_stable_sort(T, E, k, skew):
    ids = W.make_topk_ids(T, E, k, seed=T + E, skew=skew).numpy()
    rt = O.init_routing(ids, E)
    flat = ids.reshape(-1)
    np.testing.assert_array_equal(rt["counts"], np.bincount(flat, minlength=E))
    assert rt["offsets"][-1] == T * k and rt["counts"].sum() == T * k
    np.testing.assert_array_equal(rt["sorted_row_idx"], np.argsort(flat, kind="stable"))
    eri, sri = rt["expanded_row_idx"], rt["sorted_row_idx"]
    assert sorted(eri.tolist()) == list(range(T * k))
    np.testing.assert_array_equal(sri[eri], np.arange(T * k))
    for e in range(E):
        rows = sri[rt["offsets"][e]:rt["offsets"][e + 1]]
        assert np.all(flat[rows] == e)
        assert np.all(np.diff(rows // k) > 0)    # token-ascending within an expert


# --------------------------------------------------------------------- MLP --


def test_mlp_golden(golden):
    for c in golden("mlp.json")["cases"]:
        y, h = O.expert_mlp(np.array(c["x"]), np.array(c["w13"]), np.array(c["down"]), return_h=True)
        np.testing.assert_allclose(h, c["h"], rtol=1e-12, atol=1e-15, err_msg=c["derivation"])
        np.testing.assert_allclose(y, c["y"], rtol=1e-12, atol=1e-15, err_msg=c["derivation"])


def test_sigmoid_extremes():
    z = np.array([-800.0, -30.0, 0.0, 30.0, 800.0])
    s = O.sigmoid(z)
    np.testing.assert_allclose(s, scipy.special.expit(z), rtol=1e-14, atol=0)


def test_single_expert_is_dense_swiglu_mlp():
    x, Wg, w13, down, _ = tiny_layer(T=9, E=1)
    res = O.moe_forward(x, Wg[:, :1], w13, down, k=1)
    xt = torch.tensor(x, dtype=torch.float64)
    g, u = torch.chunk(xt @ torch.tensor(w13[0]), 2, dim=-1)
    ref = (torch.nn.functional.silu(g) * u) @ torch.tensor(down[0])
    np.testing.assert_allclose(res["out"], ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["topk_w"], 1.0)


def test_layer_matches_dense_every_expert_then_mask():
    x, Wg, w13, down, k = tiny_layer()
    res = O.moe_forward(x, Wg, w13, down, k)
    ref = O.dense_moe_reference(x, w13, down, res["topk_ids"], res["topk_w"])
    np.testing.assert_allclose(res["out"], ref, rtol=1e-11, atol=1e-12)


def test_layer_linear_in_down_and_token_equivariant():
    x, Wg, w13, down, k = tiny_layer(T=10, seed=8)
    base = O.moe_forward(x, Wg, w13, down, k)["out"]
    scaled = O.moe_forward(x, Wg, w13, [2.5 * d for d in down], k)["out"]
    np.testing.assert_allclose(scaled, 2.5 * base, rtol=1e-12, atol=1e-12)
    perm = np.random.default_rng(1).permutation(10)
    permuted = O.moe_forward(x[perm], Wg, w13, down, k)["out"]
    np.testing.assert_allclose(permuted, base[perm], rtol=1e-12, atol=1e-12)


def test_layer_expert_relabelling_invariant():
    x, Wg, w13, down, k = tiny_layer(T=10, seed=9)
    base = O.moe_forward(x, Wg, w13, down, k)["out"]
    perm = np.random.default_rng(2).permutation(len(w13))
    out = O.moe_forward(x, Wg[:, perm], [w13[p] for p in perm], [down[p] for p in perm], k)["out"]
    np.testing.assert_allclose(out, base, rtol=1e-12, atol=1e-12)


def test_finalize_matches_layer():
    x, Wg, w13, down, k = tiny_layer(T=7, seed=4)
    res = O.moe_forward(x, Wg, w13, down, k)
    out = O.finalize_routing(res["y2"], res["topk_w"], res["expanded_row_idx"], k)
    np.testing.assert_allclose(out, res["out"], rtol=1e-13, atol=1e-14)


def test_layer_with_logits_override_uses_given_routing():
    x, Wg, w13, down, k = tiny_layer(T=6, seed=6)
    lg = W.make_logits(6, len(w13), seed=11).numpy()
    res = O.moe_forward(x, Wg, w13, down, k, logits32=lg)
    ids, w = O.gating_topk_softmax(lg, k)
    np.testing.assert_array_equal(res["topk_ids"], ids)
    ref = O.dense_moe_reference(x, w13, down, ids, w)
    np.testing.assert_allclose(res["out"], ref, rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------ RMSNorm / MX --


def test_add_rmsnorm_matches_torch():
    rng = np.random.default_rng(0)
    x, r = rng.standard_normal((5, 64)), rng.standard_normal((5, 64))
    w = 1 + 0.1 * rng.standard_normal(64)
    s, y = O.add_rmsnorm(x, r, w, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.tensor(x + r), (64,), torch.tensor(w), eps=1e-6)
    np.testing.assert_allclose(s, x + r, rtol=0, atol=0)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-13)
    _, y0 = O.add_rmsnorm(x, None, w, 1e-6)
    ref0 = torch.nn.functional.rms_norm(torch.tensor(x), (64,), torch.tensor(w), eps=1e-6)
    np.testing.assert_allclose(y0, ref0.numpy(), rtol=1e-13)


def test_e4m3_golden(golden):
    for c in golden("e4m3.json")["cases"]:
        assert int(O.e4m3_encode(np.array([c["value"]]))[0]) == c["code"], c["derivation"]


def test_e4m3_table_matches_torch_and_roundtrips():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = O.e4m3_decode(codes)
    finite = ~np.isnan(ref)
    assert np.isnan(mine[~finite]).all()
    np.testing.assert_array_equal(mine[finite], ref[finite])
    fin_codes = codes[finite]
    np.testing.assert_array_equal(O.e4m3_encode(O.e4m3_decode(fin_codes)), fin_codes)


def test_e4m3_rounding_matches_torch_in_range():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 1e-2,
                        rng.standard_normal(20000) * 3e-3])
    v32 = v.astype(np.float32)
    ref = torch.tensor(v32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_encode(v32.astype(np.float64)), ref)


def test_mx_block_golden(golden):
    for c in golden("mx_block.json")["cases"]:
        blk = np.full((1, 32), c["fill"])
        blk[0, 5] = c["block_amax_value"]
        q, s = O.mx_quantize(blk)
        assert int(s[0, 0]) == c["scale_byte"], c["derivation"]
        assert int(q[0, 5]) == c["amax_code"], c["derivation"]


def test_mx_scale_invariants_and_error_bound():
    rng = np.random.default_rng(3)
    y = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-20, 20, size=(64, 1)))
    q, s = O.mx_quantize(y)
    X = s.astype(np.int64) - 127
    amax = np.abs(y.reshape(64, 8, 32)).max(-1)
    ratio = amax / np.exp2(X)
    assert np.all((ratio >= 256) & (ratio < 512))
    deq = O.mx_dequantize(q, s).reshape(64, 8, 32)
    yb = y.reshape(64, 8, 32)
    scale = np.exp2(X)[..., None]
    sat = np.abs(yb) > 448 * scale
    # non-saturated elements: within half an e4m3 ulp (<= 2^-4 relative for normals,
    # 2^-10 * scale absolute for subnormals)
    err = np.abs(deq - yb)
    bound = np.maximum(np.abs(yb) * 2.0 ** -4, 2.0 ** -10 * scale)
    assert np.all(err[~sat] <= bound[~sat] * (1 + 1e-12))
    np.testing.assert_array_equal(np.abs(deq[sat]), 448 * np.broadcast_to(scale, sat.shape)[sat])


def test_mx_powers_of_two_exact_and_zero_block():
    y = np.exp2(np.arange(-8, 24).astype(np.float64))[None, :] * np.array([[1.0], [-1.0]])
    y = np.concatenate([y, np.zeros((1, 32))])
    deq = O.mx_dequantize(*O.mx_quantize(y))
    # powers of two within 2^-9..2^8 of the block max survive exactly
    blkmax = 2.0 ** 23
    keep = np.abs(y) >= blkmax * 2.0 ** -17
    np.testing.assert_array_equal(deq[keep], y[keep])
    assert np.all(deq[2] == 0)


def test_mx_roundtrip_axis():
    rng = np.random.default_rng(5)
    w = rng.standard_normal((64, 10))
    a0 = O.mx_roundtrip(w, axis=0)
    a1 = O.mx_roundtrip(w.T, axis=-1).T
    np.testing.assert_array_equal(a0, a1)


def test_mx_layer_matches_dense_composition():
    rng = np.random.default_rng(12)
    T, H, E, k, I = 6, 64, 4, 2, 32
    x, r = rng.standard_normal((T, H)), rng.standard_normal((T, H))
    nw = 1 + 0.1 * rng.standard_normal(H)
    Wg = rng.standard_normal((H, E)) * 0.3
    w13 = [rng.standard_normal((H, 2 * I)) * 0.2 for _ in range(E)]
    down = [rng.standard_normal((I, H)) * 0.2 for _ in range(E)]
    res = O.moe_forward_mx(x, r, nw, 1e-6, Wg, w13, down, k)
    s, y = O.add_rmsnorm(x, r, nw, 1e-6)
    ids, w = O.gating_topk_softmax(O.router_logits_f32(y, Wg), k)
    ref = np.zeros((T, H))
    for t in range(T):
        a = O.mx_roundtrip(y[t:t + 1])
        for sl in range(k):
            e = ids[t, sl]
            h = O.swiglu(a @ O.mx_roundtrip(w13[e], axis=0))
            ref[t] += w[t, sl] * (O.mx_roundtrip(h) @ O.mx_roundtrip(down[e], axis=0))[0]
    np.testing.assert_allclose(res["out"], ref, rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------- seeded inputs --


def test_workloads_shapes_and_zipf_skew():
    cfg = W.CONFIGS["qwen3_30b_a3b_prefill_zipf"]
    inp = W.make_inputs(cfg, weights=False)
    assert inp["x"].shape == (4096, 2048) and inp["x"].dtype == torch.bfloat16
    assert torch.all(inp["x"][:, 0] == 1.0)
    lg = O.router_logits_f32(f32(inp["x"]), inp["Wg"].numpy())
    ids, _ = O.gating_topk_softmax(lg[:1024], 8)
    counts = np.bincount(ids.reshape(-1), minlength=128)
    mean = counts.sum() / 128
    assert counts.max() >= 10 * mean     # hot experts
    assert (counts == 0).sum() >= 5      # cold experts


# --------------------------------------------------------------- mutations --


def test_mutation_swapped_gate_up_is_caught(golden):
    def bad_swiglu(gu):
        n = gu.shape[-1] // 2
        g, u = gu[..., n:], gu[..., :n]
        return g * O.sigmoid(g) * u
    c = golden("mlp.json")["cases"][0]
    h = bad_swiglu(np.array(c["x"]) @ np.array(c["w13"]))
    assert not np.allclose(h, c["h"])


def test_mutation_unstable_or_wrong_tiebreak_is_caught(golden):
    c = golden("gating.json")["cases"][4]
    lg = np.array(c["logits"], np.float64)
    wrong = np.lexsort((-np.arange(len(lg)), -lg))[: c["k"]]   # ties to the HIGHER id
    assert wrong.tolist() != c["ids"]
    r = golden("routing.json")["cases"][0]
    flat = np.array(r["topk_ids"]).reshape(-1)
    unstable = np.argsort(flat, kind="quicksort")[::-1]
    assert unstable.tolist() != r["sorted_row_idx"]


def test_mutation_mx_off_by_one_exponent_is_caught(golden):
    c = golden("mx_block.json")["cases"][0]
    amax = np.array([c["block_amax_value"]])
    _, ex = np.frexp(amax)
    wrong = int(ex[0]) - 8 + 127       # forgets the -1 of frexp
    assert wrong != c["scale_byte"]


# ------------------------------------------------------------ next rows --


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.integers(-20, 20, 50000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875]]).astype(np.float32)
    ref = torch.tensor(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.bf16_round(v), ref)


def test_add_rmsnorm_cast_outputs():
    rng = np.random.default_rng(1)
    x, r = rng.standard_normal((4, 64)), rng.standard_normal((4, 64))
    w = 1 + 0.1 * rng.standard_normal(64)
    s, y, yb = O.add_rmsnorm_cast(x, r, w, 1e-6)
    _, y2 = O.add_rmsnorm(x, r, w, 1e-6)
    np.testing.assert_array_equal(y, y2)
    ref = torch.tensor(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(yb, ref)


def test_init_routing_v2_full_range_is_init_routing():
    ids = W.make_topk_ids(50, 16, 4, seed=3).numpy()
    a = O.init_routing(ids, 16)
    b = O.init_routing_v2(ids, 16, 0, 16)
    for key in ("counts", "offsets", "expanded_row_idx", "sorted_row_idx"):
        np.testing.assert_array_equal(a[key], b[key])


def test_init_routing_v2_expert_range():
    ids = W.make_topk_ids(80, 32, 4, seed=9).numpy()
    b = O.init_routing_v2(ids, 32, 8, 16)
    flat = ids.reshape(-1)
    keep = (flat >= 8) & (flat < 16)
    np.testing.assert_array_equal(b["counts"], np.bincount(flat[keep] - 8, minlength=8))
    order = np.nonzero(keep)[0][np.argsort(flat[keep], kind="stable")]
    n = int(keep.sum())
    np.testing.assert_array_equal(b["sorted_row_idx"][:n], order)
    assert np.all(b["expanded_row_idx"][~keep] == -1)
    np.testing.assert_array_equal(b["expanded_row_idx"][order], np.arange(n))


def test_re_routing_is_stable_sort_by_expert():
    rng = np.random.default_rng(2)
    cnt = rng.integers(0, 5, size=(4, 6))
    perm, offs = O.re_routing(cnt)
    labels = np.concatenate([np.full(cnt[r, e], e) for r in range(4) for e in range(6)])
    order = np.argsort(labels, kind="stable")          # output row -> received row
    np.testing.assert_array_equal(perm[order], np.arange(len(labels)))
    np.testing.assert_array_equal(offs, np.concatenate([[0], np.cumsum(cnt.sum(0))]))


def test_zero_experts_only_gives_identity_and_none_gives_v1():
    x, Wg, w13, down, k = tiny_layer(T=7, E=4, k=2)
    Z = 3
    Wz = np.concatenate([Wg, np.full((Wg.shape[0], Z), 0.0)], axis=1)
    lg = np.full((7, 4 + Z), -50.0, np.float32)
    lg[:, 4:] = [[1.0, 2.0, 0.5]] * 7                  # top-2 are zero-computation experts
    res = O.moe_forward_v2(x, None, None, 0.0, Wz, w13, down, k, num_zero_experts=Z, logits32=lg)
    np.testing.assert_allclose(res["out"], x, rtol=1e-12, atol=1e-12)   # weights sum to 1
    base = O.moe_forward(x, Wg, w13, down, k)["out"]
    v2 = O.moe_forward_v2(x, None, None, 0.0, Wg, w13, down, k)["out"]
    np.testing.assert_allclose(v2, base, rtol=1e-13, atol=1e-13)


def test_prenorm_layer_is_norm_then_layer():
    x, Wg, w13, down, k = tiny_layer(T=6, seed=11)
    rng = np.random.default_rng(0)
    r = rng.standard_normal(x.shape)
    nw = 1 + 0.1 * rng.standard_normal(x.shape[1])
    res = O.moe_forward_v2(x, r, nw, 1e-6, Wg, w13, down, k)
    _, y, yb = O.add_rmsnorm_cast(x, r, nw, 1e-6)
    lg = O.router_logits_f32(y, Wg)
    ids, w = O.gating_topk_softmax(lg, k)
    ref = O.dense_moe_reference(yb, w13, down, ids, w)
    np.testing.assert_allclose(res["out"], ref, rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------------- W4A8 --


def test_e2m1_golden(golden):
    for c in golden("e2m1.json")["cases"]:
        assert int(O.e2m1_encode(np.array([c["value"]]))[0]) == c["code"], c["derivation"]


def test_e2m1_roundtrip_and_nearest():
    codes = np.arange(16)
    vals = O.e2m1_decode(codes)
    np.testing.assert_array_equal(O.e2m1_encode(vals)[vals != 0], codes[vals != 0])
    rng = np.random.default_rng(0)
    v = rng.uniform(-6, 6, 20000)
    d = O.e2m1_decode(O.e2m1_encode(v))
    grid = np.unique(np.abs(vals))
    best = np.min(np.abs(np.abs(v)[:, None] - grid[None, :]), axis=1)
    np.testing.assert_allclose(np.abs(np.abs(v) - np.abs(d)), best, atol=1e-15)
    assert np.all(np.sign(d[d != 0]) == np.sign(v[d != 0]))


def test_mx4_scale_rule_and_error_bound():
    rng = np.random.default_rng(1)
    y = rng.standard_normal((32, 128)) * np.exp2(rng.integers(-10, 10, size=(32, 1)))
    q, s = O.mx4_quantize(y)
    X = s.astype(np.int64) - 127
    amax = np.abs(y.reshape(32, 4, 32)).max(-1)
    r = amax / np.exp2(X)
    assert np.all((r >= 4) & (r < 8))
    deq = O.mx4_roundtrip(y)
    scale = np.repeat(np.exp2(X), 32, axis=1)
    sat = np.abs(y) > 6 * scale
    err = np.abs(deq - y)
    assert np.all(err[~sat] <= np.maximum(np.abs(y[~sat]) * 0.25, 0.25 * scale[~sat]) + 1e-12)
    np.testing.assert_allclose(np.abs(deq[sat]), 6 * scale[sat])


def _mx4_block_brute_force(col):
    """One 32-element block quantised to MXFP4 element by element: the shared
    exponent from frexp of the block's largest magnitude minus the e2m1 emax (2),
    then each element the nearest e2m1 magnitude (saturating at 6), sign kept."""
    import math
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    amax = max(abs(float(v)) for v in col)
    if amax == 0.0:
        return [0.0] * len(col)
    X = math.frexp(amax)[1] - 1 - 2
    out = []
    for v in col:
        a = min(abs(float(v)) / 2.0 ** X, 6.0)
        q = min(grid, key=lambda g: abs(a - g))
        out.append(math.copysign(q * 2.0 ** X, float(v)))
    return out


def test_mx4_roundtrip_axis():
    """mx4_roundtrip along axis 0 of a non-square matrix (the weight layout: blocks
    run down the reduction axis) equals an element-by-element brute force on each
    column's 32-row blocks; the other axis (5 columns) has no 32-blocks and raises,
    and on a 64 x 96 matrix the two axes give different results."""
    rng = np.random.default_rng(21)
    w = rng.standard_normal((64, 5)) * np.exp2(rng.integers(-6, 6, size=(1, 5)))
    got = O.mx4_roundtrip(w, axis=0)
    ref = np.array([[v for b in range(2) for v in _mx4_block_brute_force(w[32 * b:32 * (b + 1), c])]
                    for c in range(5)]).T
    np.testing.assert_array_equal(got, ref)
    with pytest.raises(ValueError):
        O.mx4_roundtrip(w, axis=-1)
    w2 = rng.standard_normal((64, 96))
    assert not np.array_equal(O.mx4_roundtrip(w2, axis=0), O.mx4_roundtrip(w2, axis=1))


def test_w4a8_layer_matches_dense_composition():
    rng = np.random.default_rng(5)
    T, H, E, k, I = 5, 64, 4, 2, 32
    x, r = rng.standard_normal((T, H)), rng.standard_normal((T, H))
    nw = 1 + 0.1 * rng.standard_normal(H)
    Wg = rng.standard_normal((H, E)) * 0.3
    w13 = [rng.standard_normal((H, 2 * I)) * 0.2 for _ in range(E)]
    down = [rng.standard_normal((I, H)) * 0.2 for _ in range(E)]
    res = O.moe_forward_w4a8(x, r, nw, 1e-6, Wg, w13, down, k)
    _, y = O.add_rmsnorm(x, r, nw, 1e-6)
    ids, w = O.gating_topk_softmax(O.router_logits_f32(y, Wg), k)
    ref = np.zeros((T, H))
    for t in range(T):
        a = O.mx_roundtrip(y[t:t + 1])
        for sl in range(k):
            e = ids[t, sl]
            h = O.swiglu(a @ O.mx4_roundtrip(w13[e], axis=0))
            ref[t] += w[t, sl] * (O.mx_roundtrip(h) @ O.mx4_roundtrip(down[e], axis=0))[0]
    np.testing.assert_allclose(res["out"], ref, rtol=1e-11, atol=1e-12)


def test_expert_map_thread_pool_gives_identical_results():
    """The per-expert loop run on a thread pool (as the full-size GPU parity tests
    do) writes the same values as the serial loop, for the three layer oracles."""
    from concurrent.futures import ThreadPoolExecutor
    rng = np.random.default_rng(8)
    T, H, E, k, I = 9, 64, 6, 2, 32
    x, r = rng.standard_normal((T, H)), rng.standard_normal((T, H))
    nw = 1 + 0.1 * rng.standard_normal(H)
    Wg = rng.standard_normal((H, E)) * 0.3
    w13 = [rng.standard_normal((H, 2 * I)) * 0.2 for _ in range(E)]
    down = [rng.standard_normal((I, H)) * 0.2 for _ in range(E)]
    with ThreadPoolExecutor(4) as ex:
        a = O.moe_forward(x, Wg, w13, down, k, expert_map=ex.map)
        b = O.moe_forward_mx(x, r, nw, 1e-6, Wg, w13, down, k, expert_map=ex.map)
        c = O.moe_forward_w4a8(x, r, nw, 1e-6, Wg, w13, down, k, expert_map=ex.map)
    np.testing.assert_array_equal(a["out"], O.moe_forward(x, Wg, w13, down, k)["out"])
    np.testing.assert_array_equal(a["h"], O.moe_forward(x, Wg, w13, down, k)["h"])
    np.testing.assert_array_equal(b["out"], O.moe_forward_mx(x, r, nw, 1e-6, Wg, w13, down, k)["out"])
    np.testing.assert_array_equal(c["out"], O.moe_forward_w4a8(x, r, nw, 1e-6, Wg, w13, down, k)["out"])


def test_forced_topk_logits_give_the_requested_loads():
    """The designed logits of the token-block boundary tests route exactly the
    requested number of rows to each expert (checked with the oracle's gating)."""
    from tests._helpers import forced_topk_logits
    for counts, k in (([256, 257, 255, 512, 513, 1, 0, 254], 2), ([5, 0, 7, 3, 6], 3)):
        lg = forced_topk_logits(counts, k, seed=3)
        ids, w = O.gating_topk_softmax(lg, k)
        assert np.bincount(ids.ravel(), minlength=len(counts)).tolist() == list(counts)
        assert all(len(set(row)) == k for row in ids.tolist())
