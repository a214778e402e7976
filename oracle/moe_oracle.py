"""CPU fp64 oracle for the Qwen3-MoE-style MoE-layer forward.

TEST INFRASTRUCTURE.  This module is the plain, slow, obviously-correct statement
of what the GPU library computes.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it; the library never does,
and it imports nothing from the library.

Sources (three blog pages on Ascend CANN inference recipes; titles as printed):

* [Q3MoE] "基于Atlas A3、950训练/推理集群的Qwen3-MoE模型低时延推理性能优化实践"
  - §计算分解: each expert is an MLP ``x -> down(SiLU(gate(x)) * up(x))``; gate_proj
    and up_proj are merged into one weight ``w13`` and the SwiGLU op splits the
    product in two along the last dim (``torch.chunk(x, 2, -1)``) and returns
    ``SiLU(x[0]) * x[1]`` -- so the first half is gate, the second up.
  - §使能融合算子GMM使能和Routing优化: a per-expert loop is the slow baseline; the
    grouped matmul computes all experts at once.
  - §快速选择专家: one fused op replaces "top-k then softmax" for the router scores.
  - §高效排序和token路由: init_routing sorts tokens by expert; compute_expert_tokens
    gives each expert's token count; finalize_routing puts expert outputs back in
    token order and sums them with the router weights.
  - §融合算子优化 / 融合RMSNorm MX量化: residual add + RMSNorm + MXFP8 dynamic quant
    (round mode "rint", e4m3fn data) in one op; §融合RMSNorm Cast: the router runs
    on the fp32 normalised activations.
* The MX block format (32-element blocks, E8M0 shared scale, scale exponent
  ``floor(log2(amax)) - emax_elem``) is the OCP Microscaling Formats spec v1.0;
  the pages only name "MXFP8".

Readings where the pages are silent (the CUDA path takes the same ones):
top-k ranks the fp32 logits, ties go to the lower expert id, slot order is that
ranking; weights are renormalised over the k chosen experts; pairs are numbered
token-major (j = t*k + s) and sorted stably by expert; ``expanded_row_idx[j]`` is
the sorted position of pair j and ``sorted_row_idx`` its inverse; the layer output
is the fp64 weighted sum over slots.

All floating-point work here is fp64.  Inputs are numpy arrays holding the exact
values of the bf16 / fp32 tensors (bf16 values widened to fp32 or fp64).

Parity pins: every function below is checked in ``tests/test_oracle.py`` against
something other than itself (closed forms, library routines on special cases,
brute force, invariants, hand-derived fixtures in ``tests/golden/``).
"""
from __future__ import annotations

import itertools
from typing import Dict, Optional, Sequence

import numpy as np

# --------------------------------------------------------------------------- #
# Router                                                                       #
# --------------------------------------------------------------------------- #


def router_logits(x: np.ndarray, Wg: np.ndarray) -> np.ndarray:
    """Router scores l[t, e] = sum_h x[t, h] * Wg[h, e] in fp64.

    [Q3MoE §融合RMSNorm Cast]: the gate (router) input is kept in FP32, so the
    weights are fp32 and the product is accumulated exactly enough (fp64) that
    rounding to fp32 afterwards is the only rounding.
    """
    return np.asarray(x, np.float64) @ np.asarray(Wg, np.float64)


def router_logits_f32(x: np.ndarray, Wg: np.ndarray) -> np.ndarray:
    """The oracle's fp32 logits: one round-to-nearest of the fp64 product."""
    return router_logits(x, Wg).astype(np.float32)


# --------------------------------------------------------------------------- #
# Gating: softmax over experts, top-k, renormalise                            #
# --------------------------------------------------------------------------- #


def topk_order(logits_row: np.ndarray, k: int) -> np.ndarray:
    """Experts of one token ranked by (logit descending, expert id ascending);
    the first k.  Ranking is done on the fp32 logits themselves (exact compares)."""
    E = logits_row.shape[0]
    ids = np.arange(E)
    # np.lexsort sorts by the last key first: primary -logit, secondary id.
    order = np.lexsort((ids, -logits_row.astype(np.float64)))
    return order[:k]


def gating_topk_softmax(logits: np.ndarray, k: int, renormalize: bool = True):
    """[Q3MoE §快速选择专家] token->expert selection and weights.

    Softmax over all E experts, keep the k largest, renormalise the kept k to sum
    to 1.  Because softmax is monotone, the k largest probabilities are the k
    largest logits, and after renormalisation the full softmax denominator cancels:
    w_s = exp(l_s - m) / sum_{s'} exp(l_{s'} - m) over the chosen k (m = their max).
    That is also the pages' "top-k, then softmax".  With ``renormalize=False`` the
    weights are the full-softmax probabilities of the chosen experts.

    Returns (ids int32 (T,k), weights fp64 (T,k)); slot s is the s-th ranked expert.
    """
    logits = np.asarray(logits)
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    for t in range(T):
        row = logits[t].astype(np.float64)
        sel = topk_order(logits[t], k)
        ids[t] = sel
        if renormalize:
            z = row[sel] - row[sel].max()
            ez = np.exp(z)
            w[t] = ez / ez.sum()
        else:
            z = row - row.max()
            ez = np.exp(z)
            w[t] = ez[sel] / ez.sum()
    return ids, w


# --------------------------------------------------------------------------- #
# Routing: histogram, stable counting sort of token-expert pairs              #
# --------------------------------------------------------------------------- #


def compute_expert_tokens(topk_ids: np.ndarray, E: int):
    """[Q3MoE §高效排序和token路由] tokens each expert must compute.

    counts[e] = #{pairs j with id_j == e}; offsets is the exclusive prefix sum with
    offsets[E] = number of pairs.
    """
    flat = np.asarray(topk_ids).reshape(-1)
    counts = np.zeros(E, np.int64)
    for e in flat:
        counts[int(e)] += 1
    offsets = np.zeros(E + 1, np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    return counts.astype(np.int32), offsets.astype(np.int32)


def init_routing(topk_ids: np.ndarray, E: int):
    """[Q3MoE §高效排序和token路由] expert ordering of the token-expert pairs.

    Pairs are numbered token-major, j = t*k + s.  Pair j goes to sorted position
    p(j) = offsets[id_j] + #{j' < j : id_j' == id_j}: a stable counting sort by
    expert id.  expanded_row_idx[j] = p(j); sorted_row_idx[p(j)] = j.  Row p of the
    expanded activations is token sorted_row_idx[p] // k.
    """
    flat = np.asarray(topk_ids).reshape(-1)
    counts, offsets = compute_expert_tokens(flat, E)
    seen = np.zeros(E, np.int64)
    P = flat.shape[0]
    expanded_row_idx = np.empty(P, np.int32)
    sorted_row_idx = np.empty(P, np.int32)
    for j in range(P):
        e = int(flat[j])
        p = int(offsets[e]) + int(seen[e])
        seen[e] += 1
        expanded_row_idx[j] = p
        sorted_row_idx[p] = j
    return dict(counts=counts, offsets=offsets, expanded_row_idx=expanded_row_idx,
                sorted_row_idx=sorted_row_idx)


# --------------------------------------------------------------------------- #
# Expert MLP                                                                   #
# --------------------------------------------------------------------------- #


def sigmoid(z: np.ndarray) -> np.ndarray:
    """1 / (1 + e^-z), written to avoid overflow for large |z|."""
    z = np.asarray(z, np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def swiglu(gu: np.ndarray) -> np.ndarray:
    """[Q3MoE §计算分解] split the last dim in two halves (gate, up) and return
    SiLU(gate) * up, SiLU(z) = z * sigmoid(z)."""
    n = gu.shape[-1]
    if n % 2:
        raise ValueError("last dim must be even")
    g = gu[..., : n // 2]
    u = gu[..., n // 2:]
    return g * sigmoid(g) * u


def expert_mlp(a: np.ndarray, w13_e: np.ndarray, down_e: np.ndarray, return_h: bool = False):
    """[Q3MoE §计算分解] one expert: down(SiLU(gate(a)) * up(a)) in fp64.

    a (m,H); w13_e (H,2I) = [gate_proj | up_proj]; down_e (I,H).
    """
    a = np.asarray(a, np.float64)
    gu = a @ np.asarray(w13_e, np.float64)
    h = swiglu(gu)
    y = h @ np.asarray(down_e, np.float64)
    return (y, h) if return_h else y


# --------------------------------------------------------------------------- #
# Whole layer                                                                  #
# --------------------------------------------------------------------------- #


def moe_forward(x: np.ndarray, Wg: np.ndarray, w13: Sequence[np.ndarray], down: Sequence[np.ndarray],
                k: int, logits32: Optional[np.ndarray] = None, renormalize: bool = True,
                keep_intermediates: bool = True, expert_map=map) -> Dict[str, np.ndarray]:
    """The MoE layer: router -> gating -> init_routing -> per-expert MLP on the
    expert-sorted rows -> finalize (un-permute, weighted sum over the k slots).

    ``w13[e]`` / ``down[e]`` may be any array-likes (converted to fp64 one expert at a
    time, so fp32 copies of large bf16 weights are enough).  ``logits32`` replaces
    the router output (the fp32 logits the GPU is fed in routing-exact checks).
    ``expert_map(f, experts)`` runs the per-expert MLPs (default: the builtin
    ``map``; a thread pool's ``map`` gives the same values, since each expert's
    rows are computed on their own and written to their own slice).

    [Q3MoE §高效排序和token路由, §高性能专家计算, §计算分解]
    """
    x = np.asarray(x)
    T, H = x.shape
    E = len(w13)
    if logits32 is None:
        logits32 = router_logits_f32(x, Wg)
    ids, w = gating_topk_softmax(logits32, k, renormalize)
    rt = init_routing(ids, E)
    P = T * k
    I = np.asarray(w13[0]).shape[1] // 2
    offs = rt["offsets"]
    sri = rt["sorted_row_idx"]
    h_all = np.zeros((P, I), np.float64) if keep_intermediates else None
    y_all = np.zeros((P, H), np.float64)

    def one_expert(e):
        lo, hi = int(offs[e]), int(offs[e + 1])
        tokens = sri[lo:hi] // k
        y, h = expert_mlp(x[tokens], w13[e], down[e], return_h=True)
        y_all[lo:hi] = y
        if keep_intermediates:
            h_all[lo:hi] = h

    for _ in expert_map(one_expert, [e for e in range(E) if offs[e + 1] > offs[e]]):
        pass
    out = np.zeros((T, H), np.float64)
    eri = rt["expanded_row_idx"]
    for t in range(T):
        for s in range(k):
            out[t] += w[t, s] * y_all[eri[t * k + s]]
    res = dict(logits32=np.asarray(logits32, np.float32), topk_ids=ids, topk_w=w, out=out, **rt)
    if keep_intermediates:
        res["h"] = h_all
        res["y2"] = y_all
    return res


def finalize_routing(y2: np.ndarray, topk_w: np.ndarray, expanded_row_idx: np.ndarray, k: int) -> np.ndarray:
    """[Q3MoE §高效排序和token路由] out[t] = sum_s w[t,s] * y2[expanded_row_idx[t*k+s]]."""
    T = topk_w.shape[0]
    out = np.zeros((T, y2.shape[1]), np.float64)
    for t in range(T):
        for s in range(k):
            out[t] += float(topk_w[t, s]) * np.asarray(y2[expanded_row_idx[t * k + s]], np.float64)
    return out


# --------------------------------------------------------------------------- #
# RMSNorm and MXFP8                                                            #
# --------------------------------------------------------------------------- #


def add_rmsnorm(x: np.ndarray, r: Optional[np.ndarray], w: np.ndarray, eps: float):
    """[Q3MoE §融合RMSNorm MX量化] residual add then RMSNorm (LayerNorm without the
    mean subtraction, §RmsNorm算子优化): s = x + r; y = s / sqrt(mean(s^2) + eps) * w.
    With r None (first layer) s = x.  Returns (s, y) in fp64."""
    s = np.asarray(x, np.float64)
    if r is not None:
        s = s + np.asarray(r, np.float64)
    ms = np.mean(s * s, axis=-1, keepdims=True)
    y = s / np.sqrt(ms + eps) * np.asarray(w, np.float64)
    return s, y


E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest normal: 448 = 1.75 * 2^8
MX_BLOCK = 32


def e4m3_value(code: int) -> float:
    """Value of an 8-bit float8 e4m3fn code: 1 sign, 4 exponent (bias 7), 3 mantissa
    bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no inf."""
    s = -1.0 if (code >> 7) & 1 else 1.0
    ex = (code >> 3) & 0xF
    m = code & 0x7
    if ex == 0xF and m == 0x7:
        return float("nan")
    if ex == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (ex - 7)


_E4M3_POS = np.array([e4m3_value(c) for c in range(0x7F)], np.float64)   # codes 0x00..0x7E


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3fn value, ties to the even code, saturating to
    +-448 (the "rint" round mode of [Q3MoE §融合RMSNorm MX量化] with saturation to
    the largest finite value).  Returns uint8 codes."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    # nearest candidate among the 127 non-negative finite values (sorted ascending)
    hi = np.searchsorted(_E4M3_POS, a, side="left")
    hi = np.clip(hi, 0, len(_E4M3_POS) - 1)
    lo = np.clip(hi - 1, 0, len(_E4M3_POS) - 1)
    dlo = a - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    # the sign is kept on zero results too (-tiny rounds to -0, code 0x80)
    sign = np.signbit(v).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    table = np.array([e4m3_value(c) for c in range(256)], np.float64)
    return table[np.asarray(codes, np.int64)]


def mx_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """OCP MX v1.0 shared scale: X = floor(log2(amax)) - emax_elem, clamped to the
    E8M0 range [-127, 127]; an all-zero block gets X = -127."""
    amax = np.asarray(amax, np.float64)
    X = np.full(amax.shape, -127, np.int64)
    nz = amax > 0
    _, ex = np.frexp(amax[nz])          # amax = f * 2^ex, f in [0.5, 1)
    X[nz] = np.clip((ex - 1) - E4M3_EMAX, -127, 127)
    return X


def mx_quantize(y: np.ndarray, block: int = MX_BLOCK):
    """MXFP8 quantisation along the last axis in blocks of ``block`` elements.

    Returns (codes uint8 same shape as y, scale bytes uint8 [..., n/block]) where
    scale byte = X + 127 (E8M0) and codes = e4m3_encode(y / 2^X).
    """
    y = np.asarray(y, np.float64)
    n = y.shape[-1]
    if n % block:
        raise ValueError("last dim must be a multiple of the block")
    yb = y.reshape(y.shape[:-1] + (n // block, block))
    amax = np.max(np.abs(yb), axis=-1)
    X = mx_scale_exponent(amax)
    codes = e4m3_encode(yb / np.exp2(X.astype(np.float64))[..., None])
    return codes.reshape(y.shape), (X + 127).astype(np.uint8)


def mx_dequantize(codes: np.ndarray, scales: np.ndarray, block: int = MX_BLOCK) -> np.ndarray:
    v = e4m3_decode(codes)
    n = v.shape[-1]
    vb = v.reshape(v.shape[:-1] + (n // block, block))
    sc = np.exp2(np.asarray(scales, np.float64) - 127.0)
    return (vb * sc[..., None]).reshape(v.shape)


def mx_roundtrip(y: np.ndarray, axis: int = -1) -> np.ndarray:
    """Quantise-dequantise along ``axis`` (the GEMM reduction axis)."""
    y = np.moveaxis(np.asarray(y, np.float64), axis, -1)
    q, s = mx_quantize(y)
    return np.moveaxis(mx_dequantize(q, s), -1, axis)


def moe_forward_mx(x: np.ndarray, r: Optional[np.ndarray], norm_w: np.ndarray, eps: float,
                   Wg: np.ndarray, w13: Sequence[np.ndarray], down: Sequence[np.ndarray], k: int,
                   logits32: Optional[np.ndarray] = None, expert_map=map) -> Dict[str, np.ndarray]:
    """MXFP8 layer [Q3MoE §融合RMSNorm MX量化, §融合RMSNorm Cast].

    s = x + r; y = RMSNorm(s); the router sees the unquantised y; the experts see
    MX(y) along H, weights MX-quantised along their reduction axis (H for w13, I for
    down), and h MX-quantised along I before the down projection.  Everything is
    then computed in fp64 on the dequantised values.  ``expert_map`` as in
    ``moe_forward``.
    """
    s, y = add_rmsnorm(x, r, norm_w, eps)
    if logits32 is None:
        logits32 = router_logits_f32(y, Wg)
    yq = mx_roundtrip(y, axis=-1)
    ids, w = gating_topk_softmax(logits32, k)
    E = len(w13)
    rt = init_routing(ids, E)
    T, H = y.shape
    P = T * k
    offs, sri, eri = rt["offsets"], rt["sorted_row_idx"], rt["expanded_row_idx"]
    y_all = np.zeros((P, H), np.float64)

    def one_expert(e):
        lo, hi = int(offs[e]), int(offs[e + 1])
        a = yq[sri[lo:hi] // k]
        w13q = mx_roundtrip(w13[e], axis=0)
        downq = mx_roundtrip(down[e], axis=0)
        h = swiglu(a @ w13q)
        hq = mx_roundtrip(h, axis=-1)
        y_all[lo:hi] = hq @ downq

    for _ in expert_map(one_expert, [e for e in range(E) if offs[e + 1] > offs[e]]):
        pass
    out = np.zeros((T, H), np.float64)
    for t in range(T):
        for s_ in range(k):
            out[t] += w[t, s_] * y_all[eri[t * k + s_]]
    return dict(residual=s, y=y, logits32=np.asarray(logits32, np.float32), topk_ids=ids,
                topk_w=w, out=out, **rt)


# --------------------------------------------------------------------------- #
# Independent formulations used only to pin the oracle                        #
# --------------------------------------------------------------------------- #


def dense_moe_reference(x: np.ndarray, w13, down, topk_ids: np.ndarray, topk_w: np.ndarray) -> np.ndarray:
    """The per-expert loop formulation the pages call the slow baseline
    [Q3MoE §使能融合算子GMM使能和Routing优化]: run every expert on every token,
    then mask with a dense (T,E) routing-weight matrix.  No sorting involved."""
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    E = len(w13)
    dense_w = np.zeros((T, E), np.float64)
    for t in range(T):
        for s in range(topk_ids.shape[1]):
            dense_w[t, int(topk_ids[t, s])] += topk_w[t, s]
    out = np.zeros((T, x.shape[1]), np.float64)
    for e in range(E):
        y = expert_mlp(x, w13[e], down[e])
        out += dense_w[:, e:e + 1] * y
    return out


def brute_force_topk(logits_row: np.ndarray, k: int) -> np.ndarray:
    """Top-k by enumeration of all k-subsets (tiny E only): the chosen set is the
    one whose members each beat every non-member under (logit desc, id asc)."""
    E = logits_row.shape[0]

    def beats(a, b):
        return logits_row[a] > logits_row[b] or (logits_row[a] == logits_row[b] and a < b)

    for subset in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in subset]
        if all(beats(a, b) for a in subset for b in rest):
            members = list(subset)
            # slot order: insertion by pairwise comparison
            ordered = sorted(members, key=lambda a: sum(beats(b, a) for b in members))
            return np.array(ordered, np.int64)
    raise AssertionError("no top-k subset found")


# --------------------------------------------------------------------------- #
# Next rows: fused add + RMSNorm + cast, EP-local routing, re-routing,         #
# zero-computation experts                                                     #
# --------------------------------------------------------------------------- #


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even) and return them as fp64:
    keep the top 16 bits of the fp32 pattern after adding 0x7FFF + lsb."""
    f = np.asarray(v, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def add_rmsnorm_cast(x: np.ndarray, r: Optional[np.ndarray], w: np.ndarray, eps: float):
    """[Q3MoE §融合RMSNorm Cast] residual add + RMSNorm with two outputs: the
    normalised activations in FP32 for the gate (router) and in BF16 for the
    experts.  Returns (s, y fp64, y_bf16 as fp64 values); the bf16 output is the
    rounding of the fp32 value of y."""
    s, y = add_rmsnorm(x, r, w, eps)
    return s, y, bf16_round(y.astype(np.float32))


def init_routing_v2(topk_ids: np.ndarray, E_total: int, expert_begin: int, expert_end: int):
    """Expert-range routing [Q3MoE §计算分解(AllGather方案): init_routing_v2 keeps only
    the tokens whose expert lies in this rank's range].  Pairs whose id is in
    [expert_begin, expert_end) are sorted stably by local id (id - expert_begin);
    the others get expanded_row_idx = -1 (another rank's expert, or a zero-computation
    expert).  Ids outside [0, E_total) are invalid and also get -1."""
    flat = np.asarray(topk_ids).reshape(-1)
    El = expert_end - expert_begin
    local = np.where((flat >= expert_begin) & (flat < expert_end), flat - expert_begin, -1)
    counts = np.zeros(El, np.int64)
    for e in local:
        if e >= 0:
            counts[e] += 1
    offsets = np.zeros(El + 1, np.int64)
    for e in range(El):
        offsets[e + 1] = offsets[e] + counts[e]
    seen = np.zeros(El, np.int64)
    P = flat.shape[0]
    eri = np.full(P, -1, np.int32)
    sri = np.full(P, -1, np.int32)
    for j in range(P):
        e = int(local[j])
        if e < 0:
            continue
        p = int(offsets[e] + seen[e])
        seen[e] += 1
        eri[j] = p
        sri[p] = j
    return dict(counts=counts.astype(np.int32), offsets=offsets.astype(np.int32),
                expanded_row_idx=eri, sorted_row_idx=sri)


def re_routing(tokens_per_expert: np.ndarray):
    """[Q3MoE §计算分解(Double Routing方案): npu_moe_re_routing re-sorts the tokens received
    by the AlltoAll by local expert].  Received rows arrive grouped by source rank and,
    inside a rank's block, by local expert: counts[r][e] rows for (r, e), in that
    order.  Re-routing orders them by expert, then source rank (stable).  Returns
    (perm, expert_offsets): received row i goes to output row perm[i]."""
    cnt = np.asarray(tokens_per_expert, np.int64)
    R, El = cnt.shape
    out_base = np.zeros((R, El), np.int64)
    acc = 0
    for e in range(El):
        for r in range(R):
            out_base[r, e] = acc
            acc += cnt[r, e]
    perm = np.empty(acc, np.int64)
    i = 0
    for r in range(R):
        for e in range(El):
            for q in range(cnt[r, e]):
                perm[i] = out_base[r, e] + q
                i += 1
    offsets = np.zeros(El + 1, np.int64)
    for e in range(El):
        offsets[e + 1] = offsets[e] + cnt[:, e].sum()
    return perm.astype(np.int32), offsets.astype(np.int32)


def moe_forward_v2(x: np.ndarray, r: Optional[np.ndarray], norm_w: Optional[np.ndarray], eps: float,
                   Wg: np.ndarray, w13, down, k: int, num_zero_experts: int = 0,
                   logits32: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """The bf16 layer with the optional fused add+RMSNorm+cast in front and optional
    zero-computation experts.

    * With norm_w: s = x + r, y = RMSNorm(s); the router sees fp32 y, the experts
      bf16(y) [Q3MoE §融合RMSNorm Cast]; without, the experts and router see x.
    * Router scores cover E routed + Z zero-computation experts (ids E..E+Z-1).  A
      zero-computation expert returns its input unchanged, MoE(x) = x (page
      "基于Atlas A3集群的LongCat-Flash模型推理性能优化实践", §MoE模块实现Expert
      Parallel, copy_expert_num), so it adds w * (expert input) to the output.
    """
    E = len(w13)
    if norm_w is not None:
        s, y, ybf = add_rmsnorm_cast(x, r, norm_w, eps)
        router_in, expert_in = y, ybf
    else:
        s = None
        router_in = expert_in = np.asarray(x, np.float64)
    if logits32 is None:
        logits32 = router_logits_f32(router_in, Wg)
    ids, w = gating_topk_softmax(logits32, k)
    rt = init_routing_v2(ids, E + num_zero_experts, 0, E)
    T, H = expert_in.shape
    offs, sri, eri = rt["offsets"], rt["sorted_row_idx"], rt["expanded_row_idx"]
    y_all = np.zeros((T * k, H), np.float64)
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            y_all[lo:hi] = expert_mlp(expert_in[sri[lo:hi] // k], w13[e], down[e])
    out = np.zeros((T, H), np.float64)
    for t in range(T):
        for sl in range(k):
            j = t * k + sl
            if ids[t, sl] < E:
                out[t] += w[t, sl] * y_all[eri[j]]
            else:
                out[t] += w[t, sl] * expert_in[t]
    res = dict(logits32=np.asarray(logits32, np.float32), topk_ids=ids, topk_w=w, out=out, **rt)
    if s is not None:
        res["residual"] = s
        res["y"] = router_in
        res["y_bf16"] = expert_in
    return res


# --------------------------------------------------------------------------- #
# W4A8: MXFP4 (e2m1) expert weights, MXFP8 activations                        #
# --------------------------------------------------------------------------- #

E2M1_MAX = 6.0
E2M1_EMAX = 2          # 6 = 1.5 * 2^2


def e2m1_value(code: int) -> float:
    """Value of a 4-bit e2m1 code: 1 sign, 2 exponent (bias 1), 1 mantissa bit;
    exponent field 0 is subnormal (m/2 * 2^0); no inf or NaN (OCP MX v1.0)."""
    s = -1.0 if (code >> 3) & 1 else 1.0
    ex = (code >> 1) & 3
    m = code & 1
    if ex == 0:
        return s * 0.5 * m
    return s * (1.0 + 0.5 * m) * 2.0 ** (ex - 1)


_E2M1_POS = np.array([e2m1_value(c) for c in range(8)], np.float64)   # 0 .. 6, ascending


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Round to the nearest e2m1 value, ties to the even code, saturating at +-6
    (the page's W4A8 uses MXFP4 weights, [Q3MoE §计算分解(AllGather方案)])."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), E2M1_MAX)
    hi = np.clip(np.searchsorted(_E2M1_POS, a, side="left"), 0, 7)
    lo = np.clip(hi - 1, 0, 7)
    dlo = a - _E2M1_POS[lo]
    dhi = _E2M1_POS[hi] - a
    code = np.where((dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0)), hi, lo).astype(np.int64)
    return (code | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    table = np.array([e2m1_value(c) for c in range(16)], np.float64)
    return table[np.asarray(codes, np.int64) & 15]


def mx4_quantize(y: np.ndarray, block: int = MX_BLOCK):
    """MXFP4 along the last axis: X = floor(log2 amax) - 2 clamped to [-127,127],
    codes = e2m1(y / 2^X); returns (codes uint8, one per element, and scale bytes)."""
    y = np.asarray(y, np.float64)
    n = y.shape[-1]
    yb = y.reshape(y.shape[:-1] + (n // block, block))
    amax = np.max(np.abs(yb), axis=-1)
    X = np.full(amax.shape, -127, np.int64)
    nz = amax > 0
    _, ex = np.frexp(amax[nz])
    X[nz] = np.clip((ex - 1) - E2M1_EMAX, -127, 127)
    codes = e2m1_encode(yb / np.exp2(X.astype(np.float64))[..., None])
    return codes.reshape(y.shape), (X + 127).astype(np.uint8)


def mx4_roundtrip(y: np.ndarray, axis: int = -1) -> np.ndarray:
    y = np.moveaxis(np.asarray(y, np.float64), axis, -1)
    q, s = mx4_quantize(y)
    n = y.shape[-1]
    v = e2m1_decode(q).reshape(y.shape[:-1] + (n // MX_BLOCK, MX_BLOCK))
    v = v * np.exp2(s.astype(np.float64) - 127.0)[..., None]
    return np.moveaxis(v.reshape(y.shape), -1, axis)


def moe_forward_w4a8(x, r, norm_w, eps, Wg, w13, down, k, logits32=None, expert_map=map):
    """The MXFP8 layer of moe_forward_mx with MXFP4 expert weights: identical except
    that w13 (along H) and down (along I) are quantised to e2m1 + E8M0/32.
    ``expert_map`` as in ``moe_forward``."""
    s, y = add_rmsnorm(x, r, norm_w, eps)
    if logits32 is None:
        logits32 = router_logits_f32(y, Wg)
    yq = mx_roundtrip(y, axis=-1)
    ids, w = gating_topk_softmax(logits32, k)
    E = len(w13)
    rt = init_routing(ids, E)
    T, H = y.shape
    offs, sri, eri = rt["offsets"], rt["sorted_row_idx"], rt["expanded_row_idx"]
    y_all = np.zeros((T * k, H), np.float64)

    def one_expert(e):
        lo, hi = int(offs[e]), int(offs[e + 1])
        h = swiglu(yq[sri[lo:hi] // k] @ mx4_roundtrip(w13[e], axis=0))
        y_all[lo:hi] = mx_roundtrip(h) @ mx4_roundtrip(down[e], axis=0)

    for _ in expert_map(one_expert, [e for e in range(E) if offs[e + 1] > offs[e]]):
        pass
    out = np.zeros((T, H), np.float64)
    for t in range(T):
        for s_ in range(k):
            out[t] += w[t, s_] * y_all[eri[t * k + s_]]
    return dict(residual=s, logits32=np.asarray(logits32, np.float32), topk_ids=ids, topk_w=w, out=out, **rt)
