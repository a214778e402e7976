"""Seeded synthetic workloads for the MoE-layer forward.

This module only draws random inputs; it holds none of the layer's arithmetic, so
the CUDA path and the CPU oracle can both be fed from it without sharing any
computation.  Every tensor is drawn from ``torch.Generator`` seeded with the
config's seed, in a fixed order: x, r, W_g, the Zipf rank permutation, w13, down,
norm weight (tensors a config does not use are not drawn).

Shapes follow the Qwen3-MoE family that the page "基于Atlas A3、950训练/推理集群的
Qwen3-MoE模型低时延推理性能优化实践" optimises (single-batch decode and a 4K
prefill, §概述), with the layer written as ``x -> down(SiLU(gate(x)) * up(x))``
per expert (§计算分解).

Router skew.  The Zipf-skewed prefill gives every expert a logit bias
``-s * ln(rank_e)`` (s = 1.2, ranks 1..E from a seeded permutation).  The layer's
API has no bias input, so the bias is carried by the input itself: channel 0 of
every token is set to exactly 1.0 and row 0 of W_g holds the bias, which makes
``x @ W_g`` contain it.  The other H-1 channels keep their N(0, 1) draw.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int          # tokens
    H: int          # hidden size
    E: int          # routed experts
    k: int          # experts per token
    I: int          # expert intermediate size
    router: str = "uniform"   # "uniform" or "zipf"
    zipf_s: float = 1.2
    mx: bool = False          # MXFP8 variant (add + RMSNorm + MX quant in front)
    w4: bool = False          # with mx: MXFP4 expert weights (W4A8)
    prenorm: bool = False     # bf16 layer with fused add + RMSNorm + cast in front
    Z: int = 0                # zero-computation (identity) experts after the E routed ones
    ep_ranks: int = 0         # > 0: routing of one expert-parallel rank's experts only
    eps: float = 1e-6
    seed: int = 0

    @property
    def P(self) -> int:
        return self.T * self.k


# The five shapes this library is measured and checked on.
CONFIGS: Dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", T=16, H=256, E=8, k=2, I=128),
    "qwen3_30b_a3b_decode": MoEConfig("qwen3_30b_a3b_decode", T=32, H=2048, E=128, k=8, I=768),
    "qwen3_30b_a3b_prefill_zipf": MoEConfig("qwen3_30b_a3b_prefill_zipf", T=4096, H=2048, E=128,
                                            k=8, I=768, router="zipf"),
    "qwen3_235b_a22b_decode": MoEConfig("qwen3_235b_a22b_decode", T=64, H=4096, E=128, k=8, I=1536),
    "qwen3_235b_a22b_prefill": MoEConfig("qwen3_235b_a22b_prefill", T=8192, H=4096, E=128, k=8,
                                         I=1536),
    "mxfp8_prefill": MoEConfig("mxfp8_prefill", T=4096, H=4096, E=128, k=8, I=1536, mx=True),
    "mxfp8_decode": MoEConfig("mxfp8_decode", T=64, H=4096, E=128, k=8, I=1536, mx=True),
    # W4A8: the MXFP8 layer with MXFP4 (e2m1 + E8M0/32) expert weights, Qwen3-235B shape
    "w4a8_prefill": MoEConfig("w4a8_prefill", T=4096, H=4096, E=128, k=8, I=1536, mx=True, w4=True),
    "w4a8_decode": MoEConfig("w4a8_decode", T=64, H=4096, E=128, k=8, I=1536, mx=True, w4=True),
    # next rows: fused add+RMSNorm+cast in front of the decode layer; identity experts
    "qwen3_30b_a3b_decode_prenorm": MoEConfig("qwen3_30b_a3b_decode_prenorm", T=32, H=2048, E=128, k=8,
                                              I=768, prenorm=True),
    "zero_experts_decode": MoEConfig("zero_experts_decode", T=32, H=2048, E=128, k=8, I=768, Z=64),
    # one rank of 4-way expert parallelism at the Qwen3-235B prefill size: expert-range
    # routing of all gathered tokens plus re-routing of the received blocks
    "ep4_rank_routing_qwen3_235b_prefill": MoEConfig("ep4_rank_routing_qwen3_235b_prefill", T=8192,
                                                     H=4096, E=128, k=8, I=1536, ep_ranks=4),
}


def with_shape(cfg: MoEConfig, **kw) -> MoEConfig:
    """A copy of ``cfg`` with some fields replaced (used for small test variants)."""
    return dataclasses.replace(cfg, **kw)


def _randn(gen: torch.Generator, shape, std: float, mean: float = 0.0, device="cpu") -> torch.Tensor:
    t = torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def make_inputs(cfg: MoEConfig, device: str = "cpu", weights: bool = True) -> Dict[str, torch.Tensor]:
    """Draw the config's inputs on ``device`` (the generator lives on that device).

    Returns bf16 ``x`` (T,H), fp32 ``Wg`` (H,E+Z), bf16 ``w13`` (E,H,2I) whose first I
    columns are gate_proj and last I are up_proj, bf16 ``down`` (E,I,H); for the MXFP8
    and pre-norm variants also bf16 ``r`` (T,H) and bf16 ``norm_w`` (H,).  bf16 casts round to
    nearest even.  ``weights=False`` skips w13/down (for routing-only checks).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed)
    out: Dict[str, torch.Tensor] = {}
    x = _randn(gen, (cfg.T, cfg.H), 1.0, device=device)
    normed = cfg.mx or cfg.prenorm
    if normed:
        r = _randn(gen, (cfg.T, cfg.H), 1.0, device=device)
    Wg = _randn(gen, (cfg.H, cfg.E + cfg.Z), 0.02, device=device)
    if cfg.router == "zipf":
        perm = torch.randperm(cfg.E, generator=gen, device=device)
        rank = torch.empty(cfg.E, dtype=torch.float32, device=device)
        rank[perm] = torch.arange(1, cfg.E + 1, dtype=torch.float32, device=device)
        Wg[0, :cfg.E] = -cfg.zipf_s * torch.log(rank)
        x[:, 0] = 1.0
    elif cfg.router != "uniform":
        raise ValueError(f"unknown router kind {cfg.router!r}")
    out["x"] = x.to(torch.bfloat16)
    if normed:
        out["r"] = r.to(torch.bfloat16)
    out["Wg"] = Wg.contiguous()
    if weights:
        out["w13"] = _randn(gen, (cfg.E, cfg.H, 2 * cfg.I), 0.02, device=device).to(torch.bfloat16)
        out["down"] = _randn(gen, (cfg.E, cfg.I, cfg.H), 0.02, device=device).to(torch.bfloat16)
        if normed:
            out["norm_w"] = _randn(gen, (cfg.H,), 0.1, mean=1.0, device=device).to(torch.bfloat16)
    return out


def make_logits(T: int, E: int, seed: int, ties: bool = False, device: str = "cpu") -> torch.Tensor:
    """fp32 router logits for gating-only checks.  ``ties=True`` quantises them to a
    coarse grid so that many equal values occur in every row (exercises tie-breaks)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    lg = torch.randn(T, E, generator=gen, dtype=torch.float32, device=device)
    if ties:
        lg = torch.round(lg * 2.0) / 2.0
    return lg.contiguous()


def make_topk_ids(T: int, E: int, k: int, seed: int, skew: Optional[float] = None,
                  device: str = "cpu") -> torch.Tensor:
    """Random (T,k) int32 expert ids, distinct within each token (as top-k gives).
    ``skew`` biases the choice towards low ranks (Zipf-like loads)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    score = torch.rand(T, E, generator=gen, device=device)
    if skew is not None:
        perm = torch.randperm(E, generator=gen, device=device)
        rank = torch.empty(E, dtype=torch.float32, device=device)
        rank[perm] = torch.arange(1, E + 1, dtype=torch.float32, device=device)
        score = torch.log(score.clamp_min(1e-30)) - skew * torch.log(rank)
    ids = torch.topk(score, k, dim=1).indices
    return ids.to(torch.int32).contiguous()


def zipf_bias_magnitude(E: int, s: float) -> float:
    """Largest |bias| of the Zipf router (for docs and sanity checks)."""
    return s * math.log(E)
