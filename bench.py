#!/usr/bin/env python
"""Benchmark of the MoE-layer forward on GB300 (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME|all] [--no-cpu-baseline]

A step is one ``moe_forward`` call (router -> gating -> init_routing -> grouped GEMM
+ SwiGLU -> grouped GEMM -> finalize; the MXFP8 layer adds the fused add + RMSNorm +
MX quantisation in front) over one batch of T tokens of the workload, with inputs
and packed weights resident in HBM.

With no ``--workload`` (``all``) the five measured layer shapes run one after the
other, each in its own timed region: Qwen3-30B-A3B decode (T=32), Qwen3-30B-A3B
prefill with a Zipf-skewed router (T=4096), Qwen3-235B-A22B decode (T=64), the MXFP8
prefill (T=4096, H=4096) and, last, the largest, Qwen3-235B-A22B prefill (T=8192,
H=4096, E=128, k=8, I=1536).  The printed line is that last workload's; it carries
every workload's result under ``"workloads"``.  Each workload's full line also goes
to stderr.

Timing per workload: W untimed warm-up steps; then the headline timed region of K
steps with CUDA events only at its two ends (no event between steps, since an
event between two kernels costs their programmatic launch overlap), bracketed by a
barrier and a device synchronize, max over ranks; then a second, separate pass of
K steps with events around every step and around every grouped-GEMM launch, which
gives the per-step percentiles and the GEMM time behind the roofline; then the
end-to-end pass through pinned host buffers.  Every workload streams more weight
bytes per step than the 129 MB L2 holds (the active experts' weights), so no L2
flush is needed between steps.

Multi-GPU: tokens are independent, so N GPUs run N replicas of the layer on their
own batches with no collective on the data path (weak scaling); torch.distributed
is used only for the barrier and the max-over-ranks of the elapsed time.

``--impl reference`` times the CPU fp64 oracle (the test oracle under ``oracle/``,
unmodified) on the host cores, on the same bounded token sample as the
``cpu_baseline`` field of the GPU arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s on 1 GB300; % of HBM (decode) or tensor-core (prefill) peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
                "clocks_event_reasons.gpu_idle")
# The measured layer shapes, the largest (the headline) last.
SUITE = ("qwen3_30b_a3b_decode", "qwen3_30b_a3b_prefill_zipf", "qwen3_235b_a22b_decode",
         "mxfp8_prefill", "qwen3_235b_a22b_prefill")
HEADLINE = SUITE[-1]
# Tokens per oracle call in the CPU baseline (both arms): the whole batch of a
# decode workload, a slice of this many consecutive tokens of a prefill batch.
ORACLE_SAMPLE_TOKENS = 64


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all", help="a workload name, or 'all' (the five measured shapes)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the cpu_baseline sample")
    ap.add_argument("--shape", default="",
                    help="reduced copy of a single workload for profiling captures, e.g. E=32,T=2048 "
                         "(the line then names the changed sizes; it is not a bench result)")
    return ap.parse_args(argv)


def parse_shape(text: str) -> dict:
    """'E=32,T=2048' -> {'E': 32, 'T': 2048} (integer fields of the workload config)."""
    out = {}
    for part in filter(None, (p.strip() for p in text.split(","))):
        key, _, val = part.partition("=")
        if key not in ("T", "H", "E", "k", "I") or not val.isdigit():
            raise SystemExit(f"--shape: expected T/H/E/k/I=<int>, got {part!r}")
        out[key] = int(val)
    return out


# ----------------------------------------------------------------- helpers ---


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def sustained_bf16_peak():
    """The bf16 GEMM rate measured under a seconds-long loop at the power cap (None if
    MEASURED_PEAKS.json does not give one)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            v = json.load(f).get("bf16_tflops_sustained")
        return float(v) if v else None
    return None


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def file_sha(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the grouped-GEMM kernel from the committed ncu summary,
    or None when there is none or the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"grouped_gemm_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path, encoding="utf-8").read()
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    m_h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", txt)
    if not m_b or not m_h:
        return None
    src = os.path.join(ROOT, "top_routing_grouped_gating_gb300", "csrc",
                       "gmm_mx.cu" if workload.startswith(("mxfp8", "w4a8")) else "gmm.cu")
    if m_h.group(1) != file_sha(src):
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    def __init__(self, dev_index: int):
        import torch
        self.proc = None
        sel = []
        try:
            props = torch.cuda.get_device_properties(dev_index)
            uuid = str(getattr(props, "uuid", "") or "")
            if uuid:
                sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "10"] + sel

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.06)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_samples(out)


def parse_clock_samples(text: str):
    """Summarise nvidia-smi rows of CLOCK_FIELDS.  A sample counts as under load when
    the driver does not report the GPU idle; sm_mhz is the median SM clock of those
    samples (of all samples when none was under load, which samples_under_load = 0
    then says), and reasons are the throttle reasons seen in any sample."""
    rows = [[f.strip() for f in r.split(",")] for r in text.strip().splitlines() if r.count(",") >= 9]
    if not rows:
        return None

    def num(v):
        try:
            return float(v)
        except ValueError:
            return None

    loaded = [r for r in rows if r[9] != "Active"]
    pick = loaded if loaded else rows
    sm = [x for x in (num(r[1]) for r in pick) if x is not None]
    mx = [x for x in (num(r[2]) for r in rows) if x is not None]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded)}


# ------------------------------------------------------ algorithmic work ---


def gemm_weight_bytes(cfg, active: int) -> int:
    """The active experts' w13 and down weights as the grouped GEMM reads them: bf16,
    or e4m3 codes (e2m1: half a byte) plus one E8M0 byte per 32 elements."""
    if cfg.mx:
        return active * 3 * cfg.H * cfg.I * (17 if cfg.w4 else 33) // 32
    return active * 3 * cfg.H * cfg.I * 2


def gemm_implementation_bytes(cfg, pairs: int = -1) -> int:
    """The grouped GEMM's intermediate traffic (not credited to the roofline): the
    expert-sorted activations read, h written and read back, y2 written, for the
    token-expert pairs routed to real experts."""
    P = cfg.T * cfg.k if pairs < 0 else pairs
    if cfg.mx:
        return P * cfg.H * 33 // 32 + 2 * P * cfg.I * 33 // 32 + P * cfg.H * 2
    return P * cfg.H * 2 + 2 * P * cfg.I * 2 + P * cfg.H * 2


def layer_algorithmic_bytes(cfg, active: int) -> int:
    """Bytes the whole layer call must move at the least: the active experts' weights,
    the router weights W_g (fp32), the input x (and the residual r with the norm
    weight for the normed layers) read, the output (and residual_out) written, the
    top-k ids and weights written."""
    T, H, P = cfg.T, cfg.H, cfg.T * cfg.k
    normed = cfg.mx or cfg.prenorm
    b = gemm_weight_bytes(cfg, active)
    b += H * (cfg.E + cfg.Z) * 4
    b += T * H * 2 * (2 if normed else 1) + (H * 2 if normed else 0)
    b += T * H * 2 * (2 if normed else 1)
    b += P * 4 * 2
    return b


def l2_hint_bytes(cfg, sm_count: int, l2_bytes: int) -> int:
    """Bytes of packed w13 that the library's decode-size router launch asks L2 to
    prefetch (the same rule as the C library): 5/8 of the grouped GEMM's first wave
    (one 128-row w13 block of K = H per SM), at most 5/8 of L2 and of w13.  Only the
    CUDA-core router (T <= 64) issues it."""
    if cfg.T > 64:
        return 0
    row = cfg.H // 2 if cfg.w4 else (cfg.H if cfg.mx else 2 * cfg.H)
    return min(cfg.E * 2 * cfg.I * row, sm_count * 128 * row * 5 // 8, l2_bytes * 5 // 8)


def gemm_flops(cfg) -> float:
    return 2.0 * cfg.T * cfg.k * 3 * cfg.H * cfg.I


def is_decode(cfg) -> bool:
    """Decode-size (HBM-bound) layer: at most 16 token-expert pairs per expert."""
    return cfg.T * cfg.k <= 16 * cfg.E


def hbm_roofline(weight_bytes: int, layer_bytes: int, l2_prefetched: int, kernel_ms: float,
                 step_ms: float, peak_gbs: float) -> dict:
    """HBM roofline of a decode-size layer.  The grouped GEMM's own HBM rate counts the
    weight bytes it pulled from HBM itself, i.e. net of those the router launch had
    already asked L2 for; the whole step counts the layer's algorithmic bytes."""
    achieved = (weight_bytes - l2_prefetched) / (kernel_ms / 1e3) / 1e9
    step = layer_bytes / (step_ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak_gbs, "unit": "GB/s",
            "frac": achieved / peak_gbs, "step_achieved": step, "step_frac": step / peak_gbs}


def tensor_roofline(flops: float, kernel_ms: float, step_ms: float, peak_tflops: float) -> dict:
    achieved = flops / (kernel_ms / 1e3) / 1e12
    step = flops / (step_ms / 1e3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
            "frac": achieved / peak_tflops, "step_achieved": step, "step_frac": step / peak_tflops}


def launches_per_step(cfg, router: bool = True) -> int:
    """Kernels one forward call launches: the fused norm kernel (MXFP8 and pre-norm
    layers), the router (one CUDA-core kernel for T <= 64; else weight split/pack,
    an activation split for the pre-norm layer's fp32 activations (the MXFP8 norm
    kernel writes that split itself), and the tensor-core GEMM), gating (routing
    fused into it when P <= 4096, else histogram + scan + scatter), row expansion,
    grouped GEMM, finalize."""
    P = cfg.T * cfg.k
    routing = 0 if P <= 4096 else 3
    split_kernel = cfg.prenorm and not cfg.mx
    router_k = (1 if cfg.T <= 64 else (3 if split_kernel else 2)) if router else 0
    norm = 1 if (cfg.mx or cfg.prenorm) else 0
    return norm + router_k + 1 + routing + 1 + 1 + 1


def rank_barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max_over_ranks(v: float, world: int, device) -> float:
    """The largest v over all ranks (the slowest rank's time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(T: int, steps: int, world: int, ms_total: float) -> float:
    """Tokens processed by all ranks (each rank runs its own T-token batches) per
    second of the slowest rank's timed region."""
    return T * steps * world / (ms_total / 1e3)


def percentiles(v):
    q = sorted(v)
    at = lambda f: q[min(len(q) - 1, int(round(f * (len(q) - 1))))]
    return {"p10": at(0.1), "p50": at(0.5), "p90": at(0.9), "n": len(q)}


def pipelined_e2e_ms(dev, stream, steps, host_inputs, run, out_like, barrier=lambda: None):
    """Milliseconds for `steps` end-to-end steps as a serving loop runs them: each
    step's inputs go from pinned host memory to the device on one copy stream while
    the previous step computes, and its result comes back on another while the next
    one computes (two input slots and two result buffers; events order each slot's
    reuse).  Every step's H2D and D2H copy is inside the timed region.
    run(device_inputs, slot) launches one step on `stream` and returns its device
    result, shaped like `out_like`."""
    import torch
    dev_in = [[torch.empty_like(h, device=dev) for h in host_inputs] for _ in range(2)]
    host_out = [torch.empty_like(out_like, device="cpu").pin_memory() for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]       # input slot filled
    ev_done = [torch.cuda.Event() for _ in range(2)]     # step done with its slot and result
    ev_back = [torch.cuda.Event() for _ in range(2)]     # result copied back

    def one(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            h2d.wait_event(ev_done[b])                   # step i-2 no longer reads this slot
            for d, h in zip(dev_in[b], host_inputs):
                d.copy_(h, non_blocking=True)
            ev_in[b].record(h2d)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_back[b])                    # step i-2's result is on the host
        o = run(dev_in[b], b)
        ev_done[b].record(stream)
        o.record_stream(d2h)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_done[b])
            host_out[b].copy_(o, non_blocking=True)
            ev_back[b].record(d2h)

    for i in range(3):
        one(i)
    torch.cuda.synchronize(dev)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    e_start.record(stream)
    h2d.wait_event(e_start)
    d2h.wait_event(e_start)
    for i in range(steps):
        one(i)
    for b in range(2):
        stream.wait_event(ev_back[b])                    # the last results are on the host
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    return e_start.elapsed_time(e_end)


# ------------------------------------------------------------ CPU oracle ---


def oracle_sample_tokens(cfg) -> int:
    """Tokens per oracle call in the CPU baseline: the whole batch of a decode
    workload, a slice of consecutive tokens of a prefill batch."""
    return min(cfg.T, ORACLE_SAMPLE_TOKENS)


def host_memory_bytes() -> int:
    try:
        return os.sysconf("SC_PHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        return 0


def oracle_weight_dtype(cfg) -> str:
    """fp64 host copies of the expert weights when they take at most a quarter of
    the host memory, else fp32 (the oracle then widens one expert at a time)."""
    fp64_bytes = cfg.E * 3 * cfg.H * cfg.I * 8
    return "float64" if 4 * fp64_bytes <= host_memory_bytes() else "float32"


def oracle_arrays(inp, cfg):
    """Host copies of the inputs (untimed: the oracle's inputs at rest)."""
    import torch
    wt = torch.float64 if oracle_weight_dtype(cfg) == "float64" else torch.float32
    E = inp["w13"].shape[0]
    arr = {"w13": [inp["w13"][e].cpu().to(wt).numpy() for e in range(E)],
           "down": [inp["down"][e].cpu().to(wt).numpy() for e in range(E)]}
    for key in ("x", "Wg", "r", "norm_w"):
        if key in inp:
            arr[key] = inp[key].double().cpu().numpy()
    return arr


def oracle_step(O, arrays, cfg, rows):
    a = arrays
    if cfg.prenorm or cfg.Z:
        O.moe_forward_v2(a["x"][rows], a["r"][rows] if cfg.prenorm else None, a.get("norm_w"), cfg.eps, a["Wg"],
                         a["w13"], a["down"], cfg.k, num_zero_experts=cfg.Z)
    elif cfg.w4:
        O.moe_forward_w4a8(a["x"][rows], a["r"][rows], a["norm_w"], cfg.eps, a["Wg"], a["w13"], a["down"], cfg.k)
    elif cfg.mx:
        O.moe_forward_mx(a["x"][rows], a["r"][rows], a["norm_w"], cfg.eps, a["Wg"], a["w13"], a["down"], cfg.k)
    else:
        O.moe_forward(a["x"][rows], a["Wg"], a["w13"], a["down"], cfg.k, keep_intermediates=False)


def oracle_sample_rows(cfg, i: int):
    """The i-th sample: consecutive tokens of the batch (wrapping around)."""
    n = oracle_sample_tokens(cfg)
    return [(i * n + j) % cfg.T for j in range(n)]


def oracle_sample_text(cfg, calls: int, seconds: float) -> str:
    n = oracle_sample_tokens(cfg)
    what = "the whole batch" if n == cfg.T else f"a slice of {n} consecutive tokens of the {cfg.T}-token batch"
    held = ("pre-widened to fp64" if oracle_weight_dtype(cfg) == "float64"
            else "held in fp32 (widened to fp64 by the oracle, one expert at a time)")
    return (f"{calls} oracle calls of {n} tokens each ({what}) over {seconds:.1f} s; numpy fp64 oracle "
            f"as committed, weights {held} in host memory")


def time_oracle(O, arrays, cfg, target_s):
    """Tokens/s of the oracle on consecutive token samples until ~target_s of CPU time."""
    oracle_step(O, arrays, cfg, oracle_sample_rows(cfg, 0))   # first touch of the arrays, untimed
    calls = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < target_s or calls == 0:
        oracle_step(O, arrays, cfg, oracle_sample_rows(cfg, calls + 1))
        calls += 1
    dt = time.perf_counter() - t0
    return calls * oracle_sample_tokens(cfg) / dt, calls, dt


def run_reference(args, cfg):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    from oracle import moe_oracle as O
    from top_routing_grouped_gating_gb300 import workloads as W

    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"   # same values as the GPU arm
    inp = W.make_inputs(cfg, device=gen_dev)
    arrays = oracle_arrays(inp, cfg)
    del inp
    if gen_dev == "cuda":
        torch.cuda.empty_cache()
    for i in range(args.warmup):
        oracle_step(O, arrays, cfg, oracle_sample_rows(cfg, i))
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_step(O, arrays, cfg, oracle_sample_rows(cfg, args.warmup + i))
    dt = time.perf_counter() - t0
    value = oracle_sample_tokens(cfg) * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(cfg),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": oracle_sample_text(cfg, args.steps, dt)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(cfg):
    extra = {}
    if cfg.Z:
        extra["zero_computation_experts"] = cfg.Z
    if cfg.prenorm:
        extra["fused_add_rmsnorm_cast"] = True
    if cfg.mx:
        extra["fused_add_rmsnorm_mxquant"] = True
    return {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I, **extra,
            "router": cfg.router, "seed": cfg.seed, "parallelism": "replicas (token batches), no collective",
            "l2": "inputs larger than L2: the active experts' weights streamed per step exceed the 129 MB L2"}


# ------------------------------------------------------------------- ours ---


def make_layer(moe, cfg, inp):
    """The layer object and a step(x, r, slot) closure over two output buffer sets."""
    import torch
    x = inp["x"]
    if cfg.mx:
        cls = moe.MoELayerW4A8 if cfg.w4 else moe.MoELayerMX
        layer = cls(inp["Wg"], inp["w13"], inp["down"], inp["norm_w"], cfg.k, cfg.eps)
        out, res, ids, w = layer(x, inp["r"])
        bufs = dict(out=out, residual_out=res, topk_ids=ids, topk_w=w)
    elif cfg.prenorm or cfg.Z:
        layer = moe.MoELayerV2(inp["Wg"], inp["w13"], inp["down"], cfg.k, Z=cfg.Z,
                               norm_w=inp["norm_w"] if cfg.prenorm else None, eps=cfg.eps)
        out, res, ids, w = layer(x, inp["r"] if cfg.prenorm else None)
        bufs = dict(out=out, residual_out=res, topk_ids=ids, topk_w=w)
    else:
        layer = moe.MoELayer(inp["Wg"], inp["w13"], inp["down"], cfg.k)
        out, ids, w = layer(x)
        bufs = dict(out=out, topk_ids=ids, topk_w=w)
    # a second set of output buffers for the double-buffered end-to-end loop
    bufsets = [bufs, {key: (torch.empty_like(v) if v is not None else None) for key, v in bufs.items()}]
    has_r = cfg.mx or cfg.prenorm

    def step(xx, rr=None, bi=0):
        if has_r:
            return layer(xx, rr, **bufsets[bi])[0]
        return layer(xx, **bufsets[bi])[0]
    return layer, step, bufsets, ids


def measure(args, cfg, dev, cpu_baseline: bool):
    """One workload: warm-up, the headline timed region, the instrumented pass, the
    end-to-end pass (and the CPU baseline when asked).  Returns rank 0's JSON line
    (None on other ranks)."""
    import torch
    import top_routing_grouped_gating_gb300 as moe
    from top_routing_grouped_gating_gb300 import workloads as W

    ws, rank, local = dist_env()
    inp = W.make_inputs(cfg, device=f"cuda:{local}")
    x = inp["x"]
    r = inp.get("r") if (cfg.mx or cfg.prenorm) else None
    stream = torch.cuda.current_stream(dev)
    layer, step, bufsets, ids = make_layer(moe, cfg, inp)
    torch.cuda.synchronize(dev)
    counts = torch.bincount(ids.flatten().long(), minlength=cfg.E + cfg.Z)[:cfg.E]
    active = int((counts > 0).sum())
    routed_pairs = int(counts.sum())
    host_w = None
    if cpu_baseline and rank == 0:
        host_w = {k_: v.cpu() for k_, v in inp.items()}   # bf16/fp32 host copies, widened later
    # the packed copies are all the layer uses; drop the logical weights
    del inp["w13"], inp["down"]
    torch.cuda.empty_cache()

    def barrier():
        rank_barrier(ws)

    def max_over_ranks(v: float) -> float:
        return reduce_max_over_ranks(v, ws, dev)

    K = args.steps
    # ---- warm-up
    for _ in range(max(args.warmup, 3)):
        step(x, r)
    torch.cuda.synchronize(dev)

    # ---- headline timed region: events only at its two ends
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for _ in range(K):
        step(x, r)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end))

    # ---- instrumented pass: events around every step and every grouped-GEMM launch
    n_inst = max(K, 8)
    gb = [torch.cuda.Event(enable_timing=True) for _ in range(n_inst)]
    ge = [torch.cuda.Event(enable_timing=True) for _ in range(n_inst)]
    sb = [torch.cuda.Event(enable_timing=True) for _ in range(n_inst)]
    se = [torch.cuda.Event(enable_timing=True) for _ in range(n_inst)]
    torch.cuda.synchronize(dev)
    for i in range(n_inst):
        # torch only reports elapsed_time for events it recorded itself; record
        # both here first, the library then re-records them around the GEMM
        gb[i].record(stream)
        ge[i].record(stream)
        moe.set_gemm_events(gb[i], ge[i])
        sb[i].record(stream)
        step(x, r)
        se[i].record(stream)
    moe.set_gemm_events(None, None)
    torch.cuda.synchronize(dev)
    gemm_samples = [gb[i].elapsed_time(ge[i]) for i in range(n_inst)]
    step_samples = [sb[i].elapsed_time(se[i]) for i in range(n_inst)]
    gemm_ms = statistics.mean(gemm_samples)
    status = moe.get_device_status(dev)

    # ---- end-to-end: pinned host input -> device -> layer -> pinned host output,
    # the copies of neighbouring steps overlapping the layer calls
    has_r = r is not None
    host_in = [x.cpu().pin_memory()] + ([r.cpu().pin_memory()] if has_r else [])
    e2e_ms = max_over_ranks(pipelined_e2e_ms(
        dev, stream, K, host_in,
        lambda d, b: step(d[0], d[1] if has_r else None, bi=b), bufsets[0]["out"], barrier))

    if rank != 0:
        del layer, bufsets
        torch.cuda.empty_cache()
        return None

    hbm, bf16, peak_kind = measured_peaks()
    value = whole_job_tokens_per_s(cfg.T, K, ws, ms_total)
    step_ms = ms_total / K
    wbytes = gemm_weight_bytes(cfg, active)
    lbytes = layer_algorithmic_bytes(cfg, active)
    if is_decode(cfg):
        props = torch.cuda.get_device_properties(dev)
        l2pf = l2_hint_bytes(cfg, props.multi_processor_count, getattr(props, "L2_cache_size", 0))
        roof = hbm_roofline(wbytes, lbytes, l2pf, gemm_ms, step_ms, hbm)
        roof["peak_source"] = (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                               else "fallback 6.8 TB/s")
        roof["l2_prefetched_bytes"] = l2pf
        roof["note"] = ("frac: the grouped GEMM's weight bytes net of those the router launch asked L2 "
                        "for, over its mean launch time; step_frac: the layer's algorithmic bytes over "
                        "the headline step time")
    else:
        peak = bf16 * 2.0 if cfg.mx else bf16   # e2m1/e4m3 run in kind::mxf8f6f4 at the fp8 rate
        roof = tensor_roofline(gemm_flops(cfg), gemm_ms, step_ms, peak)
        src = "bf16_tflops x 2 (nominal MXFP8/bf16 ratio)" if cfg.mx else "bf16_tflops"
        roof["peak_source"] = (f"{peak_kind} (MEASURED_PEAKS.json {src})" if peak_kind == "measured"
                               else "fallback 1.9 PFLOP/s" + (" x 2" if cfg.mx else ""))
        roof["note"] = ("frac: the grouped GEMMs' 2*P*3*H*I FLOPs over the GEMM launch's mean time; "
                        "step_frac: the same FLOPs over the headline step time")
        sus = sustained_bf16_peak()
        if sus and peak_kind == "measured":
            # the timed loop runs long enough for the power cap to lower the clock: the
            # same achieved rate against the sustained measurement, reported beside frac
            roof["peak_sustained"] = sus * 2.0 if cfg.mx else sus
            roof["frac_sustained"] = roof["achieved"] / roof["peak_sustained"]
    roof.update({"traffic": profiled_traffic(cfg.name),
                 "kernel": "grouped_gemm_mx_kernel" if cfg.mx else
                           ("grouped_gemm_kernel" if is_decode(cfg) else "grouped_gemm_pair_kernel")
                           + " (both projections, one launch)",
                 "kernel_ms": gemm_ms, "kernel_ms_pct": percentiles(gemm_samples),
                 "algorithmic_bytes": lbytes, "gemm_weight_bytes": wbytes,
                 "implementation_bytes": gemm_implementation_bytes(cfg, routed_pairs),
                 "active_experts": active})

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms,
        "step_ms_pct": {**percentiles(step_samples),
                        "note": "single steps bracketed by events, in a separate pass after the timed region"},
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("w4a8 (weights e2m1 + e8m0/32, activations e4m3 + e8m0/32)" if cfg.w4
                                       else "mxfp8 (e4m3 + e8m0/32)" if cfg.mx else "bf16"), "data": "synthetic",
        "config": workload_config(cfg), "roofline": roof,
        "e2e": {"value": whole_job_tokens_per_s(cfg.T, K, ws, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": cfg.T * cfg.H * 2 * (2 if has_r else 1),
                "d2h_bytes_per_step": cfg.T * cfg.H * 2,
                "copies": "pinned host buffers; each step's H2D and D2H run on two copy streams "
                          "(double-buffered), overlapping the neighbouring steps' layer calls"},
        "gpu_launches": launches_per_step(cfg) * K,
        "clocks": clocks,
        "device_status": status,
    }
    del layer, bufsets
    torch.cuda.empty_cache()

    if host_w is not None:
        from oracle import moe_oracle as O
        arrays = oracle_arrays(host_w, cfg)
        del host_w
        v_cpu, calls, dt = time_oracle(O, arrays, cfg, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v_cpu, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                                "sample": oracle_sample_text(cfg, calls, dt)}
    return line


def summary(line: dict) -> dict:
    """The compact per-workload record carried by the headline line."""
    roof = line["roofline"]
    return {"value": line["value"], "unit": line["unit"], "ms_per_step": line["ms_per_step"],
            "bound": roof["bound"], "frac": roof["frac"], "step_frac": roof["step_frac"],
            "kernel_ms": roof["kernel_ms"], "e2e": line["e2e"]["value"], "dtype": line["dtype"],
            "clocks": line["clocks"], "device_status": line["device_status"]}


def run_ours(args, names):
    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from top_routing_grouped_gating_gb300 import build as B
    B.build()
    from top_routing_grouped_gating_gb300 import workloads as W

    lines = {}
    for name in names:
        cfg = W.CONFIGS[name]
        # the oracle baseline is timed for the printed workload only
        line = measure(args, cfg, dev, cpu_baseline=(not args.no_cpu_baseline and name == names[-1]))
        if line is not None:
            lines[name] = line
            if len(names) > 1:
                print(json.dumps(line), file=sys.stderr, flush=True)
    if rank == 0:
        head = dict(lines[names[-1]])
        if len(names) > 1:
            head["workloads"] = {n: summary(l) for n, l in lines.items()}
            head["gpu_launches_all_workloads"] = sum(l["gpu_launches"] for l in lines.values())
        print(json.dumps(head), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_ep_routing(args, cfg):
    """One expert-parallel rank's routing at a prefill size: init_routing_v2 keeps the
    pairs of this rank's experts (the first E/ep_ranks) and gathers their rows, then
    re_routing reorders those rows from (source rank, expert) blocks -- the token
    slices of the ep_ranks ranks -- into expert-major order.  HBM-bound: the
    algorithmic bytes are the gathered rows written and the re-routed rows read and
    written (2 bytes per element)."""
    import numpy as np
    import torch
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    if args.impl == "reference":
        print(json.dumps({"impl": "reference", "unavailable":
                          "the CPU oracle arm covers the layer workloads; this routing-only workload has none"}))
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from top_routing_grouped_gating_gb300 import build as B
    B.build()
    import top_routing_grouped_gating_gb300 as moe
    from top_routing_grouped_gating_gb300 import workloads as W
    inp = W.make_inputs(cfg, device=f"cuda:{local}", weights=False)
    x = inp["x"]
    ids, _ = moe.gating_topk_softmax(moe.router_logits(x, inp["Wg"]), cfg.k)
    El = cfg.E // cfg.ep_ranks
    R = cfg.ep_ranks
    ids_h = ids.cpu().numpy()
    blocks = np.array_split(np.arange(cfg.T), R)
    cnt = np.stack([np.bincount(ids_h[b].reshape(-1)[ids_h[b].reshape(-1) < El], minlength=El)
                    for b in blocks]).astype(np.int32)
    cnt_d = torch.from_numpy(cnt).to(dev)
    N = int(cnt.sum())

    def step(xx=x, ii=ids):
        rt = moe.init_routing_v2(ii, cfg.E, 0, El, x=xx)
        return moe.re_routing(cnt_d, rt["expanded_x"][:N], N)[2]

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    s0.record()
    for _ in range(args.steps):
        step()
    s1.record()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = s0.elapsed_time(s1)
    # end to end: this rank's inputs (x and the top-k ids) from pinned host memory,
    # the expert offsets of the re-routed rows back to the host; the copies of
    # neighbouring steps overlap, as in the layer workloads
    stream = torch.cuda.current_stream(dev)
    e2e_ms = pipelined_e2e_ms(dev, stream, args.steps, [x.cpu().pin_memory(), ids.cpu().pin_memory()],
                              lambda d, b: step(d[0], d[1]), step())
    hbm, _, kind = measured_peaks()
    nbytes = 3 * N * cfg.H * 2
    achieved = nbytes * args.steps / (ms / 1e3) / 1e9
    line = {"metric": "expert-parallel rank routing tokens/s (init_routing_v2 + re_routing)",
            "value": cfg.T * args.steps / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 rows, int32 ids", "data": "synthetic",
            "config": dict(workload_config(cfg), ep_ranks=R, local_experts=El, local_pairs=N),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "peak_source": kind, "traffic": None, "algorithmic_bytes": nbytes,
                         "kernel": "routing + gather + re-routing, whole step"},
            "e2e": {"value": cfg.T * args.steps / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": x.numel() * 2 + ids.numel() * 4, "d2h_bytes_per_step": (El + 1) * 4,
                    "copies": "pinned host buffers; each step's H2D and D2H run on two copy streams "
                              "(double-buffered), overlapping the neighbouring steps"},
            "gpu_launches": 6 * args.steps, "clocks": clocks}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    from top_routing_grouped_gating_gb300 import workloads as W
    names = list(SUITE) if args.workload == "all" else [args.workload]
    for n in names:
        if n not in W.CONFIGS:
            raise SystemExit(f"unknown workload {n}; 'all' or one of {sorted(W.CONFIGS)}")
    if args.shape:
        if len(names) != 1:
            raise SystemExit("--shape applies to a single --workload")
        base = W.CONFIGS[names[0]]
        cfg = W.with_shape(base, name=base.name + "@" + args.shape.replace(",", "_"),
                           **parse_shape(args.shape))
        W.CONFIGS = {**W.CONFIGS, cfg.name: cfg}
        names = [cfg.name]
    if len(names) == 1 and W.CONFIGS[names[0]].ep_ranks:
        return run_ep_routing(args, W.CONFIGS[names[0]])
    if args.impl == "reference":
        # the oracle on the printed (headline) workload
        return run_reference(args, W.CONFIGS[names[-1]])
    return run_ours(args, names)


if __name__ == "__main__":
    sys.exit(main())
