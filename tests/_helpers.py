"""Test helpers: tensor conversion, tolerance checks, lazy per-expert weight access."""
import os
import threading

import numpy as np
import pytest
import torch

# Output tolerance of the bf16 layer against the fp64 oracle: relative Frobenius
# error <= 1e-2 and max-abs error <= 3e-2 * max|ref|.  The GPU rounds h, y2 and the
# output to bf16 once each (relative 2^-9 per rounding) and accumulates in fp32, so
# the expected error is a few 1e-3; the bound leaves margin without hiding a wrong
# term (a dropped expert or a swapped gate/up moves the error to O(1)).
REL_FRO = 1e-2
MAX_ABS_FRAC = 3e-2
# MXFP8 layer against the oracle on dequantised inputs.
REL_FRO_MX = 4e-2


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    return t.cpu().numpy()


def rel_fro(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_close_layer(got, ref, rel=REL_FRO, max_abs_frac=MAX_ABS_FRAC, what="output"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    rf = rel_fro(got, ref)
    ma = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    lim = max_abs_frac * float(np.max(np.abs(ref))) if ref.size else 0.0
    assert rf <= rel, f"{what}: relative Frobenius error {rf:.3e} > {rel:.1e}"
    assert ma <= lim, f"{what}: max abs error {ma:.3e} > {lim:.3e}"
    return rf, ma


class LazyExperts:
    """Indexable view of a (E, a, b) torch weight tensor: w[e] -> fp32 numpy array,
    converted one expert at a time (the oracle widens it to fp64).  Safe to index
    from several threads (the oracle's per-expert loop on a thread pool)."""

    def __init__(self, w: torch.Tensor):
        self.w = w
        self._cache = {}
        self._lock = threading.Lock()

    def __len__(self):
        return self.w.shape[0]

    def __getitem__(self, e):
        e = int(e)
        with self._lock:
            v = self._cache.get(e)
            if v is None:
                if len(self._cache) >= 32:
                    self._cache.pop(next(iter(self._cache)))
                v = self._cache[e] = self.w[e].float().cpu().numpy()
            return v


def oracle_threads() -> int:
    """Host threads for the oracle's per-expert loop in the full-size tests."""
    return max(1, min(32, os.cpu_count() or 1))


def expert_coverage(ids: np.ndarray, rows: np.ndarray, E: int):
    """(experts hit by the compared tokens, experts active in the whole batch)."""
    active = np.unique(ids.ravel())
    active = active[active < E]
    hit = np.unique(ids[rows].ravel())
    hit = hit[hit < E]
    return int(hit.size), int(active.size)


@pytest.fixture(scope="session")
def cuda_dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from top_routing_grouped_gating_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    return dev


def routing_margin_ok(logits32: np.ndarray, k: int, tol: np.ndarray) -> np.ndarray:
    """Tokens whose top-k set cannot change under logit perturbations of size tol[t]
    (gap between the k-th and (k+1)-th largest logit exceeds 2*tol, and the slot
    order is not within 2*tol either)."""
    srt = -np.sort(-logits32.astype(np.float64), axis=1)
    gaps = srt[:, :-1] - srt[:, 1:]
    if logits32.shape[1] > k:
        need = gaps[:, :k]
    else:
        need = gaps[:, :k - 1]
    return np.all(need > 2 * tol[:, None], axis=1)


def forced_topk_logits(counts, k: int, seed: int) -> np.ndarray:
    """fp32 router logits (T, E) whose top-k picks give expert e exactly counts[e]
    rows (T = sum(counts) / k; every count at most T, so a token's k picks are
    distinct).  The expert ids, sorted, are dealt out in k column blocks of T, the
    tokens are shuffled, and slot s of a token gets the logit 4 - s; all other
    logits lie near -2."""
    counts = np.asarray(counts, np.int64)
    E = counts.size
    T = int(counts.sum()) // k
    assert T * k == counts.sum() and counts.max() <= T
    rng = np.random.default_rng(seed)
    flat = np.repeat(np.arange(E), counts)
    picks = flat.reshape(k, T).T[rng.permutation(T)]
    lg = (rng.standard_normal((T, E)) * 0.1 - 2.0).astype(np.float32)
    for s in range(k):
        lg[np.arange(T), picks[:, s]] = np.float32(4.0 - s)
    return lg
