"""The allocation-free init_routing entry point (moe_init_routing_noalloc).

It serves callers that cannot allocate device scratch (code inside a host
framework that owns all device memory, or a serving loop that must not allocate
after start-up): the same routing as moe_init_routing, with its scratch in a
fixed array inside the library.  Checked here through the C ABI against the
workspace-taking entry point, twice in a row (the shared scratch keeps the
previous call's contents), on the chunked multi-CTA path that uses the scratch
and on the single-CTA path.  Routing is integer work, so the comparison is exact.

This file is named to be collected last.
"""
import ctypes

import pytest
import torch

import top_routing_grouped_gating_gb300 as moe
from top_routing_grouped_gating_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc(ids, E, x):
    T, k = ids.shape
    H = x.shape[1]
    dev = ids.device
    P = T * k
    out = dict(expanded_row_idx=torch.full((P,), -7, dtype=torch.int32, device=dev),
               sorted_row_idx=torch.full((P,), -7, dtype=torch.int32, device=dev),
               expert_offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
               counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
               expanded_x=torch.zeros(P, H, dtype=torch.bfloat16, device=dev))
    st = moe.lib().moe_init_routing_noalloc(
        x.data_ptr(), ids.data_ptr(), T, H, E, k, out["expanded_x"].data_ptr(),
        out["expanded_row_idx"].data_ptr(), out["sorted_row_idx"].data_ptr(),
        out["expert_offsets"].data_ptr(), out["counts"].data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert st == 0, moe.lib().moe_status_string(st)
    return out


@pytest.mark.parametrize("T,E,k,skew", [(1024, 128, 8, 1.2), (8192, 128, 8, None), (40, 64, 8, None)])
def test_noalloc_routing_matches_workspace_entry_point(cuda_dev, T, E, k, skew):
    H = 256
    for call in range(2):
        ids = W.make_topk_ids(T, E, k, seed=100 * call + T, skew=skew).to(cuda_dev)
        x = torch.randn(T, H, generator=torch.Generator().manual_seed(call)).to(torch.bfloat16).to(cuda_dev)
        ref = moe.init_routing(ids, E, x=x)
        got = _noalloc(ids, E, x)
        torch.cuda.synchronize()
        for key in ("expanded_row_idx", "sorted_row_idx", "expert_offsets", "counts"):
            assert torch.equal(got[key], ref[key]), (call, key)
        assert torch.equal(got["expanded_x"].view(torch.int16), ref["expanded_x"].view(torch.int16))
    assert moe.get_device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_dev):
    T, k, E = 65536 // 8 + 1, 8, 128
    p = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    st = moe.lib().moe_init_routing_noalloc(None, p, T, 0, E, k, None, p, p, p, None, None)
    assert st == 2  # MOE_ERR_UNSUPPORTED_SHAPE
