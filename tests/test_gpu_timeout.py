"""The bounded device waits of the grouped GEMM, run out on purpose and recovered from.

Every wait in the library's kernels (on an mbarrier or on a global counter) is
bounded in wall-clock time; when one runs out the kernel sets MOE_DEV_WAIT_TIMEOUT
in the device status word and its roles unwind without trapping.  Here a test hook
(moe_debug_set_gemm_stall) makes the TMA producer of the decode-size grouped GEMM
stop issuing at a given pipeline stage and bounds every wait of that launch by
2 ms.  Nothing is in flight when the MMA thread's wait for the missing stage runs
out: the copies and MMAs issued before it complete before the CTA frees its TMEM
and exits.  The call must return quickly, report the timeout bit, and leave the
context usable: the next normal call matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

import top_routing_grouped_gating_gb300 as moe
from oracle import moe_oracle as O
from tests._helpers import LazyExperts, assert_close_layer, to_np
from top_routing_grouped_gating_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("stage", [0, 40])
def test_gemm_wait_timeout_reports_and_recovers(cuda_dev, stage):
    cfg = W.CONFIGS["qwen3_30b_a3b_decode"]
    inp = W.make_inputs(cfg, device="cuda")
    layer = moe.MoELayer(inp["Wg"], inp["w13"], inp["down"], cfg.k)
    x = inp["x"]
    moe.clear_device_status()
    layer(x)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    try:
        # stage 0: no stage is ever fed; stage 40: every CTA stalls inside its second
        # unit (a gate/up unit has H / 64 = 32 stages), after MMAs have run
        moe.debug_set_gemm_stall(stage, 2_000_000)
        t0 = time.perf_counter()
        layer(x)
        status = moe.get_device_status()          # synchronises the stream
        dt = time.perf_counter() - t0
    finally:
        moe.debug_set_gemm_stall(-1)
    assert status & moe.DEV_WAIT_TIMEOUT, f"status {status:#x}"
    assert dt < 1.0, f"the launch took {dt:.3f} s: it did not end on the 2 ms limit"
    moe.clear_device_status()
    assert moe.get_device_status() == 0

    # the context is still usable: a normal call matches the oracle
    xn = to_np(x)
    lg32 = O.router_logits_f32(xn, to_np(inp["Wg"]))
    out, ids, w = layer(x, logits_override=torch.from_numpy(lg32).to(x.device))
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    ref = O.moe_forward(xn, None, LazyExperts(inp["w13"]), LazyExperts(inp["down"]), cfg.k,
                        logits32=lg32, keep_intermediates=False)
    np.testing.assert_array_equal(to_np(ids), ref["topk_ids"])
    assert_close_layer(to_np(out), ref["out"], what="after a timed-out launch")
