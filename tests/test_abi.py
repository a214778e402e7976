"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, exports
every symbol the public header declares, and rejects bad arguments on the host
before touching a device."""
import ctypes
import re

import pytest

from top_routing_grouped_gating_gb300 import _binding as B
from top_routing_grouped_gating_gb300 import build as BLD

HEADER = BLD.INCLUDE + "/moe_gb300.h"


def header_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    BLD.build()
    return B.lib()


def test_header_declares_the_operator_set():
    names = header_functions()
    for required in ["moe_gating_topk_softmax", "moe_init_routing", "moe_compute_expert_tokens",
                     "moe_grouped_matmul_swiglu", "moe_grouped_matmul", "moe_finalize_routing",
                     "moe_forward"]:
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name
    # and the binding knows each of them (no undeclared extras either)
    assert set(header_functions()) == set(B.exported_symbols())


def test_status_strings(L):
    assert L.moe_abi_version() >= 1
    for s in range(6):
        assert L.moe_status_string(s)
    assert b"unknown" in L.moe_status_string(99)


def test_workspace_queries_are_host_only(L):
    small = L.moe_forward_workspace_size(16, 256, 8, 2, 128)
    big = L.moe_forward_workspace_size(4096, 2048, 128, 8, 768)
    assert 0 < small < big
    # expanded_x + h + y2 dominate at prefill sizes: P*(H + I + H)*2 bytes
    P = 4096 * 8
    assert big >= P * (2048 + 768 + 2048) * 2
    assert L.moe_forward_workspace_size(16, 200, 8, 2, 128) == 0      # H % 128 != 0
    assert L.moe_forward_workspace_size(16, 256, 300, 2, 128) == 0    # E > 256
    assert L.moe_packed_weight_bytes(8, 256, 128, 0) == 8 * 256 * 256 * 2
    assert L.moe_packed_weight_bytes(8, 256, 128, 1) == 8 * 128 * 256 * 2


def test_null_pointers_rejected_before_device_use(L):
    # MOE_ERR_INVALID_ARG == 1, returned by host validation (no GPU here)
    assert L.moe_forward(None, None, None, None, None, 16, 256, 8, 2, 128, None, None, None, None, 0,
                         None) == 1
    assert L.moe_gating_topk_softmax(None, 4, 8, 2, 1, None, None, None) == 1
    assert L.moe_finalize_routing(None, None, None, 4, 2, 256, None, None) == 1
    assert L.moe_get_device_status(None, None) == 1
    assert L.moe_grouped_matmul(None, None, None, 8, 16, 256, 256, None, None, 0, None) == 1


def test_misaligned_pointer_rejected(L):
    # a fake, misaligned "device" address never reaches the device: validation stops it
    bad = ctypes.c_void_p(0x1003)
    assert L.moe_grouped_matmul_swiglu(bad, bad, bad, 8, 16, 256, 128, bad, None, 0, None) == 1


def test_unsupported_arch_without_gpu(L):
    # With no usable sm_103 device the first device query fails cleanly
    st = L.moe_clear_device_status(None)
    assert st in (3, 5)


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        B.gating_topk_softmax(torch.zeros(2, 4), 2)


def test_out_of_range_shapes_rejected_before_device_use(L):
    """Empty and out-of-range shapes fail host validation (MOE_ERR_UNSUPPORTED_SHAPE = 2)
    with fake, aligned pointers that are never dereferenced."""
    f = ctypes.c_void_p(0x10000)
    for T, H, E, k, I in [(0, 256, 8, 2, 128),      # no tokens
                          (16, 256, 8, 9, 128),     # k > E
                          (16, 256, 300, 2, 128),   # E > 256
                          (16, 256, 64, 33, 128),   # k > 32
                          (16, 200, 8, 2, 128)]:    # H % 128 != 0
        assert L.moe_forward(f, f, None, f, f, T, H, E, k, I, f, None, None, f, 1 << 30, None) == 2
        assert L.moe_forward_workspace_size(T, H, E, k, I) == 0
        assert L.moe_forward_mx_workspace_size(T, H, E, k, I) == 0
        assert L.moe_forward_w4a8_workspace_size(T, H, E, k, I) == 0
    assert L.moe_grouped_matmul_mx_workspace_size(8, 0, 256, 128, 1) == 0     # no rows
    assert L.moe_grouped_matmul_mx_workspace_size(300, 16, 256, 128, 1) == 0  # E > 256
    assert L.moe_grouped_matmul_mx_workspace_size(8, 16, 200, 128, 0) == 0    # K % 128 != 0
    assert L.moe_packed_weight_bytes_mx4(8, 256, 128, 0) == 8 * 256 * 128     # 2I x H codes / 2


def test_pair_light_hook_validates_on_the_host(L):
    # host-only: sets the hook state, touches no device
    assert L.moe_debug_set_pair_light(3) == 1                   # not a mode
    assert L.moe_debug_set_pair_light(-1) == 1
    assert L.moe_debug_set_pair_light(2) == 0
    assert L.moe_debug_set_pair_light(0) == 0                   # automatic, the default


def test_gemm_stall_hook_validates_on_the_host(L):
    # host-only: sets or clears the hook state, touches no device
    assert L.moe_debug_set_gemm_stall(3, 10) == 1               # wait limit below 1 us
    assert L.moe_debug_set_gemm_stall(3, 3_000_000_000) == 1    # above the 2 s library limit
    assert L.moe_debug_set_gemm_stall(-1, 0) == 0               # off
