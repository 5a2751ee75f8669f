"""The C-ABI library: it loads, exports every entry point include/qs_moe.h declares,
and rejects invalid arguments on the host before touching a GPU (no device needed)."""
import ctypes
import os
import re

import pytest

from bit_quantized_moe_router_gb300 import qs_moe as qm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(qs_[a-z0-9_]+)\s*\(", src))
    return names


def test_header_declares_the_binding_exports():
    assert declared_functions() == set(qm.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = qm.load()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version_and_status_strings():
    assert qm.qs_abi_version() == 1
    for c in range(6):
        assert qm.status_string(c)
    assert qm.status_string(99) == "unknown status"


def test_workspace_size():
    good = qm.make_shape(2048, 256, 8, 512, 512, qm.QS_BF16)
    assert qm.qs_moe_workspace_bytes(good, 1) > 256
    assert qm.qs_moe_workspace_bytes(good, 2048) > qm.qs_moe_workspace_bytes(good, 1)
    for bad in [qm.make_shape(100, 256, 8, 512, 512, 1), qm.make_shape(2048, 256, 0, 512, 512, 1),
                qm.make_shape(2048, 4, 8, 512, 512, 1), qm.make_shape(2048, 256, 8, 500, 512, 1),
                qm.make_shape(2048, 256, 8, 512, 100, 1), qm.make_shape(2048, 256, 8, 512, 512, 7),
                qm.make_shape(2048, 2000, 8, 512, 512, 1), qm.make_shape(2048, 256, 33, 512, 512, 1)]:
        assert qm.qs_moe_workspace_bytes(bad, 1) == 0
    assert qm.qs_moe_workspace_bytes(good, 0) == 0


def test_invalid_arguments_are_rejected_before_any_launch():
    L = qm.load()
    shape = qm.make_shape(2048, 256, 8, 512, 512, qm.QS_BF16)
    bad_shape = qm.make_shape(2000, 256, 8, 512, 512, qm.QS_BF16)
    fake = 1 << 40                       # never dereferenced: validation fails first
    ex = qm.make_experts(fake, 1032192)
    ex_bad = qm.make_experts(fake, 1000)
    ex_mis = qm.make_experts(fake + 4, 1032192)
    sh = qm.make_shared(fake, fake, fake, fake)
    B = ctypes.byref
    INV, WS = qm.QS_ERR_INVALID, qm.QS_ERR_WORKSPACE
    assert L.qs_moe_ffn(B(bad_shape), fake, fake, None, B(ex), B(sh), fake, 1, fake, 1 << 30, None) == INV
    assert L.qs_moe_ffn(B(shape), None, fake, None, B(ex), B(sh), fake, 1, fake, 1 << 30, None) == INV
    assert L.qs_moe_ffn(B(shape), fake, fake, None, B(ex), B(sh), fake, 0, fake, 1 << 30, None) == INV
    assert L.qs_moe_ffn(B(shape), fake, fake, None, B(ex_bad), B(sh), fake, 1, fake, 1 << 30, None) == INV
    assert L.qs_moe_ffn(B(shape), fake, fake, None, B(ex_mis), B(sh), fake, 1, fake, 1 << 30, None) == INV
    assert L.qs_moe_ffn(B(shape), fake + 2, fake, None, B(ex), B(sh), fake, 1, fake, 1 << 30, None) == INV
    assert L.qs_moe_ffn(B(shape), fake, fake, None, B(ex), B(sh), fake, 1, None, 1 << 30, None) == WS
    assert L.qs_moe_ffn(B(shape), fake, fake, None, B(ex), B(sh), fake, 1, fake, 64, None) == WS
    assert L.qs_moe_ffn(B(shape), fake, fake, None, B(ex), B(sh), fake, 1, fake + 16, 1 << 30, None) == WS
    assert L.qs_route_topk(B(shape), fake, fake, None, 0, fake, fake, fake, 1 << 30, None) == INV
    assert L.qs_route_topk(B(shape), fake, fake, None, 1, None, fake, fake, 1 << 30, None) == INV
    assert L.qs_group_tokens(B(shape), None, 1, fake, fake, fake, None) == INV
    assert L.qs_q2k_gemv_grouped(B(shape), fake, B(ex_bad), fake, fake, 1, fake, None) == INV
    assert L.qs_q2k_down_combine(B(shape), B(ex), None, fake, fake, 1, fake, 0, None) == INV
    assert L.qs_shared_expert_ffn(B(shape), fake, None, 1, fake, 0, fake, 1 << 30, None) == INV
    assert L.qs_q2k_quantize(fake, 4, 100, fake, None) == INV
    assert L.qs_q2k_quantize(fake + 4, 4, 256, fake, None) == INV
    assert L.qs_workspace_init(None, 1024, None) == WS
    assert L.qs_workspace_init(fake + 8, 1024, None) == WS
    assert L.qs_test_wait_timeout(fake, 1024, 0, None) == INV
    assert L.qs_read_device_status(None, None) == WS


def test_steering_arguments_are_checked_before_any_launch():
    L = qm.load()
    fake = 1 << 40
    INV = qm.QS_ERR_INVALID
    assert L.qs_steer_rows(None, fake, 1.0, 1, 2048, None) == INV
    assert L.qs_steer_rows(fake, None, 1.0, 1, 2048, None) == INV
    assert L.qs_steer_rows(fake, fake, 1.0, 0, 2048, None) == INV
    assert L.qs_steer_rows(fake, fake, 1.0, 1, 2046, None) == INV   # hidden not a multiple of 4
    assert L.qs_steer_rows(fake, fake, 1.0, 1, 0, None) == INV
    assert L.qs_steer_rows(fake + 4, fake, 1.0, 1, 2048, None) == INV
    assert L.qs_steer_rows(fake, fake + 8, 1.0, 1, 2048, None) == INV
    # scale 0 is the unsteered path: accepted, and nothing is launched (no device here)
    assert L.qs_steer_rows(fake, fake, 0.0, 1, 2048, None) == qm.QS_OK


def test_q4k_arguments_are_checked_before_any_launch():
    L = qm.load()
    fake = 1 << 40
    B = ctypes.byref
    INV, WS = qm.QS_ERR_INVALID, qm.QS_ERR_WORKSPACE
    shape = qm.make_shape(2048, 256, 8, 512, 512, qm.QS_BF16)
    need = 144 * 3 * 512 * 2048 // 256
    ex = qm.make_q4k_experts(fake, need)
    sh = qm.make_shared(fake, fake, fake, fake)
    assert L.qs_moe_ffn_q4k(B(shape), fake, fake, None, B(qm.make_q4k_experts(fake, need - 16)), B(sh), fake, 1,
                            fake, 1 << 30, None) == INV          # stride below the expert's Q4_K bytes
    assert L.qs_moe_ffn_q4k(B(shape), fake, fake, None, B(qm.make_q4k_experts(fake + 8, need)), B(sh), fake, 1,
                            fake, 1 << 30, None) == INV          # misaligned blocks
    assert L.qs_moe_ffn_q4k(B(shape), None, fake, None, B(ex), B(sh), fake, 1, fake, 1 << 30, None) == INV
    assert L.qs_moe_ffn_q4k(B(shape), fake, fake, None, B(ex), B(sh), fake, 0, fake, 1 << 30, None) == INV
    assert L.qs_moe_ffn_q4k(B(shape), fake, fake, None, B(ex), B(sh), fake, 1, None, 1 << 30, None) == WS
    assert L.qs_moe_ffn_q4k(B(shape), fake, fake, None, B(ex), B(sh), fake, 1, fake, 64, None) == WS
    assert L.qs_q4k_quantize(fake, 4, 100, fake, None) == INV
    assert L.qs_q4k_quantize(fake + 4, 4, 256, fake, None) == INV
    assert L.qs_q4k_quantize(fake, 0, 256, fake, None) == INV


def test_host_buffer_call_checks_before_any_copy():
    L = qm.load()
    fake = 1 << 40
    B = ctypes.byref
    INV, WS = qm.QS_ERR_INVALID, qm.QS_ERR_WORKSPACE
    shape = qm.make_shape(2048, 256, 8, 512, 512, qm.QS_BF16)
    ex = qm.make_experts(fake, 1032192)
    sh = qm.make_shared(fake, fake, fake, fake)
    need = L.qs_moe_host_workspace_bytes(B(shape), 4)
    assert need > L.qs_moe_workspace_bytes(B(shape), 4) + 4 * 2048 * 2 + 4 * 2048 * 4 - 1
    assert L.qs_moe_ffn_host(B(shape), None, fake, None, B(ex), B(sh), fake, 4, fake, need, None) == INV
    assert L.qs_moe_ffn_host(B(shape), fake, fake, None, B(ex), B(sh), None, 4, fake, need, None) == INV
    assert L.qs_moe_ffn_host(B(shape), fake, fake, None, B(ex), B(sh), fake, 0, fake, need, None) == INV
    assert L.qs_moe_ffn_host(B(shape), fake, fake, None, B(ex), B(sh), fake, 4, fake, need - 256, None) == WS
    assert L.qs_moe_ffn_host(B(shape), fake, fake, None, B(ex), B(sh), fake, 4, fake + 16, need, None) == WS
    assert L.qs_moe_ffn_host(B(shape), fake, fake, None, B(ex), B(sh), fake, 4, None, need, None) == WS


def test_binding_refuses_tensors_on_the_wrong_side():
    """The binding passes device addresses only for contiguous CUDA tensors and host addresses
    only for contiguous host tensors; anything else raises before the library is called."""
    import torch
    shape = qm.make_shape(256, 8, 2, 256, 256, qm.QS_F32)
    host = torch.zeros((2, 256), dtype=torch.float32)
    with pytest.raises(ValueError, match="device memory"):
        qm.make_experts(torch.zeros(64512 * 8, dtype=torch.uint8), 64512)
    with pytest.raises(ValueError, match="device memory"):
        qm.make_shared(host, host, host, host)
    with pytest.raises(ValueError, match="device memory"):
        qm.qs_steer_rows(host, torch.zeros(256), 1.0, 2)
    ex = qm.make_experts(1 << 40, 64512)
    with pytest.raises(ValueError, match="device memory"):
        qm.qs_moe_ffn(shape, host, 1 << 40, None, ex, None, 1 << 40, 2, torch.zeros(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError, match="contiguous"):
        qm._hptr(torch.zeros((256, 2)).t())
    assert qm._hptr(host) == host.data_ptr() and qm._dptr(1 << 40) == 1 << 40 and qm._dptr(None) is None


def test_binding_refuses_short_x_or_out():
    """The layer calls check that x and out hold n_tokens rows before the library reads or writes them."""
    import torch
    shape = qm.make_shape(256, 8, 2, 256, 256, qm.QS_BF16)
    ex = qm.make_experts(1 << 40, 64512)
    x_short = torch.zeros((3, 256), dtype=torch.int16)     # 3 rows of bf16 bits
    out_ok = torch.zeros((4, 256), dtype=torch.float32)
    with pytest.raises(ValueError, match="x: 1536 bytes, need 4 rows of 512 bytes"):
        qm.qs_moe_ffn(shape, x_short, 1 << 40, None, ex, None, out_ok, 4, torch.zeros(16, dtype=torch.uint8))
    x_ok = torch.zeros((4, 256), dtype=torch.int16)
    out_short = torch.zeros((4, 255), dtype=torch.float32)
    with pytest.raises(ValueError, match="out: "):
        qm.qs_moe_ffn_host(shape, x_ok, 1 << 40, None, ex, None, out_short, 4, torch.zeros(16, dtype=torch.uint8))
