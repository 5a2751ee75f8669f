"""Thin ctypes binding of libqs_moe.so (include/qs_moe.h), same entry-point names.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (device memory supplied by PyTorch);
the stream defaults to torch's current stream.  If the library is missing this
module raises -- there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

QS_OK, QS_ERR_INVALID, QS_ERR_CUDA, QS_ERR_TIMEOUT, QS_ERR_UNSUPPORTED, QS_ERR_WORKSPACE = range(6)
QS_F32, QS_BF16 = 0, 1

# the entry points include/qs_moe.h declares
EXPORTS = (
    "qs_status_string", "qs_abi_version", "qs_last_cuda_error", "qs_moe_workspace_bytes", "qs_workspace_init",
    "qs_read_device_status", "qs_route_topk", "qs_group_tokens", "qs_q2k_gemv_grouped", "qs_q2k_down_combine",
    "qs_shared_expert_ffn", "qs_moe_ffn", "qs_moe_ffn_launches", "qs_moe_ffn_q4k_launches", "qs_q2k_quantize",
    "qs_test_wait_timeout",
    "qs_moe_ffn_noalloc", "qs_steer_rows", "qs_moe_ffn_q4k", "qs_q4k_quantize", "qs_moe_host_workspace_bytes",
    "qs_moe_ffn_host", "qs_noalloc_read_device_status", "qs_read_routing", "qs_moe_ffn_cluster",
)


class QsError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class qs_moe_shape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("expert_ffn", ctypes.c_int32), ("shared_ffn", ctypes.c_int32), ("x_dtype", ctypes.c_int32)]


class qs_q2k_experts(ctypes.Structure):
    _fields_ = [("blocks", ctypes.c_void_p), ("expert_stride", ctypes.c_int64)]


class qs_q4k_experts(ctypes.Structure):
    _fields_ = [("blocks", ctypes.c_void_p), ("expert_stride", ctypes.c_int64)]


class qs_shared_expert(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("w_gate_sig", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libqs_moe.so (building it in-tree first if asked and needed)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"CUDA library not built: {_build.LIB} is missing (run the package build)")
    L = ctypes.CDLL(_build.LIB)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    SP = ctypes.POINTER(qs_moe_shape)
    EP = ctypes.POINTER(qs_q2k_experts)
    HP = ctypes.POINTER(qs_shared_expert)
    L.qs_status_string.restype = ctypes.c_char_p
    L.qs_status_string.argtypes = [i32]
    L.qs_abi_version.restype = i32
    L.qs_last_cuda_error.restype = i32
    L.qs_moe_workspace_bytes.restype = sz
    L.qs_moe_workspace_bytes.argtypes = [SP, i32]
    L.qs_workspace_init.argtypes = [P, sz, P]
    L.qs_read_device_status.argtypes = [P, P]
    L.qs_route_topk.argtypes = [SP, P, P, P, i32, P, P, P, sz, P]
    L.qs_group_tokens.argtypes = [SP, P, i32, P, P, P, P]
    L.qs_q2k_gemv_grouped.argtypes = [SP, P, EP, P, P, i32, P, P]
    L.qs_q2k_down_combine.argtypes = [SP, EP, P, P, P, i32, P, i32, P]
    L.qs_shared_expert_ffn.argtypes = [SP, P, HP, i32, P, i32, P, sz, P]
    L.qs_moe_ffn.argtypes = [SP, P, P, P, EP, HP, P, i32, P, sz, P]
    L.qs_moe_ffn_cluster.argtypes = [SP, P, P, P, EP, HP, P, i32, P, sz, P]
    L.qs_moe_ffn_launches.argtypes = [SP, i32, i32]
    L.qs_moe_ffn_q4k_launches.argtypes = [SP, i32, i32]
    L.qs_moe_ffn_noalloc.argtypes = [SP, P, P, P, EP, HP, P, i32, P]
    L.qs_noalloc_read_device_status.restype = i32
    L.qs_read_routing.argtypes = [SP, i32, P, sz, P, P, P]
    L.qs_noalloc_read_device_status.argtypes = [P]
    L.qs_q2k_quantize.argtypes = [P, i64, i64, P, P]
    L.qs_test_wait_timeout.argtypes = [P, sz, i32, P]
    L.qs_steer_rows.argtypes = [P, P, ctypes.c_float, i32, i32, P]
    L.qs_moe_ffn_q4k.argtypes = [SP, P, P, P, ctypes.POINTER(qs_q4k_experts), HP, P, i32, P, sz, P]
    L.qs_q4k_quantize.argtypes = [P, i64, i64, P, P]
    L.qs_moe_host_workspace_bytes.restype = sz
    L.qs_moe_host_workspace_bytes.argtypes = [SP, i32]
    L.qs_moe_ffn_host.argtypes = [SP, P, P, P, EP, HP, P, i32, P, sz, P]
    for name in EXPORTS:
        if name not in ("qs_status_string", "qs_abi_version", "qs_last_cuda_error", "qs_moe_workspace_bytes",
                        "qs_moe_host_workspace_bytes"):
            getattr(L, name).restype = i32
    _lib = L
    return L


def status_string(code: int) -> str:
    return load().qs_status_string(code).decode()


def _dptr(t):
    """Address of a contiguous CUDA tensor; None and raw integer addresses pass through."""
    if t is None or isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"expected a tensor in device memory, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _hptr(t):
    """Address of a contiguous host tensor (pinned, for asynchronous copies)."""
    if t is None or isinstance(t, int):
        return t
    if t.is_cuda:
        raise ValueError("expected a tensor in host memory, got one on the device")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need_rows(t, n_tokens, row_bytes, what):
    """Reject a tensor smaller than n_tokens rows of row_bytes (a raw address is taken as given)."""
    if t is None or isinstance(t, int):
        return
    have = t.numel() * t.element_size()
    if have < n_tokens * row_bytes:
        raise ValueError(f"{what}: {have} bytes, need {n_tokens} rows of {row_bytes} bytes")


def _layer_io(shape, x, out, n_tokens):
    _need_rows(x, n_tokens, shape.hidden * (2 if shape.x_dtype == QS_BF16 else 4), "x")
    _need_rows(out, n_tokens, shape.hidden * 4, "out")


def _check(rc: int, what: str):
    if rc != QS_OK:
        raise QsError(rc, what)


def make_shape(hidden, n_experts, top_k, expert_ffn, shared_ffn, x_dtype) -> qs_moe_shape:
    return qs_moe_shape(hidden, n_experts, top_k, expert_ffn, shared_ffn, x_dtype)


def make_experts(blocks, expert_stride: int) -> qs_q2k_experts:
    return qs_q2k_experts(_dptr(blocks), expert_stride)


def make_q4k_experts(blocks, expert_stride: int) -> qs_q4k_experts:
    return qs_q4k_experts(_dptr(blocks), expert_stride)


def make_shared(w_gate, w_up, w_down, w_gate_sig) -> qs_shared_expert:
    return qs_shared_expert(_dptr(w_gate), _dptr(w_up), _dptr(w_down), _dptr(w_gate_sig))


# ------------------------------------------------------------------ entry points

def qs_abi_version() -> int:
    return load().qs_abi_version()


def qs_last_cuda_error() -> int:
    return load().qs_last_cuda_error()


def qs_moe_workspace_bytes(shape: qs_moe_shape, max_tokens: int) -> int:
    return load().qs_moe_workspace_bytes(ctypes.byref(shape), max_tokens)


def qs_workspace_init(workspace, stream=None):
    _check(load().qs_workspace_init(_dptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "qs_workspace_init")


def qs_read_device_status(workspace, stream=None) -> int:
    return load().qs_read_device_status(_dptr(workspace), _stream(stream))


def qs_route_topk(shape, x, router_w, router_bias, n_tokens, topk_ids, topk_w, workspace, stream=None):
    _check(load().qs_route_topk(ctypes.byref(shape), _dptr(x), _dptr(router_w), _dptr(router_bias), n_tokens,
                                _dptr(topk_ids), _dptr(topk_w), _dptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)), "qs_route_topk")


def qs_group_tokens(shape, topk_ids, n_tokens, counts, offsets, perm, stream=None):
    _check(load().qs_group_tokens(ctypes.byref(shape), _dptr(topk_ids), n_tokens, _dptr(counts), _dptr(offsets),
                                  _dptr(perm), _stream(stream)), "qs_group_tokens")


def qs_q2k_gemv_grouped(shape, x, experts: qs_q2k_experts, offsets, perm, n_tokens, h_out, stream=None):
    _check(load().qs_q2k_gemv_grouped(ctypes.byref(shape), _dptr(x), ctypes.byref(experts), _dptr(offsets),
                                      _dptr(perm), n_tokens, _dptr(h_out), _stream(stream)), "qs_q2k_gemv_grouped")


def qs_q2k_down_combine(shape, experts: qs_q2k_experts, h, topk_ids, topk_w, n_tokens, out, accumulate=False,
                        stream=None):
    _check(load().qs_q2k_down_combine(ctypes.byref(shape), ctypes.byref(experts), _dptr(h), _dptr(topk_ids),
                                      _dptr(topk_w), n_tokens, _dptr(out), int(bool(accumulate)), _stream(stream)),
           "qs_q2k_down_combine")


def qs_shared_expert_ffn(shape, x, shared: qs_shared_expert, n_tokens, out, workspace, accumulate=False,
                         stream=None):
    _check(load().qs_shared_expert_ffn(ctypes.byref(shape), _dptr(x), ctypes.byref(shared), n_tokens, _dptr(out),
                                       int(bool(accumulate)), _dptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)),
           "qs_shared_expert_ffn")


def qs_moe_ffn(shape, x, router_w, router_bias, experts: qs_q2k_experts, shared, out, n_tokens, workspace,
               stream=None):
    _layer_io(shape, x, out, n_tokens)
    _check(load().qs_moe_ffn(ctypes.byref(shape), _dptr(x), _dptr(router_w), _dptr(router_bias),
                             ctypes.byref(experts), None if shared is None else ctypes.byref(shared), _dptr(out),
                             n_tokens, _dptr(workspace), workspace.numel() * workspace.element_size(),
                             _stream(stream)), "qs_moe_ffn")


def qs_moe_ffn_cluster(shape, x, router_w, router_bias, experts: qs_q2k_experts, shared, out, n_tokens, workspace,
                       stream=None):
    """The whole layer through the cluster decode kernel alone (QsError QS_ERR_UNSUPPORTED outside its plan)."""
    _layer_io(shape, x, out, n_tokens)
    _check(load().qs_moe_ffn_cluster(ctypes.byref(shape), _dptr(x), _dptr(router_w), _dptr(router_bias),
                                     ctypes.byref(experts), None if shared is None else ctypes.byref(shared), _dptr(out),
                                     n_tokens, _dptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)), "qs_moe_ffn_cluster")


def qs_moe_ffn_noalloc(shape, x, router_w, router_bias, experts: qs_q2k_experts, shared, out, n_tokens,
                       stream=None):
    """The whole layer with its scratch in a fixed array inside the library (no workspace argument)."""
    _layer_io(shape, x, out, n_tokens)
    _check(load().qs_moe_ffn_noalloc(ctypes.byref(shape), _dptr(x), _dptr(router_w), _dptr(router_bias),
                                     ctypes.byref(experts), None if shared is None else ctypes.byref(shared),
                                     _dptr(out), n_tokens, _stream(stream)), "qs_moe_ffn_noalloc")


def qs_read_routing(shape, n_tokens, workspace, stream=None):
    """(ids int32 [n_tokens, k], weights fp32 [n_tokens, k]) the last qs_moe_ffn call on workspace used."""
    k = shape.top_k
    ids = np.zeros((n_tokens, k), np.int32)
    w = np.zeros((n_tokens, k), np.float32)
    _check(load().qs_read_routing(ctypes.byref(shape), n_tokens, _dptr(workspace),
                                  workspace.numel() * workspace.element_size(), ids.ctypes.data, w.ctypes.data,
                                  _stream(stream)), "qs_read_routing")
    return ids, w


def qs_noalloc_read_device_status(stream=None) -> int:
    """Sticky device status of the qs_moe_ffn_noalloc array on the current device, cleared by the read."""
    return load().qs_noalloc_read_device_status(_stream(stream))


def qs_steer_rows(out, direction, scale, n_tokens, stream=None):
    """In place, per row of out [n_tokens, hidden] fp32: y <- y - scale * direction * (direction . y)."""
    _check(load().qs_steer_rows(_dptr(out), _dptr(direction), float(scale), n_tokens, out.shape[-1],
                                _stream(stream)), "qs_steer_rows")


def qs_moe_ffn_host(shape, x_host, router_w, router_bias, experts: qs_q2k_experts, shared, out_host, n_tokens,
                    workspace, stream=None):
    """The whole layer with x_host and out_host in (pinned) host memory; copies are queued on the stream."""
    _layer_io(shape, x_host, out_host, n_tokens)
    _check(load().qs_moe_ffn_host(ctypes.byref(shape), _hptr(x_host), _dptr(router_w), _dptr(router_bias),
                                  ctypes.byref(experts), None if shared is None else ctypes.byref(shared),
                                  _hptr(out_host), n_tokens, _dptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "qs_moe_ffn_host")


def alloc_host_workspace(shape: qs_moe_shape, max_tokens: int, device="cuda"):
    """A zero-initialised workspace for qs_moe_ffn_host."""
    n = load().qs_moe_host_workspace_bytes(ctypes.byref(shape), max_tokens)
    if n == 0:
        raise QsError(QS_ERR_INVALID, "qs_moe_host_workspace_bytes")
    ws = torch.zeros(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def qs_moe_ffn_launches(shape, n_tokens, has_shared=True) -> int:
    return load().qs_moe_ffn_launches(ctypes.byref(shape), n_tokens, int(bool(has_shared)))


def qs_moe_ffn_q4k_launches(shape, n_tokens, has_shared=True) -> int:
    return load().qs_moe_ffn_q4k_launches(ctypes.byref(shape), n_tokens, int(bool(has_shared)))


def qs_q2k_quantize(w, out, stream=None):
    rows, K = w.shape
    _check(load().qs_q2k_quantize(_dptr(w), rows, K, _dptr(out), _stream(stream)), "qs_q2k_quantize")


def qs_q4k_quantize(w, out, stream=None):
    rows, K = w.shape
    _check(load().qs_q4k_quantize(_dptr(w), rows, K, _dptr(out), _stream(stream)), "qs_q4k_quantize")


def qs_moe_ffn_q4k(shape, x, router_w, router_bias, experts: qs_q4k_experts, shared, out, n_tokens, workspace,
                   stream=None):
    """The whole layer with Q4_K routed experts (same arguments as qs_moe_ffn)."""
    _layer_io(shape, x, out, n_tokens)
    _check(load().qs_moe_ffn_q4k(ctypes.byref(shape), _dptr(x), _dptr(router_w), _dptr(router_bias),
                                 ctypes.byref(experts), None if shared is None else ctypes.byref(shared), _dptr(out),
                                 n_tokens, _dptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)), "qs_moe_ffn_q4k")


def qs_test_wait_timeout(workspace, limit_us, stream=None):
    _check(load().qs_test_wait_timeout(_dptr(workspace), workspace.numel() * workspace.element_size(), limit_us,
                                       _stream(stream)), "qs_test_wait_timeout")


# ------------------------------------------------------------------ conveniences

def alloc_workspace(shape: qs_moe_shape, max_tokens: int, device="cuda"):
    """A zero-initialised workspace tensor (256-byte aligned by the CUDA caching allocator)."""
    n = qs_moe_workspace_bytes(shape, max_tokens)
    if n == 0:
        raise QsError(QS_ERR_INVALID, "qs_moe_workspace_bytes")
    ws = torch.zeros(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws
