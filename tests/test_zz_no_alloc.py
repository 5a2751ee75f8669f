"""qs_moe_ffn_noalloc: the layer for callers that cannot allocate device memory.

Such callers (an operator inside a framework that owns every device
allocation, a serving loop under a fixed memory budget) pass only inputs and
outputs; the scratch lives in a fixed array inside the library.  This checks,
through the C ABI, on two calls in a row: the rows are bitwise the rows of the
workspace entry point (the same deterministic kernel on the same inputs), they
match the oracle within the layer's tolerance, and the fixed array's status
word reads QS_OK after each call.  The file is collected last on purpose, and
it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import qs_inputs as qi
from bit_quantized_moe_router_gb300 import qs_moe as qm
from helpers import Layer, assert_close

pytestmark = pytest.mark.gpu


def _dev(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


@pytest.mark.parametrize("T", [1, 4])
def test_noalloc_matches_workspace_entry_point_twice(T):
    shape = qi.LayerShape(2048, 32, 8, 512, 512, qi.BF16)
    L = Layer(shape, 700 + T, 0, n_x=2 * T, zipf=1.1, expert_subset="routed")
    s = qm.make_shape(shape.hidden, shape.n_experts, shape.top_k, shape.expert_ffn, shape.shared_ffn, shape.x_dtype)
    x = _dev(L.xb)
    Wr = _dev(L.Wr)
    bias = _dev(L.bias)
    blob = _dev(L.experts)
    ex = qm.make_experts(blob, L.stride)
    sh = {k: _dev(v) for k, v in L.shared.items()}
    shared = qm.make_shared(sh["gate"], sh["up"], sh["down"], sh["sig"])
    ws = qm.alloc_workspace(s, T)
    oracle_y = L.oracle()["y"]
    for call in range(2):                     # two calls in a row share the library's scratch
        xt = x[call * T:(call + 1) * T].contiguous()
        ref = torch.full((T, shape.hidden), float("nan"), device="cuda")
        got = torch.full((T, shape.hidden), float("nan"), device="cuda")
        qm.qs_moe_ffn(s, xt, Wr, bias, ex, shared, ref, T, ws)
        qm.qs_moe_ffn_noalloc(s, xt, Wr, bias, ex, shared, got, T)
        assert qm.qs_noalloc_read_device_status() == qm.QS_OK
        assert qm.qs_read_device_status(ws) == qm.QS_OK
        g, r = got.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(g))
        assert np.array_equal(g, r), f"noalloc call {call}: not bitwise equal to qs_moe_ffn"
        assert_close(g, oracle_y[call * T:(call + 1) * T], what=f"noalloc call {call} vs oracle")


def test_noalloc_rejects_what_it_cannot_hold():
    s = qm.make_shape(2048, 32, 8, 512, 512, qm.QS_BF16)
    fake = 1 << 40                            # never dereferenced: rejected before any launch
    ex = qm.make_experts(fake, 1032192)
    L = qm.load()
    rc = L.qs_moe_ffn_noalloc(ctypes.byref(s), fake, fake, None, ctypes.byref(ex), None, fake, 64, None)
    assert rc == qm.QS_ERR_UNSUPPORTED        # beyond the persistent kernel's token range
    rc = L.qs_moe_ffn_noalloc(ctypes.byref(s), None, fake, None, ctypes.byref(ex), None, fake, 1, None)
    assert rc == qm.QS_ERR_INVALID
    big = qm.make_shape(8192, 1024, 16, 8192, 0, qm.QS_BF16)   # exchange area beyond the 4 MiB array
    ex_big = qm.make_experts(fake, 84 * 3 * 8192 * 8192 // 256)
    rc = L.qs_moe_ffn_noalloc(ctypes.byref(big), fake, fake, None, ctypes.byref(ex_big), None, fake, 16, None)
    assert rc in (qm.QS_ERR_WORKSPACE, qm.QS_ERR_UNSUPPORTED)
