"""qs_moe_ffn_host (x and out in pinned host memory) against qs_moe_ffn on device buffers.

The host-buffer call copies x into its workspace, runs the same layer and copies the
result back, all on the caller's stream, so its rows must be bitwise those of the
device-buffer call on the same inputs, on every implementation the layer picks
(persistent decode kernel, tensor-core path, per-step kernels).
"""
import numpy as np
import pytest
import torch

import qs_inputs as qi
from bit_quantized_moe_router_gb300 import qs_moe as qm
from helpers import Layer

pytestmark = pytest.mark.gpu


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


CASES = {
    "tiny_f32_persistent": (qi.WORKLOADS["tiny"].shape, 4, 1, dict()),
    "decode_persistent": (qi.WORKLOADS["decode_35b_a3b"].shape, 2, 1, dict(expert_subset="routed")),
    "tensor_core_path": (qi.LayerShape(2048, 32, 8, 512, 512, qi.BF16), 40, 8, dict()),
    # fp32 x and more tokens than the persistent kernel plans for: neither one-kernel path
    "per_step_path": (qi.LayerShape(768, 8, 3, 512, 256, qi.F32), 20, 5, dict()),
}


@pytest.mark.parametrize("name", list(CASES))
def test_host_buffers_match_device_buffers(name):
    shape, T, launches, kw = CASES[name]
    L = Layer(shape, seed=5, n_x=T, **kw)
    s = qm.make_shape(shape.hidden, shape.n_experts, shape.top_k, shape.expert_ffn, shape.shared_ffn, shape.x_dtype)
    assert qm.qs_moe_ffn_launches(s, T, True) == launches
    blob = dev(L.experts)
    ex = qm.make_experts(blob, L.stride)
    d = {k: dev(v) for k, v in L.shared.items()}
    sh = qm.make_shared(d["gate"], d["up"], d["down"], d["sig"])
    Wr = dev(L.Wr)
    xb = np.ascontiguousarray(L.xb[:T])
    # device buffers
    ws = qm.alloc_workspace(s, T)
    out = torch.full((T, shape.hidden), float("nan"), device="cuda")
    qm.qs_moe_ffn(s, dev(xb), Wr, None, ex, sh, out, T, ws)
    torch.cuda.synchronize()
    # host buffers (pinned), twice on one workspace
    x_host = torch.from_numpy(xb.view(np.int16) if xb.dtype == np.uint16 else xb).pin_memory()
    out_host = torch.full((T, shape.hidden), float("nan")).pin_memory()
    wsh = qm.alloc_host_workspace(s, T)
    for _ in range(2):
        qm.qs_moe_ffn_host(s, x_host, Wr, None, ex, sh, out_host, T, wsh)
        torch.cuda.synchronize()
        assert np.array_equal(out_host.numpy(), out.cpu().numpy())
    assert qm.qs_read_device_status(wsh) == qm.QS_OK
