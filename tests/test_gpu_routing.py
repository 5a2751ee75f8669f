"""GPU parity of the routing the whole-layer call actually uses, read back bitwise.

qs_moe_ffn picks one of its implementations per call: the cluster decode kernel
(up to 8 tokens), the persistent decode kernel (up to 16 tokens on shapes it
plans for), the tensor-core path (many tokens, bf16 x) or the per-step kernels.
Each records the expert ids and routing weights its own top-k chose, and
qs_read_routing reads them back.  The acceptance (the layer's statement): ids
bit-exact against the oracle's top-k except tokens whose k-th/(k+1)-th logit
margin is below 1e-5; weights within 1e-6 and summing to 1.  The experts are
left zero: routing depends only on x, the router and its bias.
"""
import numpy as np
import pytest
import torch

import oracle
import qs_inputs as qi
from bit_quantized_moe_router_gb300 import qs_moe as qm
from helpers import Layer

pytestmark = pytest.mark.gpu

MARGIN = 1e-5


def _dev(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def _check_calls(shape, L, T, calls, launches, w_tol=1e-6):
    s = qm.make_shape(shape.hidden, shape.n_experts, shape.top_k, shape.expert_ffn, shape.shared_ffn, shape.x_dtype)
    assert qm.qs_moe_ffn_launches(s, T, True) == launches
    x = _dev(L.xb)
    Wr = _dev(L.Wr)
    bias = None if L.bias is None else _dev(L.bias)
    blob = torch.zeros(shape.n_experts * L.stride, dtype=torch.uint8, device="cuda")
    ex = qm.make_experts(blob, L.stride)
    sh = {k: _dev(v) for k, v in L.shared.items()}
    shared = qm.make_shared(sh["gate"], sh["up"], sh["down"], sh["sig"])
    ws = qm.alloc_workspace(s, T)
    out = torch.empty((T, shape.hidden), device="cuda")
    rids, rp, margin, _ = oracle.route(L.xb, L.x_dtype, L.Wr, L.bias, shape.top_k)
    checked = 0
    for c in range(calls):
        qm.qs_moe_ffn(s, x[c * T:(c + 1) * T].contiguous(), Wr, bias, ex, shared, out, T, ws)
        gi, gp = qm.qs_read_routing(s, T, ws)
        assert qm.qs_read_device_status(ws) == qm.QS_OK
        sl = slice(c * T, (c + 1) * T)
        ok = margin[sl] >= MARGIN
        assert np.array_equal(gi[ok], rids[sl][ok]), f"call {c}: expert ids differ from the oracle's top-k"
        assert np.allclose(gp[ok], rp[sl][ok], rtol=0, atol=w_tol), f"call {c}: routing weights"
        assert np.allclose(gp.sum(1), 1.0, atol=1e-6)
        checked += int(ok.sum())
    assert checked > 0


@pytest.mark.parametrize("wl,T,calls,launches", [
    ("decode_35b_a3b", 1, 16, 1),   # one-kernel decode path
    ("decode_35b_a3b", 4, 4, 1),
    ("verify8_zipf", 8, 4, 1),
    ("decode_h4096", 1, 8, 1),
    ("decode_h4096", 4, 2, 1),
    ("decode_35b_a3b", 12, 2, 8),   # past the decode kernels: tensor-core path
    ("decode_35b_a3b", 64, 1, 8),
])
def test_product_routing_bit_exact(wl, T, calls, launches):
    w = qi.WORKLOADS[wl]
    L = Layer(w.shape, w.seed, 0, n_x=T * calls, zipf=w.zipf_bias, expert_subset=[])
    _check_calls(w.shape, L, T, calls, launches)


def test_product_routing_bit_exact_persistent_kernel():
    """16 tokens on 64 experts: beyond the cluster kernel's 8 tokens, inside the persistent one's plan."""
    shape = qi.LayerShape(2048, 64, 8, 512, 512, qi.BF16)
    L = Layer(shape, 311, 0, n_x=32, zipf=1.1, expert_subset=[])
    _check_calls(shape, L, 16, 2, 1)


@pytest.mark.slow
def test_product_routing_bit_exact_prefill_sampled():
    """2048 tokens through the tensor-core router (three exact bf16 planes) and its top-k.  Its fp32
    logits are summed in another order than the decode kernels' (split-K partial tiles), so a
    logit differs from the exact one by up to a few 1e-6 (H = 2048 fp32 additions of terms near
    0.02); a weight moves by at most half its logit's error plus its neighbours': 1e-5."""
    w = qi.WORKLOADS["prefill_2048"]
    L = Layer(w.shape, w.seed, 0, n_x=w.tokens[0], expert_subset=[])
    _check_calls(w.shape, L, w.tokens[0], 1, 8, w_tol=1e-5)
