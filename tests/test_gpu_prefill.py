"""GPU parity of the tensor-core path of the layer (many tokens per call) against the oracle.

qs_moe_ffn takes this path when the persistent decode kernel does not: more
than 16 tokens, or shapes outside the decode kernel's plan.  It routes with a
three-plane bf16 split of the fp32 router on the tensor cores, runs the experts
as grouped GEMMs with Q2_K weights dequantised to fp16 (bf16 for the shared
expert) and fp32 accumulation, and sums each token's fp16 routed contributions
in slot order.  Acceptance is
the layer's: rel-L2 <= 2e-3 and max-abs <= 1e-2 * max|oracle| over the tokens
whose k-th/(k+1)-th logit margin is at least 1e-5.

The shapes cover each way the kernels stage raw weights: Q2_K rows whose byte
length is a multiple of 16 (column boxes through a 3-D tensor map) and rows that
are not (whole 128-row tiles through one bulk copy), for both the gate/up and
the down matrices, plus bf16 shared-expert tiles.  Token counts cover a ragged
last tile and experts that receive more than one 128-token tile.
"""
import numpy as np
import pytest
import torch

import qs_inputs as qi
from bit_quantized_moe_router_gb300 import qs_moe as qm
from helpers import Layer, assert_close

pytestmark = pytest.mark.gpu

MARGIN = 1e-5

SHAPES = {
    # name: (shape, note)
    "h256_f256": qi.LayerShape(256, 8, 2, 256, 256, qi.BF16),       # gate/up and down as whole tiles
    "h1024_f768": qi.LayerShape(1024, 16, 4, 768, 512, qi.BF16),    # gate/up columns, down tile (252-byte rows)
    "h2048_f512": qi.LayerShape(2048, 32, 8, 512, 512, qi.BF16),    # the 35B-A3B layer's row shapes
    "h4096_f2048": qi.LayerShape(4096, 16, 8, 2048, 2048, qi.BF16),  # columns for both
}


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def run_layer(L, T, shared=True):
    s = L.shape
    shape = qm.make_shape(s.hidden, s.n_experts, s.top_k, s.expert_ffn,
                          s.shared_ffn if (shared and L.shared is not None) else 0, s.x_dtype)
    assert qm.qs_moe_ffn_launches(shape, T, shared and L.shared is not None) == 8, "not the tensor-core path"
    x = dev(L.xb[:T])
    Wr = dev(L.Wr)
    bias = None if L.bias is None else dev(L.bias)
    blob = dev(L.experts)
    ex = qm.make_experts(blob, L.stride)
    sh = None
    if shared and L.shared is not None:
        d = {k: dev(v) for k, v in L.shared.items()}
        sh = qm.make_shared(d["gate"], d["up"], d["down"], d["sig"])
    ws = qm.alloc_workspace(shape, T)
    out = torch.full((T, s.hidden), float("nan"), device="cuda")
    qm.qs_moe_ffn(shape, x, Wr, bias, ex, sh, out, T, ws)
    torch.cuda.synchronize()
    st = qm.qs_read_device_status(ws)
    # on a device-side time-out the header also records which wait gave up, where
    assert st == qm.QS_OK, f"status {st}, header {ws[:32].view(torch.int32).tolist()}"
    return out.cpu().numpy()


def compare(L, got, T, what):
    ref = L.oracle(tokens=list(range(T)), threads=8)
    keep = ref["margin"][:T] >= MARGIN
    assert keep.any()
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert_close(got[keep], ref["y"][:T][keep], what=what)


@pytest.mark.parametrize("name,T", [("h256_f256", 17), ("h256_f256", 300), ("h1024_f768", 40),
                                    ("h1024_f768", 129), ("h2048_f512", 17), ("h2048_f512", 64),
                                    ("h4096_f2048", 24)])
def test_prefill_parity(name, T):
    shape = SHAPES[name]
    L = Layer(shape, 900 + T, 0, n_x=T, expert_subset="routed")
    got = run_layer(L, T)
    compare(L, got, T, f"{name} T={T}")


def test_prefill_skewed_routing_multi_tile_experts():
    """Zipf-biased router over few experts: the favourite experts get several 128-token tiles."""
    shape = qi.LayerShape(1024, 8, 4, 512, 256, qi.BF16)
    T = 200
    L = Layer(shape, 950, 0, n_x=T, zipf=1.1)
    got = run_layer(L, T)
    compare(L, got, T, "skewed")


def test_prefill_without_shared_expert():
    shape = SHAPES["h2048_f512"]
    T = 33
    L = Layer(shape, 960, 0, n_x=T, shared=False, expert_subset="routed")
    got = run_layer(L, T, shared=False)
    compare(L, got, T, "no shared")


def test_prefill_repeated_calls_reuse_workspace():
    """Two calls on one workspace with different x: the second must not see the first's state."""
    shape = SHAPES["h1024_f768"]
    T = 48
    L = Layer(shape, 970, 0, n_x=2 * T, expert_subset="routed")
    s = L.shape
    qshape = qm.make_shape(s.hidden, s.n_experts, s.top_k, s.expert_ffn, s.shared_ffn, s.x_dtype)
    Wr = dev(L.Wr)
    blob = dev(L.experts)
    ex = qm.make_experts(blob, L.stride)
    d = {k: dev(v) for k, v in L.shared.items()}
    sh = qm.make_shared(d["gate"], d["up"], d["down"], d["sig"])
    ws = qm.alloc_workspace(qshape, T)
    ref = L.oracle(tokens=list(range(2 * T)), threads=8)
    for call in range(2):
        x = dev(L.xb[call * T:(call + 1) * T])
        out = torch.full((T, s.hidden), float("nan"), device="cuda")
        qm.qs_moe_ffn(qshape, x, Wr, None, ex, sh, out, T, ws)
        torch.cuda.synchronize()
        assert qm.qs_read_device_status(ws) == qm.QS_OK
        keep = ref["margin"][call * T:(call + 1) * T] >= MARGIN
        assert_close(out.cpu().numpy()[keep], ref["y"][call * T:(call + 1) * T][keep], what=f"call {call}")


def test_prefill_is_deterministic():
    """No floating-point atomics: two calls on the same inputs give the same bits."""
    shape = SHAPES["h2048_f512"]
    T = 150
    L = Layer(shape, 980, 0, n_x=T, expert_subset="routed")
    a = run_layer(L, T)
    b = run_layer(L, T)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
