"""GPU parity of directional steering, y <- y - scale * d * (d . y) per output row.

Definition: QuarkStar (q36) README, "Steering" (the DwarfStar (ds4) page's
"Steering" section uses the same projection).  Two levels:

- qs_steer_rows alone against the oracle's double-precision steering of the
  same fp32 rows.  Both sides start from identical fp32 inputs, so the only
  difference is the kernel's fp32 arithmetic: a length-H dot product (fixed
  summation order) and one fused multiply-add per element.  For N(0,1) rows
  and a unit direction the rounding error of the dot is O(sqrt(H) * 2^-24)
  relative, and each updated element adds at most one rounding of its own, so
  the kernel is held to rel-L2 <= 1e-6 and max-abs <= 1e-5 * max|y|, about ten
  times the error these inputs produce.
- The whole layer followed by steering, against the oracle's layer followed by
  the oracle's steering, at the layer's acceptance (rel-L2 <= 2e-3, max-abs <=
  1e-2 * max|oracle|), on the persistent decode kernel and on the tensor-core
  path.
"""
import numpy as np
import pytest
import torch

import oracle
import qs_inputs as qi
from bit_quantized_moe_router_gb300 import qs_moe as qm
from helpers import Layer, assert_close

pytestmark = pytest.mark.gpu

MARGIN = 1e-5


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def steer_gpu(y, d, scale, n=None):
    out = dev(y.astype(np.float32))
    dd = dev(d)
    qm.qs_steer_rows(out, dd, scale, out.shape[0] if n is None else n)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("H", [4, 12, 256, 1000, 2048, 4096])
@pytest.mark.parametrize("T", [1, 5, 130])
@pytest.mark.parametrize("scale", [1.0, 0.8, -0.5, 2.0])
def test_kernel_against_oracle(H, T, scale):
    y = qi.gen_rows(T, H, seed=H + T)
    d = qi.gen_direction(H, seed=7)
    got = steer_gpu(y, d, scale)
    ref = oracle.steer_rows(y, d, scale)
    assert_close(got, ref, rel=1e-6, maxabs_frac=1e-5 * float(np.max(np.abs(y))) / float(np.max(np.abs(ref))),
                 what=f"H={H} T={T} scale={scale}")


def test_unit_direction_is_removed():
    y = qi.gen_rows(64, 2048, seed=3)
    d = qi.gen_direction(2048, seed=4)
    got = steer_gpu(y, d, 1.0).astype(np.float64)
    along = got @ d.astype(np.float64)
    assert np.max(np.abs(along)) <= 1e-5 * np.max(np.linalg.norm(y, axis=1))


def test_scale_zero_leaves_rows_untouched():
    y = qi.gen_rows(3, 2048, seed=5)
    d = qi.gen_direction(2048, seed=6)
    assert np.array_equal(steer_gpu(y, d, 0.0), y)


def test_rows_beyond_n_tokens_untouched_and_deterministic():
    y = qi.gen_rows(9, 2048, seed=8)
    d = qi.gen_direction(2048, seed=9)
    a = steer_gpu(y, d, 0.8, n=7)
    b = steer_gpu(y, d, 0.8, n=7)
    assert np.array_equal(a[7:], y[7:])
    assert np.array_equal(a, b)
    assert not np.array_equal(a[:7], y[:7])


def _layer_then_steer(L, T, scale, expect_launches):
    s = L.shape
    shape = qm.make_shape(s.hidden, s.n_experts, s.top_k, s.expert_ffn, s.shared_ffn, s.x_dtype)
    assert qm.qs_moe_ffn_launches(shape, T, True) == expect_launches
    x = dev(L.xb[:T])
    blob = dev(L.experts)
    ex = qm.make_experts(blob, L.stride)
    sd = {k: dev(v) for k, v in L.shared.items()}
    sh = qm.make_shared(sd["gate"], sd["up"], sd["down"], sd["sig"])
    d = qi.gen_direction(s.hidden, L.seed, L.copy)
    dd = dev(d)
    ws = qm.alloc_workspace(shape, T)
    out = torch.full((T, s.hidden), float("nan"), device="cuda")
    qm.qs_moe_ffn(shape, x, dev(L.Wr), None if L.bias is None else dev(L.bias), ex, sh, out, T, ws)
    qm.qs_steer_rows(out, dd, scale, T)
    torch.cuda.synchronize()
    assert qm.qs_read_device_status(ws) == qm.QS_OK
    got = out.cpu().numpy()
    ref = L.oracle(x=L.xb[:T], threads=8)
    keep = ref["margin"] >= MARGIN
    want = oracle.steer_rows(ref["y"], d, scale)
    assert keep.any()
    assert_close(got[keep], want[keep], what=f"layer + steering T={T}")


def test_tiny_layer_then_steering():
    L = Layer(qi.WORKLOADS["tiny"].shape, seed=0, n_x=4)
    _layer_then_steer(L, 4, 0.8, 1)


def test_decode_layer_then_steering():
    L = Layer(qi.WORKLOADS["decode_35b_a3b"].shape, seed=1, n_x=2, expert_subset="routed")
    _layer_then_steer(L, 2, 1.0, 1)


def test_tensor_core_path_then_steering():
    shape = qi.LayerShape(2048, 32, 8, 512, 512, qi.BF16)
    L = Layer(shape, seed=21, n_x=40)
    _layer_then_steer(L, 40, -0.5, 8)
