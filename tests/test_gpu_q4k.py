"""GPU parity of the layer with Q4_K routed experts against the double-precision oracle.

The Q4_K block is read as the GGUF layout the pages keep (QuarkStar (q36) README,
"Acknowledgements"; Q4_K experts in its "Model Weights" section).  The device encoder
takes every decision in fp32 in the oracle encoder's order, so its bytes must be
identical.  The layer (qs_moe_ffn_q4k) routes exactly like the Q2_K layer; expert ids are
bit-exact except tokens whose k-th/(k+1)-th logit margin is below 1e-5, and the output is
held to the layer's acceptance: rel-L2 <= 2e-3 and max-abs <= 1e-2 * max|oracle|.
"""
import numpy as np
import pytest
import torch

import oracle
import qs_inputs as qi
from bit_quantized_moe_router_gb300 import qs_moe as qm
from helpers import assert_close

pytestmark = pytest.mark.gpu

MARGIN = 1e-5


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def q4k_bytes(shape):
    return 144 * 3 * shape.expert_ffn * shape.hidden // 256


ENCODER_CASES = ["gauss", "positive", "negative", "zero_rows", "mixed_scale", "constant"]


@pytest.mark.parametrize("case", ENCODER_CASES)
def test_encoder_bit_exact(case):
    rng = np.random.default_rng(100 + ENCODER_CASES.index(case))
    w = (rng.standard_normal((48, 1024)) * 0.02).astype(np.float32)
    if case == "positive":
        w = np.abs(w)
    elif case == "negative":
        w = -np.abs(w)
    elif case == "zero_rows":
        w[::3] = 0.0
    elif case == "mixed_scale":
        w *= np.exp(rng.uniform(-8, 8, (48, 1))).astype(np.float32)
    elif case == "constant":
        w[:] = np.float32(0.0123)
    out = torch.zeros((48, 1024 // 256 * 144), dtype=torch.uint8, device="cuda")
    qm.qs_q4k_quantize(dev(w), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.q4k_quantize(w))


class Q4Layer:
    def __init__(self, shape, seed, T, shared=True, zipf=0.0, subset_routed=False):
        self.shape, self.T = shape, T
        self.xb, _ = qi.gen_x(shape, seed, T)
        self.Wr = qi.gen_router(shape, seed, 0)
        self.bias = qi.gen_bias(shape, seed, 0, zipf)
        self.shared = qi.gen_shared(shape, seed, 0) if shared and shape.shared_ffn > 0 else None
        x_dtype = oracle.X_BF16 if shape.x_dtype == qi.BF16 else oracle.X_F32
        if subset_routed:
            ids, _, _, _ = oracle.route(self.xb, x_dtype, self.Wr, self.bias, shape.top_k)
            todo = sorted(set(int(e) for e in np.unique(ids)))
        else:
            todo = range(shape.n_experts)
        self.stride = q4k_bytes(shape)
        self.experts = np.zeros(shape.n_experts * self.stride, np.uint8)
        for e in todo:
            self.experts[e * self.stride:(e + 1) * self.stride] = oracle.quantize_expert(
                *qi.gen_expert_f32(shape, seed, 0, e), fmt="q4k")

    def run_gpu(self):
        s = self.shape
        S = s.shared_ffn if self.shared is not None else 0
        shape = qm.make_shape(s.hidden, s.n_experts, s.top_k, s.expert_ffn, S, s.x_dtype)
        blob = dev(self.experts)
        ex = qm.make_q4k_experts(blob, self.stride)
        sh = None
        if self.shared is not None:
            d = {k: dev(v) for k, v in self.shared.items()}
            sh = qm.make_shared(d["gate"], d["up"], d["down"], d["sig"])
        ws = qm.alloc_workspace(shape, self.T)
        out = torch.full((self.T, s.hidden), float("nan"), device="cuda")
        qm.qs_moe_ffn_q4k(shape, dev(self.xb), dev(self.Wr), None if self.bias is None else dev(self.bias), ex, sh,
                          out, self.T, ws)
        torch.cuda.synchronize()
        assert qm.qs_read_device_status(ws) == qm.QS_OK
        return out.cpu().numpy()

    def run_oracle(self):
        return oracle.moe_ffn(self.shape, self.xb, self.Wr, self.bias, self.experts, self.stride, self.shared,
                              threads=8, fmt="q4k")


SHAPES = {
    "tiny_f32": (qi.LayerShape(256, 8, 2, 256, 256, qi.F32), 4, dict()),
    "tiny_ragged": (qi.LayerShape(256, 8, 2, 256, 256, qi.F32), 13, dict()),
    "h512_no_shared": (qi.LayerShape(512, 16, 4, 256, 256, qi.BF16), 7, dict(shared=False)),
    "h768_three_blocks": (qi.LayerShape(768, 8, 3, 512, 256, qi.BF16), 5, dict()),
    "k_equals_E": (qi.LayerShape(256, 4, 4, 256, 0, qi.F32), 3, dict()),
    "e1_k1": (qi.LayerShape(512, 1, 1, 256, 256, qi.BF16), 2, dict()),
    "decode_35b_t1": (qi.LayerShape(2048, 256, 8, 512, 512, qi.BF16), 1, dict(subset_routed=True)),
    "decode_35b_t4_zipf": (qi.LayerShape(2048, 256, 8, 512, 512, qi.BF16), 4, dict(subset_routed=True, zipf=1.1)),
    "h4096_f2048": (qi.LayerShape(4096, 16, 8, 2048, 2048, qi.BF16), 2, dict()),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_layer_against_oracle(name):
    shape, T, kw = SHAPES[name]
    L = Q4Layer(shape, seed=31 + len(name), T=T, **kw)
    got = L.run_gpu()
    ref = L.run_oracle()
    keep = ref["margin"] >= MARGIN
    assert keep.any()
    assert np.all(np.isfinite(got))
    assert_close(got[keep], ref["y"][keep], what=name)


def test_run_to_run_bitwise():
    shape = qi.LayerShape(2048, 32, 8, 512, 512, qi.BF16)
    L = Q4Layer(shape, seed=77, T=6)
    a = L.run_gpu()
    b = L.run_gpu()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("T,launches", [(1, 1), (4, 1), (20, 6)])
def test_layer_paths(T, launches):
    """The persistent decode kernel takes the call where it plans it (one launch), the per-step
    kernels the rest; both against the oracle."""
    shape = qi.LayerShape(1024, 64, 8, 512, 512, qi.BF16)
    s = qm.make_shape(shape.hidden, shape.n_experts, shape.top_k, shape.expert_ffn, shape.shared_ffn, shape.x_dtype)
    assert qm.qs_moe_ffn_q4k_launches(s, T, True) == launches
    L = Q4Layer(shape, seed=90 + T, T=T)
    got = L.run_gpu()
    ref = L.run_oracle()
    keep = ref["margin"] >= MARGIN
    assert keep.any()
    assert_close(got[keep], ref["y"][keep], what=f"Q4_K layer, {T} tokens, {launches} launch(es)")


def test_one_kernel_batch_equals_single_calls():
    """One call of 4 tokens on the persistent kernel gives each token the bits of its own call."""
    shape = qi.LayerShape(2048, 32, 8, 512, 512, qi.BF16)
    L = Q4Layer(shape, seed=55, T=4)
    s = qm.make_shape(shape.hidden, shape.n_experts, shape.top_k, shape.expert_ffn, shape.shared_ffn, shape.x_dtype)
    assert qm.qs_moe_ffn_q4k_launches(s, 4, True) == 1 and qm.qs_moe_ffn_q4k_launches(s, 1, True) == 1
    batch = L.run_gpu()
    xb = L.xb
    singles = []
    for t in range(4):
        L.xb, L.T = xb[t:t + 1], 1
        singles.append(L.run_gpu())
    L.xb, L.T = xb, 4
    assert np.array_equal(batch, np.concatenate(singles))
