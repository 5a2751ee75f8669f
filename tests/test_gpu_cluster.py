"""GPU parity of the cluster decode kernel (qs_moe_ffn_cluster) against the oracle.

The kernel's grid is clusters of 8 CTAs that own whole routed experts and share
h through distributed shared memory.  qs_moe_ffn tries the persistent kernel
first (measured faster), so this entry point is checked on its own: the
layer's float acceptance (rel-L2 <= 2e-3, max-abs <= 1e-2 * max|oracle|),
routing bit-exact outside the 1e-5 margin, bitwise batch invariance and
run-to-run determinism, and the calls outside its plan.
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


def _dev(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


class _Dev:
    def __init__(self, L):
        s = L.shape
        self.L = L
        self.shape = qm.make_shape(s.hidden, s.n_experts, s.top_k, s.expert_ffn,
                                   s.shared_ffn if L.shared is not None else 0, s.x_dtype)
        self.x = _dev(L.xb)
        self.Wr = _dev(L.Wr)
        self.bias = None if L.bias is None else _dev(L.bias)
        self.blob = _dev(L.experts)
        self.ex = qm.make_experts(self.blob, L.stride)
        if L.shared is not None:
            self.sh = {k: _dev(v) for k, v in L.shared.items()}
            self.shared = qm.make_shared(self.sh["gate"], self.sh["up"], self.sh["down"], self.sh["sig"])
        else:
            self.shared = None

    def call(self, t0, n, ws=None):
        ws = qm.alloc_workspace(self.shape, n) if ws is None else ws
        out = torch.full((n, self.L.shape.hidden), float("nan"), device="cuda")
        qm.qs_moe_ffn_cluster(self.shape, self.x[t0:t0 + n].contiguous(), self.Wr, self.bias, self.ex, self.shared,
                              out, n, ws)
        torch.cuda.synchronize()
        assert qm.qs_read_device_status(ws) == qm.QS_OK
        return out.cpu().numpy(), ws


def _check(L, ref, got, tokens, what):
    ok = [i for i, t in enumerate(tokens) if ref["margin"][t] >= MARGIN]
    assert ok, f"{what}: every token within the routing margin"
    assert_close(got[ok], ref["y"][[tokens[i] for i in ok]], what=what)


SHAPES = {
    "tiny": qi.WORKLOADS["tiny"].shape,
    "h2048_f512": qi.LayerShape(2048, 32, 8, 512, 512, qi.BF16),
    "h4096_f2048": qi.LayerShape(4096, 16, 8, 2048, 256, qi.BF16),
    "e1_k1": qi.LayerShape(512, 1, 1, 256, 256, qi.F32),
    "k_eq_e": qi.LayerShape(256, 4, 4, 256, 256, qi.BF16),
}


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("T", [1, 3, 8])
def test_cluster_kernel_parity_small(name, T):
    shape = SHAPES[name]
    if T * shape.top_k > 64:
        pytest.skip("beyond the kernel's 64 entries")
    if name == "h4096_f2048" and T == 8:
        pytest.skip("8 tokens of x, their int16 fragments and two h buffers of 2048 leave too few stages")
    L = Layer(shape, 800 + T, 0, n_x=T)
    D = _Dev(L)
    got, _ = D.call(0, T)
    _check(L, L.oracle(), got, list(range(T)), f"cluster {name} T={T}")


def test_cluster_kernel_without_shared_expert_and_routing_record():
    shape = SHAPES["h2048_f512"]
    L = Layer(shape, 830, 0, n_x=4, shared=False)
    D = _Dev(L)
    got, ws = D.call(0, 4)
    ref = L.oracle()
    _check(L, ref, got, list(range(4)), "cluster, no shared expert")
    ids, w = qm.qs_read_routing(D.shape, 4, ws)
    ok = ref["margin"][:4] >= MARGIN
    assert np.array_equal(ids[ok], ref["ids"][:4][ok])
    assert np.allclose(w[ok], ref["p"][:4][ok], rtol=0, atol=1e-6)


@pytest.mark.slow
@pytest.mark.parametrize("wl,T,calls", [("decode_35b_a3b", 1, 4), ("verify8_zipf", 8, 1), ("decode_h4096", 1, 2)])
def test_cluster_kernel_full_size_sampled(wl, T, calls):
    w = qi.WORKLOADS[wl]
    L = Layer(w.shape, w.seed, 0, n_x=T * calls, zipf=w.zipf_bias, expert_subset="routed")
    D = _Dev(L)
    ref = L.oracle(threads=8)
    for c in range(calls):
        got, _ = D.call(c * T, T)
        _check(L, ref, got, list(range(c * T, (c + 1) * T)), f"cluster {wl} call {c}")


def test_cluster_kernel_batch_equals_single_calls_and_repeats():
    shape = qi.LayerShape(2048, 64, 8, 512, 512, qi.BF16)
    L = Layer(shape, 840, 0, n_x=8, zipf=1.1)
    D = _Dev(L)
    batch, ws = D.call(0, 8)
    again, _ = D.call(0, 8, ws)
    assert np.array_equal(batch, again)
    singles = np.concatenate([D.call(t, 1)[0] for t in range(8)])
    assert np.array_equal(batch, singles)


def test_cluster_kernel_rejects_what_it_does_not_plan():
    shape = SHAPES["h2048_f512"]
    L = Layer(shape, 850, 0, n_x=9, expert_subset=[])
    D = _Dev(L)
    ws = qm.alloc_workspace(D.shape, 9)
    out = torch.zeros((9, shape.hidden), device="cuda")
    with pytest.raises(qm.QsError) as ei:
        qm.qs_moe_ffn_cluster(D.shape, D.x, D.Wr, None, D.ex, D.shared, out, 9, ws)
    assert ei.value.code == qm.QS_ERR_UNSUPPORTED
