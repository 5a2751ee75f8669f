"""GPU parity: every entry point of the C ABI against the double-precision oracle.

Acceptance (the layer's statement): expert ids and the grouping permutation are
bit-exact, except tokens whose k-th/(k+1)-th logit margin is below 1e-5; the
Q2_K encoder is bit-exact; floating outputs reach rel-L2 <= 2e-3 and
max-abs <= 1e-2 * max|oracle|.  Routing weights are fp32 softmax values and
are held to 1e-6 absolute.
"""
import numpy as np
import pytest
import torch

import oracle
import qs_inputs as qi
from bit_quantized_moe_router_gb300 import qs_moe as qm
from helpers import Layer, assert_close, build_experts

pytestmark = pytest.mark.gpu

MARGIN = 1e-5


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


class DevLayer:
    def __init__(self, L: Layer):
        s = L.shape
        self.L = L
        self.shape = qm.make_shape(s.hidden, s.n_experts, s.top_k, s.expert_ffn,
                                   s.shared_ffn if L.shared is not None else 0, s.x_dtype)
        self.x = dev(L.xb)
        self.Wr = dev(L.Wr)
        self.bias = None if L.bias is None else dev(L.bias)
        self.blob = dev(L.experts)
        self.experts = qm.make_experts(self.blob, L.stride)
        if L.shared is not None:
            self.sh = {k: dev(v) for k, v in L.shared.items()}
            self.shared = qm.make_shared(self.sh["gate"], self.sh["up"], self.sh["down"], self.sh["sig"])
        else:
            self.shared = None

    def xrows(self, t0, n):
        return self.x[t0:t0 + n].contiguous()

    def moe(self, t0, n):
        H = self.L.shape.hidden
        ws = qm.alloc_workspace(self.shape, n)
        out = torch.full((n, H), float("nan"), device="cuda")
        qm.qs_moe_ffn(self.shape, self.xrows(t0, n), self.Wr, self.bias, self.experts, self.shared, out, n, ws)
        torch.cuda.synchronize()
        assert qm.qs_read_device_status(ws) == qm.QS_OK
        return out.cpu().numpy()


def check_layer_outputs(L, ref, got_y, tokens, what):
    """Compare y token by token, skipping tokens whose routing is within the margin."""
    skipped = 0
    rows_g, rows_r = [], []
    for i, t in enumerate(tokens):
        if ref["margin"][t] < MARGIN:
            skipped += 1
            continue
        rows_g.append(got_y[i])
        rows_r.append(ref["y"][t])
    assert rows_g, f"{what}: every token was within the routing margin"
    assert_close(np.array(rows_g), np.array(rows_r), what=what)
    return skipped


# ------------------------------------------------------------------ encoder

def test_quantize_bit_exact_against_oracle():
    rng = np.random.default_rng(0)
    w = (rng.standard_normal((96, 1024)) * 0.02).astype(np.float32)
    w[0] = 0.0
    w[1] = 0.0123
    w[2] = -np.abs(w[2])
    w[3] = np.abs(w[3])
    w[4, :256] = 1e-9                      # subnormal fp16 scales
    w[5] *= 1e3                            # large values
    ref = oracle.q2k_quantize(w)
    out = torch.zeros(ref.shape, dtype=torch.uint8, device="cuda")
    qm.qs_q2k_quantize(dev(w), out)
    got = out.cpu().numpy()
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} bytes differ"


def test_quantize_layer_expert_bit_exact():
    sh = qi.WORKLOADS["decode_35b_a3b"].shape
    g, u, d = qi.gen_expert_f32(sh, 1, 0, 17)
    for m in (g, u, d):
        ref = oracle.q2k_quantize(m)
        out = torch.zeros(ref.shape, dtype=torch.uint8, device="cuda")
        qm.qs_q2k_quantize(dev(m), out)
        assert np.array_equal(out.cpu().numpy(), ref)


# ------------------------------------------------------------------ (a) routing

# decode_35b_a3b at 6 tokens stages exactly 48 KB of x in shared memory (the routing kernel
# has static shared memory too, so the launch needs the opt-in); at 7, 56 KB.
@pytest.mark.parametrize("wl,T", [("tiny", 4), ("tiny", 13), ("decode_35b_a3b", 6), ("decode_35b_a3b", 7),
                                  ("decode_35b_a3b", 64), ("verify8_zipf", 64), ("decode_h4096", 24)])
def test_route_topk_parity(wl, T):
    w = qi.WORKLOADS[wl]
    L = Layer(w.shape, w.seed, 0, n_x=T, zipf=w.zipf_bias, shared=False, expert_subset=[])
    D = DevLayer(L)
    k = w.shape.top_k
    ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    pw = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    ws = qm.alloc_workspace(D.shape, T)
    for rep in range(2):   # the second call checks the tickets were re-armed
        qm.qs_route_topk(D.shape, D.x, D.Wr, D.bias, T, ids, pw, ws)
        torch.cuda.synchronize()
        rids, rp, margin, _ = oracle.route(L.xb, L.x_dtype, L.Wr, L.bias, k)
        gi, gp = ids.cpu().numpy(), pw.cpu().numpy()
        ok = margin >= MARGIN
        assert np.array_equal(gi[ok], rids[ok])
        assert np.allclose(gp[ok], rp[ok], rtol=0, atol=1e-6)
        assert np.allclose(gp.sum(1), 1.0, atol=1e-6)


# ------------------------------------------------------------------ (b) grouping

@pytest.mark.parametrize("T,k,E", [(1, 8, 256), (8, 8, 256), (13, 2, 8), (64, 8, 256), (2048, 8, 256),
                                   (300, 4, 1000), (5, 1, 1)])
def test_group_tokens_bit_exact(T, k, E):
    rng = np.random.default_rng(T + 7 * k + E)
    probs = 1.0 / np.arange(1, E + 1) ** 1.1          # skewed load: a few experts take most tokens
    probs /= probs.sum()
    ids = np.stack([rng.choice(E, k, replace=False, p=probs) for _ in range(T)]).astype(np.int32)
    rc, ro, rp = oracle.group(ids, E)
    shape = qm.make_shape(256, E, k, 256, 0, 0)
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    offs = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
    qm.qs_group_tokens(shape, dev(ids), T, counts, offs, perm)
    torch.cuda.synchronize()
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offs.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)


# ------------------------------------------------------------------ (c) gate/up, (d) down, shared

SHAPES = {
    "tiny": qi.WORKLOADS["tiny"].shape,
    "h768_f512": qi.LayerShape(768, 16, 4, 512, 256, qi.BF16),      # 3 blocks per row: shared-memory reduction
    "h2048_f512": qi.LayerShape(2048, 32, 8, 512, 512, qi.BF16),
    "h4096_f2048": qi.LayerShape(4096, 16, 8, 2048, 256, qi.BF16),  # 64 threads per row
    "e1_k1": qi.LayerShape(512, 1, 1, 256, 256, qi.F32),
    "k_eq_e": qi.LayerShape(256, 4, 4, 256, 256, qi.BF16),
}


def _grouped_h(D, L, T):
    """Group the oracle's ids on the GPU, then run the grouped gate/up on them."""
    k = L.shape.top_k
    ref = L.oracle(tokens=range(T))
    ids = dev(ref["ids"][:T])
    E = L.shape.n_experts
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    offs = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    qm.qs_group_tokens(D.shape, ids, T, counts, offs, perm)
    h = torch.full((T * k, L.shape.expert_ffn), float("nan"), device="cuda")
    qm.qs_q2k_gemv_grouped(D.shape, D.xrows(0, T), D.experts, offs, perm, T, h)
    torch.cuda.synchronize()
    return ref, ids, h


@pytest.mark.parametrize("name", list(SHAPES))
def test_gemv_grouped_parity(name):
    shape = SHAPES[name]
    T = 5
    L = Layer(shape, 100, 0, n_x=T)
    D = DevLayer(L)
    ref, _, h = _grouped_h(D, L, T)
    assert_close(h.cpu().numpy(), ref["h"][:T * shape.top_k], what=f"h {name}")


@pytest.mark.parametrize("name", list(SHAPES))
def test_down_combine_parity(name):
    shape = SHAPES[name]
    T = 5
    L = Layer(shape, 101, 0, n_x=T)
    D = DevLayer(L)
    k, H = shape.top_k, shape.hidden
    ref = L.oracle(tokens=range(T))
    h = dev(ref["h"][:T * k].astype(np.float32))
    ids = dev(ref["ids"][:T])
    pw = dev(ref["p"][:T].astype(np.float32))
    out = torch.full((T, H), float("nan"), device="cuda")
    qm.qs_q2k_down_combine(D.shape, D.experts, h, ids, pw, T, out)
    torch.cuda.synchronize()
    expect = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ref["ids"][t, j]
            blob = L.experts[e * L.stride:(e + 1) * L.stride]
            expect[t] += np.float32(ref["p"][t, j]) * oracle.expert_down(H, shape.expert_ffn, blob,
                                                                          ref["h"][t * k + j].astype(np.float32))
    assert_close(out.cpu().numpy(), expect, what=f"down {name}")
    # accumulate=1 adds on top
    qm.qs_q2k_down_combine(D.shape, D.experts, h, ids, pw, T, out, accumulate=True)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), 2 * expect, what=f"down acc {name}")


@pytest.mark.parametrize("name", ["tiny", "h768_f512", "h2048_f512", "h4096_f2048"])
def test_shared_expert_parity(name):
    shape = SHAPES[name]
    T = 6
    L = Layer(shape, 102, 0, n_x=T, expert_subset=[])
    D = DevLayer(L)
    H, S = shape.hidden, shape.shared_ffn
    out = torch.full((T, H), float("nan"), device="cuda")
    ws = qm.alloc_workspace(D.shape, T)
    qm.qs_shared_expert_ffn(D.shape, D.x, D.shared, T, out, ws)
    torch.cuda.synchronize()
    xw = L.xf.astype(np.float64)
    expect = np.stack([oracle.shared_expert(H, S, L.shared, xw[t])[2] for t in range(T)])
    assert_close(out.cpu().numpy(), expect, what=f"shared {name}")


# ------------------------------------------------------------------ the whole layer

@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("T", [1, 4, 13])
def test_moe_ffn_parity_small(name, T):
    shape = SHAPES[name]
    L = Layer(shape, 200 + T, 0, n_x=T)
    D = DevLayer(L)
    got = D.moe(0, T)
    ref = L.oracle()
    check_layer_outputs(L, ref, got, range(T), f"moe {name} T={T}")


def test_moe_ffn_tiny_workload():
    w = qi.WORKLOADS["tiny"]
    L = Layer(w.shape, w.seed, 0, n_x=w.tokens[0])
    D = DevLayer(L)
    got = D.moe(0, w.tokens[0])
    ref = L.oracle()
    check_layer_outputs(L, ref, got, range(w.tokens[0]), "tiny workload")


def test_moe_ffn_without_shared_expert():
    shape = SHAPES["h2048_f512"]
    L = Layer(shape, 300, 0, n_x=3, shared=False)
    D = DevLayer(L)
    got = D.moe(0, 3)
    check_layer_outputs(L, L.oracle(), got, range(3), "no shared")


# ------------------------------------------------------------------ the largest batches and top-k

def test_moe_ffn_decode_kernel_at_its_entry_limit():
    """16 tokens x top-8 = 128 (token, slot) entries: the most the single-kernel decode path takes
    (with 64 experts its candidate buffer holds them; its int16 h cache leaves one stage)."""
    shape = qi.LayerShape(2048, 64, 8, 512, 512, qi.BF16)
    L = Layer(shape, 310, 0, n_x=16)
    D = DevLayer(L)
    assert qm.qs_moe_ffn_launches(D.shape, 16, True) == 1
    check_layer_outputs(L, L.oracle(threads=8), D.moe(0, 16), range(16), "decode kernel, 128 entries")


@pytest.mark.parametrize("T,x_dtype,launches", [(4, qi.BF16, 1), (5, qi.BF16, 8), (5, qi.F32, 5)])
def test_moe_ffn_top_k_32(T, x_dtype, launches):
    """top-k at its maximum (32) on each path: the decode kernel (4 x 32 = 128 entries), the
    tensor-core path (160 entries, bf16 x) and the per-step kernels (fp32 x)."""
    shape = qi.LayerShape(256, 64, 32, 256, 256, x_dtype)
    L = Layer(shape, 320 + T, 0, n_x=T)
    D = DevLayer(L)
    assert qm.qs_moe_ffn_launches(D.shape, T, True) == launches
    check_layer_outputs(L, L.oracle(), D.moe(0, T), range(T), f"top-32, {T} tokens, {launches} launches")


@pytest.mark.slow
def test_moe_ffn_35b_shape_between_decode_and_prefill_batches():
    """The 35B-A3B layer at 12 tokens: past the decode kernel's candidate buffer (8 tokens at 256
    experts, top-8), below the smallest batch the tensor-core tests take."""
    w = qi.WORKLOADS["decode_35b_a3b"]
    L = Layer(w.shape, w.seed, 0, n_x=12, expert_subset="routed")
    D = DevLayer(L)
    assert qm.qs_moe_ffn_launches(D.shape, 12, True) == 8
    check_layer_outputs(L, L.oracle(threads=8), D.moe(0, 12), range(12), "35B-A3B layer, 12 tokens")


@pytest.mark.slow
@pytest.mark.parametrize("wl,T,calls", [("decode_35b_a3b", 1, 4), ("verify8_zipf", 8, 1), ("decode_h4096", 1, 2),
                                        ("decode_h4096", 4, 1)])
def test_moe_ffn_full_size_sampled(wl, T, calls):
    """Full layer shape and the launch configuration of the bench; only the experts the sampled
    tokens route to are synthesised (the rest of the layer is zero and must never be read)."""
    w = qi.WORKLOADS[wl]
    n = T * calls
    L = Layer(w.shape, w.seed, 0, n_x=n, zipf=w.zipf_bias, expert_subset="routed")
    D = DevLayer(L)
    ref = L.oracle(threads=8)
    for c in range(calls):
        got = D.moe(c * T, T)
        check_layer_outputs(L, ref, got, range(c * T, (c + 1) * T), f"{wl} call {c}")


@pytest.mark.slow
def test_moe_ffn_prefill_sampled():
    w = qi.WORKLOADS["prefill_2048"]
    T = w.tokens[0]
    sample = list(range(0, T, 97))[:16]
    L = Layer(w.shape, w.seed, 0, n_x=T, expert_subset=[])
    ids, _, _, _ = oracle.route(L.xb[sample], L.x_dtype, L.Wr, L.bias, w.shape.top_k)
    L.experts = build_experts(w.shape, w.seed, 0, np.unique(ids))
    D = DevLayer(L)
    got = D.moe(0, T)
    ref = L.oracle(tokens=sample, threads=8)
    check_layer_outputs(L, ref, got[sample], sample, "prefill sampled")


def test_n_invariance_batch_equals_single_calls():
    shape = qi.LayerShape(2048, 64, 8, 512, 512, qi.BF16)
    L = Layer(shape, 400, 0, n_x=8, zipf=1.1)
    D = DevLayer(L)
    batch = D.moe(0, 8)
    singles = np.concatenate([D.moe(t, 1) for t in range(8)])
    assert np.array_equal(batch, singles)


# ------------------------------------------------------------------ errors, status, bounds

def test_short_workspace_is_rejected():
    shape = SHAPES["tiny"]
    L = Layer(shape, 500, 0, n_x=2)
    D = DevLayer(L)
    ws = qm.alloc_workspace(D.shape, 1)
    out = torch.zeros((2, shape.hidden), device="cuda")
    with pytest.raises(qm.QsError) as ei:
        qm.qs_moe_ffn(D.shape, D.x, D.Wr, None, D.experts, D.shared, out, 2, ws)
    assert ei.value.code == qm.QS_ERR_WORKSPACE


def test_wait_timeout_reports_status():
    shape = SHAPES["tiny"]
    ws = qm.alloc_workspace(qm.make_shape(shape.hidden, shape.n_experts, shape.top_k, shape.expert_ffn,
                                          shape.shared_ffn, shape.x_dtype), 1)
    assert qm.qs_read_device_status(ws) == qm.QS_OK
    qm.qs_test_wait_timeout(ws, 2000)
    assert qm.qs_read_device_status(ws) == qm.QS_ERR_TIMEOUT
    qm.qs_workspace_init(ws)
    assert qm.qs_read_device_status(ws) == qm.QS_OK


def test_output_guard_regions_untouched():
    shape = SHAPES["h2048_f512"]
    T = 3
    L = Layer(shape, 600, 0, n_x=T)
    D = DevLayer(L)
    H = shape.hidden
    pad = 4096
    buf = torch.full((T * H + 2 * pad,), 12345.0, device="cuda")
    out = buf[pad:pad + T * H].view(T, H)
    ws = qm.alloc_workspace(D.shape, T)
    qm.qs_moe_ffn(D.shape, D.x, D.Wr, None, D.experts, D.shared, out, T, ws)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:pad] == 12345.0) and np.all(b[-pad:] == 12345.0)
    check_layer_outputs(L, L.oracle(), out.cpu().numpy(), range(T), "guarded")
