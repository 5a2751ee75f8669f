"""Pins of the oracle's routing, grouping and layer composition.

Each check compares the oracle with something it does not compute itself: a
full sort done here, closed-form softmax values, numpy matrix products on the
(separately pinned) dequantised matrices, and textbook special cases of the
layer (one expert = a SwiGLU MLP, diagonal experts = elementwise SwiGLU, a zero
router = uniform weights, a zero gate vector = gate 1/2).
"""
import math

import numpy as np
import pytest

import oracle
import qs_inputs as qi


def _silu(z):
    return z / (1.0 + np.exp(-z))


def _mlp(Wg, Wu, Wd, x):
    return Wd @ (_silu(Wg @ x) * (Wu @ x))


def _random_layer(shape, seed=0, copy=0):
    E, F, H = shape.n_experts, shape.expert_ffn, shape.hidden
    blobs = [oracle.quantize_expert(*qi.gen_expert_f32(shape, seed, copy, e)) for e in range(E)]
    experts = np.concatenate(blobs)
    return experts, shape.expert_bytes


def _dense_expert(shape, experts, e):
    F, H = shape.expert_ffn, shape.hidden
    blob = experts[e * shape.expert_bytes:(e + 1) * shape.expert_bytes]
    g_bytes = F * H // 256 * 84
    Wg = oracle.q2k_dequant(blob[:g_bytes], F, H)
    Wu = oracle.q2k_dequant(blob[g_bytes:2 * g_bytes], F, H)
    Wd = oracle.q2k_dequant(blob[2 * g_bytes:], H, F)
    return Wg, Wu, Wd


# ------------------------------------------------------------------ routing

def test_router_logits_are_the_matrix_product():
    shape = qi.LayerShape(512, 16, 4, 256, 256, qi.BF16)
    xb, xf = qi.gen_x(shape, 9, 5)
    Wr = qi.gen_router(shape, 9, 0)
    b = qi.gen_bias(shape, 9, 0, 1.1)
    ids, p, margin, logits = oracle.route(xb, oracle.X_BF16, Wr, b, shape.top_k)
    ref = xf.astype(np.float64) @ Wr.astype(np.float64).T + b.astype(np.float64)
    assert np.allclose(logits, ref, rtol=1e-12, atol=1e-12)


def test_topk_equals_full_sort_and_weights_sum_to_one():
    shape = qi.LayerShape(256, 64, 8, 256, 256, qi.F32)
    xb, _ = qi.gen_x(shape, 11, 32)
    Wr = qi.gen_router(shape, 11, 0)
    ids, p, margin, logits = oracle.route(xb, oracle.X_F32, Wr, None, shape.top_k)
    for t in range(32):
        order = sorted(range(shape.n_experts), key=lambda e: (-logits[t, e], e))
        assert list(ids[t]) == order[:shape.top_k]
        assert margin[t] == logits[t, order[7]] - logits[t, order[8]]
        assert abs(p[t].sum() - 1.0) <= 1e-15 * shape.top_k
        assert np.all(np.diff(p[t]) <= 0)
        # softmax over the selected logits = full softmax renormalised over the selection
        full = np.exp(logits[t] - logits[t].max())
        full /= full.sum()
        sel = full[ids[t]] / full[ids[t]].sum()
        assert np.allclose(p[t], sel, rtol=1e-13, atol=0)


def test_topk_ties_go_to_lower_index():
    H, E, k = 256, 8, 3
    Wr = np.zeros((E, H), np.float32)
    Wr[:, 0] = [1, 2, 2, 0, 2, 1, 0, 2]     # logits = column 0 when x = e_0
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1
    ids, p, margin, _ = oracle.route(x, oracle.X_F32, Wr, None, k)
    assert list(ids[0]) == [1, 2, 4]
    assert margin[0] == 0.0
    assert np.allclose(p[0], [1 / 3] * 3, rtol=1e-15)


def test_softmax_closed_form():
    H, E, k = 256, 4, 2
    Wr = np.zeros((E, H), np.float32)
    Wr[:, 0] = [3, 1, 2, 0]
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1
    ids, p, margin, _ = oracle.route(x, oracle.X_F32, Wr, None, k)
    assert list(ids[0]) == [0, 2]
    e = math.e
    assert abs(p[0, 0] - e / (e + 1)) < 1e-15 and abs(p[0, 1] - 1 / (e + 1)) < 1e-15
    assert margin[0] == 1.0


def test_k_equal_E_has_infinite_margin():
    H, E = 256, 4
    Wr = qi.gen_router(qi.LayerShape(H, E, E, 256, 256, qi.F32), 2, 0)
    xb, _ = qi.gen_x(qi.LayerShape(H, E, E, 256, 256, qi.F32), 2, 3)
    ids, p, margin, _ = oracle.route(xb, oracle.X_F32, Wr, None, E)
    assert np.all(np.isinf(margin))
    assert all(sorted(r) == list(range(E)) for r in ids)


# ------------------------------------------------------------------ grouping

@pytest.mark.parametrize("T,k,E", [(1, 8, 256), (8, 8, 256), (64, 2, 8), (5, 3, 4)])
def test_grouping_against_brute_force(T, k, E):
    rng = np.random.default_rng(T * 100 + k)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = oracle.group(ids, E)
    flat = ids.reshape(-1)
    assert counts.sum() == T * k
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert sorted(perm) == list(range(T * k))
    expect = sorted(range(T * k), key=lambda i: (flat[i], i))
    assert list(perm) == expect


# ------------------------------------------------------------------ layer composition

def test_single_expert_is_a_swiglu_mlp():
    shape = qi.LayerShape(512, 1, 1, 256, 0, qi.F32)      # F != H catches a transposed matrix
    experts, stride = _random_layer(shape, 21)
    Wg, Wu, Wd = _dense_expert(shape, experts, 0)
    xb, xf = qi.gen_x(shape, 21, 3)
    Wr = np.zeros((1, 512), np.float32)
    out = oracle.moe_ffn(shape, xb, Wr, None, experts, stride, None)
    for t in range(3):
        ref = _mlp(Wg, Wu, Wd, xf[t].astype(np.float64))
        assert out["p"][t, 0] == 1.0 and out["ids"][t, 0] == 0
        assert np.allclose(out["y"][t], ref, rtol=1e-11, atol=1e-13)
        assert np.allclose(out["h"][t], _silu(Wg @ xf[t]) * (Wu @ xf[t]), rtol=1e-11, atol=1e-14)


def _diag_q2k(n):
    """n x n identity as Q2_K rows (one block row per 256 columns): w[r, r] = 1."""
    nb = n // 256
    rows = np.zeros((n, nb * 84), np.uint8)
    for r in range(n):
        b, i = divmod(r, 256)
        blk = rows[r, b * 84:(b + 1) * 84]
        blk[0:16] = 0x01                     # scale nibble 1, min nibble 0
        hh, rem = divmod(i, 128)
        j, l = divmod(rem, 32)
        blk[16 + 32 * hh + l] = 1 << (2 * j)  # q = 1 at weight i
        blk[80:82] = [0x00, 0x3c]           # d = 1
    return rows.reshape(-1)


def test_diagonal_expert_gives_elementwise_swiglu():
    n = 256
    shape = qi.LayerShape(n, 1, 1, n, 0, qi.F32)
    blob = np.concatenate([_diag_q2k(n)] * 3)
    x = np.zeros((1, n), np.float32)
    x[0, :4] = [0.0, 1.0, -1.0, 2.0]
    out = oracle.moe_ffn(shape, x, np.zeros((1, n), np.float32), None, blob, shape.expert_bytes, None)
    y = out["y"][0]
    # silu(x) * x = x^2 / (1 + e^-x)
    assert y[0] == 0.0
    assert abs(y[1] - 1 / (1 + math.exp(-1))) < 1e-15
    assert abs(y[2] - 1 / (1 + math.exp(1))) < 1e-15
    assert abs(y[3] - 4 / (1 + math.exp(-2))) < 1e-15
    assert np.all(y[4:] == 0)


def test_expert_blob_keeps_gate_up_down_roles():
    # Three different matrices for the three roles (gate 2I, up I, down I/2), each quantised on
    # its own for the expectation: the layer's h and y must follow the matrix each role was made
    # from, whatever order the expert's blob stores them in.
    n = 256
    shape = qi.LayerShape(n, 1, 1, n, 0, qi.F32)
    eye = np.eye(n, dtype=np.float32)
    gate, up, down = 2.0 * eye, eye, 0.5 * eye
    blob = oracle.quantize_expert(gate, up, down)
    Wg, Wu, Wd = (oracle.q2k_dequant(oracle.q2k_quantize(a), n, n) for a in (gate, up, down))
    x = np.zeros((1, n), np.float32)
    x[0, :3] = [1.0, -0.5, 2.0]
    out = oracle.moe_ffn(shape, x, np.zeros((1, n), np.float32), None, blob, shape.expert_bytes, None)
    xf = x[0].astype(np.float64)
    h = _silu(Wg @ xf) * (Wu @ xf)
    assert not np.allclose(h, _silu(Wu @ xf) * (Wg @ xf))   # the roles are told apart
    assert np.allclose(out["h"][0], h, rtol=1e-12, atol=1e-15)
    assert np.allclose(out["y"][0], Wd @ h, rtol=1e-12, atol=1e-15)


def test_zero_router_gives_uniform_weights_and_sum_of_mlps():
    shape = qi.LayerShape(256, 4, 2, 256, 0, qi.F32)
    experts, stride = _random_layer(shape, 31)
    xb, xf = qi.gen_x(shape, 31, 2)
    out = oracle.moe_ffn(shape, xb, np.zeros((4, 256), np.float32), None, experts, stride, None)
    W0, W1 = _dense_expert(shape, experts, 0), _dense_expert(shape, experts, 1)
    for t in range(2):
        assert list(out["ids"][t]) == [0, 1] and np.all(out["p"][t] == 0.5)
        ref = 0.5 * _mlp(*W0, xf[t].astype(np.float64)) + 0.5 * _mlp(*W1, xf[t].astype(np.float64))
        assert np.allclose(out["y"][t], ref, rtol=1e-11, atol=1e-13)


def test_zero_gate_vector_gives_half_the_shared_mlp():
    shape = qi.LayerShape(256, 2, 1, 256, 256, qi.BF16)
    zero_experts = np.zeros(2 * shape.expert_bytes, np.uint8)    # all-zero blocks decode to 0
    sh = qi.gen_shared(shape, 41, 0)
    sh["sig"] = np.zeros_like(sh["sig"])
    xb, xf = qi.gen_x(shape, 41, 2)
    out = oracle.moe_ffn(shape, xb, qi.gen_router(shape, 41, 0), None, zero_experts, shape.expert_bytes, sh)
    Wg = qi.bf16_bits_to_f32(sh["gate"]).astype(np.float64)
    Wu = qi.bf16_bits_to_f32(sh["up"]).astype(np.float64)
    Wd = qi.bf16_bits_to_f32(sh["down"]).astype(np.float64)
    for t in range(2):
        assert out["gate"][t] == 0.5
        ref = 0.5 * _mlp(Wg, Wu, Wd, xf[t].astype(np.float64))
        assert np.allclose(out["y"][t], ref, rtol=1e-11, atol=1e-14)


def test_full_tiny_layer_against_dense_brute_force():
    wl = qi.WORKLOADS["tiny"]
    shape = wl.shape
    experts, stride = _random_layer(shape, wl.seed)
    xb, xf = qi.gen_x(shape, wl.seed, wl.tokens[0])
    Wr = qi.gen_router(shape, wl.seed, 0)
    sh = qi.gen_shared(shape, wl.seed, 0)
    out = oracle.moe_ffn(shape, xb, Wr, None, experts, stride, sh)
    Sg = qi.bf16_bits_to_f32(sh["gate"]).astype(np.float64)
    Su = qi.bf16_bits_to_f32(sh["up"]).astype(np.float64)
    Sd = qi.bf16_bits_to_f32(sh["down"]).astype(np.float64)
    ssig = qi.bf16_bits_to_f32(sh["sig"]).astype(np.float64)
    dense = [_dense_expert(shape, experts, e) for e in range(shape.n_experts)]
    for t in range(wl.tokens[0]):
        x = xf[t].astype(np.float64)
        l = Wr.astype(np.float64) @ x
        top = sorted(range(shape.n_experts), key=lambda e: (-l[e], e))[:shape.top_k]
        w = np.exp(l[top] - l[top].max())
        w /= w.sum()
        ref = sum(w[j] * _mlp(*dense[e], x) for j, e in enumerate(top))
        ref = ref + _mlp(Sg, Su, Sd, x) / (1.0 + math.exp(-(ssig @ x)))
        assert list(out["ids"][t]) == top
        assert np.allclose(out["p"][t], w, rtol=1e-13)
        assert np.allclose(out["y"][t], ref, rtol=1e-10, atol=1e-13)


def test_token_subset_and_threads_match_full_run():
    wl = qi.WORKLOADS["tiny"]
    shape = wl.shape
    experts, stride = _random_layer(shape, wl.seed)
    xb, _ = qi.gen_x(shape, wl.seed, 6)
    Wr = qi.gen_router(shape, wl.seed, 0)
    sh = qi.gen_shared(shape, wl.seed, 0)
    full = oracle.moe_ffn(shape, xb, Wr, None, experts, stride, sh)
    part = oracle.moe_ffn(shape, xb, Wr, None, experts, stride, sh, tokens=[1, 4], threads=2)
    for t in (1, 4):
        assert np.array_equal(full["y"][t], part["y"][t])
    assert np.all(part["y"][0] == 0)
