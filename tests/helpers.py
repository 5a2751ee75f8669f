"""Test-side layer builders: seeded inputs (qs_inputs) quantised by the oracle's encoder.

Nothing here comes from the CUDA path: every byte the oracle reads is produced
on the host from the shared generators and the oracle's own Q2_K encoder.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle
import qs_inputs as qi

_THREADS = max(1, min(16, os.cpu_count() or 1))


def build_experts(shape: qi.LayerShape, seed: int, copy: int, subset=None) -> np.ndarray:
    """E * expert_bytes Q2_K blob; experts outside `subset` (if given) are left zero."""
    stride = shape.expert_bytes
    blob = np.zeros(shape.n_experts * stride, np.uint8)
    todo = range(shape.n_experts) if subset is None else sorted(set(int(e) for e in subset))

    def one(e):
        blob[e * stride:(e + 1) * stride] = oracle.quantize_expert(*qi.gen_expert_f32(shape, seed, copy, e))

    with cf.ThreadPoolExecutor(_THREADS) as ex:
        list(ex.map(one, todo))
    return blob


class Layer:
    """One seeded synthetic layer plus an x pool, on the host."""

    def __init__(self, shape: qi.LayerShape, seed: int, copy: int = 0, n_x: int = 8, zipf: float = 0.0,
                 shared: bool = True, expert_subset="all", x_start: int = 0):
        self.shape, self.seed, self.copy = shape, seed, copy
        self.xb, self.xf = qi.gen_x(shape, seed, n_x, x_start)
        self.Wr = qi.gen_router(shape, seed, copy)
        self.bias = qi.gen_bias(shape, seed, copy, zipf)
        self.shared = qi.gen_shared(shape, seed, copy) if (shared and shape.shared_ffn > 0) else None
        if isinstance(expert_subset, str) and expert_subset == "routed":
            ids, _, _, _ = oracle.route(self.xb, self.x_dtype, self.Wr, self.bias, shape.top_k)
            expert_subset = np.unique(ids)
        all_experts = isinstance(expert_subset, str) and expert_subset == "all"
        self.experts = build_experts(shape, seed, copy, None if all_experts else expert_subset)
        self.stride = shape.expert_bytes

    @property
    def x_dtype(self):
        return oracle.X_BF16 if self.shape.x_dtype == qi.BF16 else oracle.X_F32

    def oracle(self, tokens=None, threads=1, x=None):
        return oracle.moe_ffn(self.shape, self.xb if x is None else x, self.Wr, self.bias, self.experts,
                              self.stride, self.shared, tokens=tokens, threads=threads)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_close(got, ref, rel=2e-3, maxabs_frac=1e-2, what=""):
    """The layer's float acceptance: rel-L2 <= 2e-3 and max-abs <= 1e-2 * max|ref|."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    r = rel_l2(got, ref)
    m = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    lim = maxabs_frac * float(np.max(np.abs(ref))) if ref.size else 0.0
    assert r <= rel and m <= lim, f"{what}: rel-L2 {r:.3e} (<= {rel}), max-abs {m:.3e} (<= {lim:.3e})"
    return r, m
