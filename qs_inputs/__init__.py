"""Seeded synthetic inputs for the Q2_K mixture-of-experts FFN layer.

This module is shared by the tests, the bench and the oracle-driven checks.  It
holds no arithmetic of the layer itself: it draws random numbers, rounds them
to the storage types the layer consumes (fp32, bf16 bit patterns) and describes
the five workload shapes.  Quantisation of expert weights to Q2_K is *not* done
here: the test side quantises with the oracle's encoder, the product side with
the library's device encoder.

Random numbers come from one counter-based generator so any element of any
tensor can be regenerated on its own:

  * key     = SplitMix64 chain over (seed, stream, tensor tag, expert index)
  * u64(i)  = SplitMix64 finaliser of key + i * 0x9E3779B97F4A7C15
  * normals = Box-Muller on the pair (u64(2n), u64(2n+1)); element 2n takes the
              cosine branch, element 2n+1 the sine branch.

SplitMix64 is the generator of Steele, Lea and Flood, "Fast splittable
pseudorandom number generators" (OOPSLA 2014); Box-Muller is the textbook
transform of two uniforms into two independent standard normals.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor tags of the key chain
TAG_X = 1
TAG_ROUTER = 2
TAG_BIAS_PERM = 3
TAG_GATE = 10
TAG_UP = 11
TAG_DOWN = 12
TAG_SH_GATE = 20
TAG_SH_UP = 21
TAG_SH_DOWN = 22
TAG_SH_SIG = 23
TAG_DIRECTION = 30
TAG_ROWS = 31

F32 = 0
BF16 = 1


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix_scalar(v: int) -> int:
    with np.errstate(over="ignore"):
        return int(_mix(np.array([v & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0])


def make_key(seed: int, stream: int, tag: int, index: int = 0) -> int:
    """64-bit key of one tensor: SplitMix64 over (seed, stream, tag, index)."""
    k = _mix_scalar(seed)
    k = _mix_scalar(k + stream)
    k = _mix_scalar(k + tag)
    k = _mix_scalar(k + index)
    return k


def uniform_bits(key: int, start: int, count: int) -> np.ndarray:
    """u64 draws number start .. start+count-1 of the stream `key`."""
    i = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + i * _GOLDEN
        return _mix(z)


def normal(key: int, start: int, count: int) -> np.ndarray:
    """Standard normals number start .. start+count-1 of stream `key` (float64)."""
    if count <= 0:
        return np.zeros(0, dtype=np.float64)
    p0 = start // 2
    p1 = (start + count - 1) // 2
    npair = p1 - p0 + 1
    bits = uniform_bits(key, 2 * p0, 2 * npair).reshape(npair, 2)
    u1 = ((bits[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (bits[:, 1] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    a = 2.0 * math.pi * u2
    z = np.empty((npair, 2), dtype=np.float64)
    z[:, 0] = r * np.cos(a)
    z[:, 1] = r * np.sin(a)
    z = z.reshape(-1)
    off = start - 2 * p0
    return z[off:off + count]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (storage conversion only)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Shape of one MoE-FFN layer (hidden H, experts E, top-k, expert ffn F, shared ffn S)."""
    hidden: int
    n_experts: int
    top_k: int
    expert_ffn: int
    shared_ffn: int
    x_dtype: int  # F32 or BF16

    @property
    def blocks_per_row_h(self) -> int:
        return self.hidden // 256

    @property
    def blocks_per_row_f(self) -> int:
        return self.expert_ffn // 256

    @property
    def expert_bytes(self) -> int:
        """Q2_K bytes of one expert: gate [F x H] + up [F x H] + down [H x F], 84 B per 256 weights."""
        return 84 * (2 * self.expert_ffn * self.hidden + self.hidden * self.expert_ffn) // 256


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    tokens: tuple          # token counts the workload is run at
    copies: int            # distinct layer copies cycled to defeat L2
    seed: int
    zipf_bias: float = 0.0  # exponent of the Zipf router bias, 0 = none


WORKLOADS = {
    "tiny": Workload("tiny", LayerShape(256, 8, 2, 256, 256, F32), (4,), 1, 0),
    "decode_35b_a3b": Workload("decode_35b_a3b", LayerShape(2048, 256, 8, 512, 512, BF16), (1,), 4, 1),
    "verify8_zipf": Workload("verify8_zipf", LayerShape(2048, 256, 8, 512, 512, BF16), (8,), 4, 2, zipf_bias=1.1),
    "prefill_2048": Workload("prefill_2048", LayerShape(2048, 256, 8, 512, 512, BF16), (2048,), 1, 3),
    "decode_h4096": Workload("decode_h4096", LayerShape(4096, 256, 8, 2048, 2048, BF16), (1, 4), 2, 4),
}

X_POOL = 64


def stream_of(seed: int, copy: int) -> int:
    return seed * 1000 + copy


def gen_x(shape: LayerShape, seed: int, n: int, start: int = 0):
    """x pool rows start..start+n-1, N(0,1).  Returns (storage array, fp32 view).

    fp32 layers store fp32; bf16 layers store bf16 bit patterns (uint16)."""
    key = make_key(seed, 0, TAG_X)
    z = normal(key, start * shape.hidden, n * shape.hidden).astype(np.float32).reshape(n, shape.hidden)
    if shape.x_dtype == BF16:
        b = f32_to_bf16_bits(z)
        return b, bf16_bits_to_f32(b)
    return z, z


def gen_router(shape: LayerShape, seed: int, copy: int) -> np.ndarray:
    key = make_key(seed, stream_of(seed, copy), TAG_ROUTER)
    return (0.02 * normal(key, 0, shape.n_experts * shape.hidden)).astype(np.float32).reshape(
        shape.n_experts, shape.hidden)


def gen_bias(shape: LayerShape, seed: int, copy: int, zipf: float):
    """Zipf(zipf) log-bias over experts: b[e] = -zipf * ln(rank[e]), rank a seeded permutation of 1..E."""
    if zipf == 0.0:
        return None
    key = make_key(seed, stream_of(seed, copy), TAG_BIAS_PERM)
    order = np.argsort(uniform_bits(key, 0, shape.n_experts), kind="stable")
    rank = np.empty(shape.n_experts, dtype=np.float64)
    rank[order] = np.arange(1, shape.n_experts + 1, dtype=np.float64)
    return (-zipf * np.log(rank)).astype(np.float32)


def gen_shared(shape: LayerShape, seed: int, copy: int) -> dict:
    """bf16 shared expert: gate/up [S x H], down [H x S], sigmoid-gate vector [H]; N(0, 0.02)."""
    S, H = shape.shared_ffn, shape.hidden
    st = stream_of(seed, copy)

    def draw(tag, n):
        return f32_to_bf16_bits((0.02 * normal(make_key(seed, st, tag), 0, n)).astype(np.float32))

    return {
        "gate": draw(TAG_SH_GATE, S * H).reshape(S, H),
        "up": draw(TAG_SH_UP, S * H).reshape(S, H),
        "down": draw(TAG_SH_DOWN, H * S).reshape(H, S),
        "sig": draw(TAG_SH_SIG, H),
    }


def gen_expert_f32(shape: LayerShape, seed: int, copy: int, e: int):
    """Expert e's unquantised weights N(0, 0.02): gate [F x H], up [F x H], down [H x F] (fp32)."""
    F, H = shape.expert_ffn, shape.hidden
    st = stream_of(seed, copy)

    def draw(tag, rows, cols):
        return (0.02 * normal(make_key(seed, st, tag, e), 0, rows * cols)).astype(np.float32).reshape(rows, cols)

    return draw(TAG_GATE, F, H), draw(TAG_UP, F, H), draw(TAG_DOWN, H, F)


def gen_direction(hidden: int, seed: int, copy: int = 0) -> np.ndarray:
    """A steering direction [hidden] fp32: N(0,1) scaled to unit length (stored normalised)."""
    z = normal(make_key(seed, stream_of(seed, copy), TAG_DIRECTION), 0, hidden)
    return (z / np.sqrt(np.sum(z * z))).astype(np.float32)


def gen_rows(n: int, hidden: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """n rows of hidden fp32 values, N(0, scale^2): stand-ins for a layer's output rows."""
    z = normal(make_key(seed, 0, TAG_ROWS), 0, n * hidden).reshape(n, hidden)
    return (scale * z).astype(np.float32)
