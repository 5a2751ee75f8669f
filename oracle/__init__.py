"""CPU oracle of the Q2_K mixture-of-experts FFN layer (ctypes over qs_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
bench's CPU-baseline leg, never by the product library.  It shares no code with
the CUDA path.  See qs_oracle.c for the definition it computes and its sources.

The shared object is compiled on first use with the host C compiler (plain
-O2, no fast-math, no floating-point contraction) into oracle/_build/.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qs_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libqs_oracle.so")
_lock = threading.Lock()
_lib = None

X_F32 = 0
X_BF16 = 1

# expert weight formats of qs_oracle.c
FMT = {"q2k": 0, "q4k": 1}
BLOCK_BYTES = {"q2k": 84, "q4k": 144}


def build(force: bool = False) -> str:
    """Compile qs_oracle.c into a shared object (idempotent)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int, ctypes.c_int64
            L.qso_half_to_double.restype = ctypes.c_double
            L.qso_half_to_double.argtypes = [ctypes.c_uint16]
            L.qso_bf16_to_double.restype = ctypes.c_double
            L.qso_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.qso_float_to_half.restype = ctypes.c_uint16
            L.qso_float_to_half.argtypes = [ctypes.c_float]
            L.qso_q2k_unpack.argtypes = [P, P, P, P, P]
            L.qso_q2k_pack.argtypes = [P, P, ctypes.c_uint16, ctypes.c_uint16, P]
            L.qso_q2k_dequant_rows.argtypes = [P, i64, i64, P]
            L.qso_q2k_quantize_rows.argtypes = [P, i64, i64, P]
            L.qso_route.restype = i32
            L.qso_route.argtypes = [i32, i32, i32, i32, P, i32, P, P, P, P, P, P]
            L.qso_group.argtypes = [i32, i32, i32, P, P, P, P]
            L.qso_expert_gateup.argtypes = [i32, i32, P, P, P]
            L.qso_expert_down.argtypes = [i32, i32, P, P, P]
            L.qso_shared_expert.argtypes = [i32, i32, P, P, P, P, P, P, P, P]
            L.qso_moe_ffn.restype = i32
            L.qso_moe_ffn.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, i32, P, P, P, i64,
                                      P, P, P, P, P, P, P, P, P, P, P]
            L.qso_steer_rows.argtypes = [i32, i32, P, ctypes.c_double, P]
            L.qso_q4k_unpack.argtypes = [P, P, P, P, P, P]
            L.qso_q4k_pack.argtypes = [P, P, P, ctypes.c_uint16, ctypes.c_uint16, P]
            L.qso_q4k_dequant_rows.argtypes = [P, i64, i64, P]
            L.qso_q4k_quantize_rows.argtypes = [P, i64, i64, P]
            L.qso_expert_gateup_fmt.argtypes = [i32, i32, i32, P, P, P]
            L.qso_expert_down_fmt.argtypes = [i32, i32, i32, P, P, P]
            L.qso_moe_ffn_fmt.restype = i32
            L.qso_moe_ffn_fmt.argtypes = [i32] + L.qso_moe_ffn.argtypes
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ storage types

def half_to_double(h: int) -> float:
    return lib().qso_half_to_double(h)


def bf16_to_double(b: int) -> float:
    return lib().qso_bf16_to_double(b)


def float_to_half(f: float) -> int:
    return lib().qso_float_to_half(f)


# ------------------------------------------------------------------ Q2_K

def q2k_unpack(block: np.ndarray):
    """84 bytes -> (scales[16] u8, q[256] u8, d bits, dmin bits)."""
    b = _c(block, np.uint8)
    assert b.size == 84
    sc = np.zeros(16, np.uint8)
    q = np.zeros(256, np.uint8)
    d = np.zeros(1, np.uint16)
    m = np.zeros(1, np.uint16)
    lib().qso_q2k_unpack(_p(b), _p(sc), _p(q), _p(d), _p(m))
    return sc, q, int(d[0]), int(m[0])


def q2k_pack(scales, q, d: int, dmin: int) -> np.ndarray:
    sc = _c(scales, np.uint8)
    qq = _c(q, np.uint8)
    out = np.zeros(84, np.uint8)
    lib().qso_q2k_pack(_p(sc), _p(qq), d, dmin, _p(out))
    return out


def q2k_dequant(rows: np.ndarray, n_rows: int, K: int) -> np.ndarray:
    """Q2_K bytes of n_rows rows of K weights -> float64 [n_rows, K] (exact)."""
    b = _c(rows, np.uint8).reshape(-1)
    assert b.size >= n_rows * K // 256 * 84
    w = np.zeros((n_rows, K), np.float64)
    lib().qso_q2k_dequant_rows(_p(b), n_rows, K, _p(w))
    return w


def q2k_quantize(w: np.ndarray) -> np.ndarray:
    """fp32 [rows, K] -> Q2_K bytes [rows, K/256*84] (round-to-nearest encoder)."""
    a = _c(w, np.float32)
    rows, K = a.shape
    assert K % 256 == 0
    out = np.zeros((rows, K // 256 * 84), np.uint8)
    lib().qso_q2k_quantize_rows(_p(a), rows, K, _p(out))
    return out


def q4k_unpack(block: np.ndarray):
    """144 bytes -> (sc[8] u8, m[8] u8, q[256] u8, d bits, dmin bits)."""
    b = _c(block, np.uint8)
    assert b.size == 144
    sc = np.zeros(8, np.uint8)
    m = np.zeros(8, np.uint8)
    q = np.zeros(256, np.uint8)
    d = np.zeros(1, np.uint16)
    dm = np.zeros(1, np.uint16)
    lib().qso_q4k_unpack(_p(b), _p(sc), _p(m), _p(q), _p(d), _p(dm))
    return sc, m, q, int(d[0]), int(dm[0])


def q4k_pack(sc, m, q, d: int, dmin: int) -> np.ndarray:
    out = np.zeros(144, np.uint8)
    lib().qso_q4k_pack(_p(_c(sc, np.uint8)), _p(_c(m, np.uint8)), _p(_c(q, np.uint8)), d, dmin, _p(out))
    return out


def q4k_dequant(rows: np.ndarray, n_rows: int, K: int) -> np.ndarray:
    """Q4_K bytes of n_rows rows of K weights -> float64 [n_rows, K] (exact)."""
    b = _c(rows, np.uint8).reshape(-1)
    assert b.size >= n_rows * K // 256 * 144
    w = np.zeros((n_rows, K), np.float64)
    lib().qso_q4k_dequant_rows(_p(b), n_rows, K, _p(w))
    return w


def q4k_quantize(w: np.ndarray) -> np.ndarray:
    """fp32 [rows, K] -> Q4_K bytes [rows, K/256*144] (round-to-nearest encoder)."""
    a = _c(w, np.float32)
    rows, K = a.shape
    assert K % 256 == 0
    out = np.zeros((rows, K // 256 * 144), np.uint8)
    lib().qso_q4k_quantize_rows(_p(a), rows, K, _p(out))
    return out


def quantize_expert(gate, up, down, fmt: str = "q2k") -> np.ndarray:
    """One expert's blob in format fmt ("q2k" or "q4k"): gate rows, up rows, down rows, concatenated."""
    qz = q4k_quantize if fmt == "q4k" else q2k_quantize
    return np.concatenate([qz(gate).reshape(-1), qz(up).reshape(-1), qz(down).reshape(-1)])


# ------------------------------------------------------------------ the layer

def route(x, x_dtype, Wr, bias, k):
    """Router for all tokens of x: returns ids [T,k] i32, p [T,k], margin [T], logits [T,E]."""
    Wr = _c(Wr, np.float32)
    E, H = Wr.shape
    xa = _c(x, np.uint16 if x_dtype == X_BF16 else np.float32).reshape(-1, H)
    T = xa.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    ids = np.zeros((T, k), np.int32)
    p = np.zeros((T, k), np.float64)
    margin = np.zeros(T, np.float64)
    logits = np.zeros((T, E), np.float64)
    rc = lib().qso_route(H, E, k, T, _p(xa), x_dtype, _p(Wr), _p(b), _p(ids), _p(p), _p(margin), _p(logits))
    if rc:
        raise ValueError(f"qso_route failed ({rc})")
    return ids, p, margin, logits


def group(ids, E):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    lib().qso_group(E, k, T, _p(ids), _p(counts), _p(offsets), _p(perm))
    return counts, offsets, perm


def expert_gateup(H, F, blob, xw):
    h = np.zeros(F, np.float64)
    lib().qso_expert_gateup(H, F, _p(_c(blob, np.uint8)), _p(_c(xw, np.float64)), _p(h))
    return h


def expert_down(H, F, blob, h):
    y = np.zeros(H, np.float64)
    lib().qso_expert_down(H, F, _p(_c(blob, np.uint8)), _p(_c(h, np.float64)), _p(y))
    return y


def shared_expert(H, S, sh, xw):
    hs = np.zeros(S, np.float64)
    g = np.zeros(1, np.float64)
    y = np.zeros(H, np.float64)
    lib().qso_shared_expert(H, S, _p(_c(sh["gate"], np.uint16)), _p(_c(sh["up"], np.uint16)),
                            _p(_c(sh["down"], np.uint16)), _p(_c(sh["sig"], np.uint16)),
                            _p(_c(xw, np.float64)), _p(hs), _p(g), _p(y))
    return hs, float(g[0]), y


def moe_ffn(shape, x, Wr, bias, experts, expert_stride, shared, tokens=None, threads=1, fmt="q2k"):
    """The whole layer in double precision.

    shape: qs_inputs.LayerShape; x: [T,H] fp32 or bf16 bits; experts: uint8 blob
    (E * expert_stride bytes); shared: dict of bf16 bit arrays or None.
    tokens: optional list of token indices to compute (others left zero).
    threads: >1 splits the tokens over Python threads (the C call releases the GIL).
    Returns dict: ids, p, margin, y, h [T*k,F], hs [T,S], gate [T].
    """
    H, E, k, F, S = shape.hidden, shape.n_experts, shape.top_k, shape.expert_ffn, shape.shared_ffn
    xd = X_BF16 if shape.x_dtype == 1 else X_F32
    xa = _c(x, np.uint16 if xd == X_BF16 else np.float32).reshape(-1, H)
    T = xa.shape[0]
    Wr = _c(Wr, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    ex = _c(experts, np.uint8).reshape(-1)
    if shared is None:
        S = 0
        sg = su = sd = ss = None
    else:
        sg, su, sd, ss = (_c(shared[n], np.uint16) for n in ("gate", "up", "down", "sig"))
    ids = np.zeros((T, k), np.int32)
    p = np.zeros((T, k), np.float64)
    margin = np.zeros(T, np.float64)
    y = np.zeros((T, H), np.float64)
    h = np.zeros((T * k, F), np.float64)
    hs = np.zeros((T, max(S, 1)), np.float64)
    gate = np.zeros(T, np.float64)
    todo = list(range(T)) if tokens is None else sorted(set(int(t) for t in tokens))
    L = lib()

    errors = []

    def run(ts):
        for t in ts:
            rc = L.qso_moe_ffn_fmt(FMT[fmt], H, E, k, F, S, t, 1, _p(xa), xd, _p(Wr), _p(b), _p(ex), expert_stride,
                               _p(sg), _p(su), _p(sd), _p(ss), _p(ids), _p(p), _p(margin), _p(y),
                               _p(h), _p(hs), _p(gate))
            if rc:
                errors.append(rc)
                return

    if threads <= 1 or len(todo) <= 1:
        run(todo)
    else:
        parts = [todo[i::threads] for i in range(threads)]
        ths = [threading.Thread(target=run, args=(pt,)) for pt in parts if pt]
        for th in ths:
            th.start()
        for th in ths:
            th.join()
    if errors:
        raise ValueError(f"qso_moe_ffn failed ({errors[0]})")
    return {"ids": ids, "p": p, "margin": margin, "y": y, "h": h, "hs": hs[:, :S], "gate": gate}


def steer_rows(y, d, scale):
    """Directional steering of FFN output rows, y <- y - scale * d * (d . y), per row.

    QuarkStar (q36) README, "Steering".  y: [T, H] (any float type, widened to
    double); d: [H] fp32 direction (used as given); returns a new [T, H] float64.
    """
    yy = np.array(y, dtype=np.float64, order="C").reshape(-1, np.shape(y)[-1]).copy()
    T, H = yy.shape
    dd = _c(d, np.float32).reshape(-1)
    if dd.shape[0] != H:
        raise ValueError("direction length differs from the row length")
    lib().qso_steer_rows(H, T, _p(dd), float(scale), _p(yy))
    return yy
