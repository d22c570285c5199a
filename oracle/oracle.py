"""ctypes front of the plain C oracle (``q8_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this module.  The CUDA library and its
Python binding never do.

The shared object is compiled on first use with the system C compiler
(``-O2 -ffp-contract=off``, no fast-math, optional OpenMP over output rows)
into ``oracle/_build/``.  Everything here only marshals numpy arrays; the
arithmetic lives in the C file, whose comments cite the passages it follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

QK = 32


def build(force: bool = False) -> str:
    """Compile the oracle shared object if it is missing or stale."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB + f".{os.getpid()}.tmp"
    base = [cc, "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            i64, vp = C.c_int64, C.c_void_p
            sig = {
                "orc_threads": (C.c_int, []),
                "orc_set_threads": (None, [C.c_int]),
                "orc_f16_to_f32": (C.c_float, [C.c_uint16]),
                "orc_f32_to_f16": (C.c_uint16, [C.c_float]),
                "orc_q8_pack": (i64, [vp, i64, i64, vp, vp]),
                "orc_rmsnorm": (None, [vp, vp, i64, i64, C.c_float, vp, vp]),
                "orc_residual_add": (None, [vp, vp, i64, i64, vp]),
                "orc_exp_f32": (C.c_float, [C.c_float]),
                "orc_swiglu": (None, [vp, i64, i64, vp]),
                "orc_kv_write": (i64, [vp, i64, i64, vp, i64, i64, i64, vp, vp]),
                "orc_act_quant_i8": (None, [vp, i64, i64, vp, vp]),
                "orc_act_quant_i8x2": (None, [vp, i64, i64, vp, vp, vp]),
                "orc_block_dots": (None, [vp, vp, vp, i64, i64, i64, vp]),
                "orc_proj_q": (None, [vp, vp, vp, vp, vp, i64, i64, i64, vp, vp]),
                "orc_proj_f64": (None, [vp, vp, vp, i64, i64, i64, vp, vp]),
                "orc_argmax_f32": (None, [vp, i64, i64, vp, vp]),
                "orc_argmax_f64": (None, [vp, i64, i64, vp, vp]),
                "orc_near_tie": (C.c_int, [C.c_double, C.c_double]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def threads() -> int:
    return _load().orc_threads()


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def f16_to_f32(bits: int) -> float:
    return float(_load().orc_f16_to_f32(int(bits)))


def f32_to_f16(v: float) -> int:
    return int(_load().orc_f32_to_f16(float(np.float32(v))))


def f32_to_f16_array(v: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(v, dtype=np.float32).ravel()
    return np.array([lib.orc_f32_to_f16(float(x)) for x in flat], dtype=np.uint16).reshape(np.shape(v))


def q8_pack(w: np.ndarray):
    """Q8_0 pack of f32 weights [N, K] -> (q int8 [N,K], s fp16 bits [N,K/32], overflow)."""
    w = _c(w, np.float32)
    n, k = w.shape
    if k % QK:
        raise ValueError("K must be a multiple of 32")
    q = np.empty((n, k), np.int8)
    s = np.empty((n, k // QK), np.uint16)
    ov = _load().orc_q8_pack(_p(w), n, k, _p(q), _p(s))
    return q, s, int(ov)


def rmsnorm(h: np.ndarray, g: np.ndarray | None = None, eps: float = 1e-5):
    """RMSNorm rows of h -> (x f32 [rows, K], r f64 [rows])."""
    h = _c(h, np.float32)
    rows, k = h.shape
    if g is not None:
        g = _c(g, np.float32)
        if g.shape != (k,):
            raise ValueError("gain must have shape (K,)")
    x = np.empty_like(h)
    r = np.empty(rows, np.float64)
    _load().orc_rmsnorm(_p(h), _p(g), rows, k, float(eps), _p(x), _p(r))
    return x, r


def residual_add(h: np.ndarray, r: np.ndarray):
    """The residual added before the norm: s = h + r (f32, one rounding)."""
    h = _c(h, np.float32)
    r = _c(r, np.float32)
    if h.shape != r.shape:
        raise ValueError("h and r must have the same shape")
    rows, k = h.shape
    s = np.empty_like(h)
    _load().orc_residual_add(_p(h), _p(r), rows, k, _p(s))
    return s


def exp_f32(x: float) -> float:
    """e^x in binary32 by the oracle's one definition (Cody-Waite + Taylor)."""
    return float(_load().orc_exp_f32(float(x)))


def swiglu(gu: np.ndarray):
    """SwiGLU producer input: gu [rows, 2F] (gate | up) -> x f32 [rows, F]."""
    gu = _c(gu, np.float32)
    rows, f2 = gu.shape
    if f2 % 2:
        raise ValueError("gate+up row must have an even length")
    x = np.empty((rows, f2 // 2), np.float32)
    _load().orc_swiglu(_p(gu), rows, f2 // 2, _p(x))
    return x


def kv_write(y: np.ndarray, pos, kv_col: int, d: int, k_cache: np.ndarray, v_cache: np.ndarray):
    """Row m's K/V slices of y into cache row pos[m] (caches [rows, n_pos, d],
    updated in place); returns the number of positions out of range."""
    y = _c(y, np.float32)
    rows, n = y.shape
    pos = _c(np.asarray(pos, dtype=np.int32), np.int32)
    if k_cache.dtype != np.float32 or v_cache.dtype != np.float32:
        raise ValueError("caches must be float32")
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("caches must be contiguous")
    if k_cache.shape != v_cache.shape or k_cache.shape[0] != rows or k_cache.shape[2] != d:
        raise ValueError("caches must be [rows, n_pos, d]")
    if kv_col < 0 or kv_col + 2 * d > n:
        raise ValueError("K/V columns out of the row")
    return int(_load().orc_kv_write(_p(y), rows, n, _p(pos), kv_col, d, k_cache.shape[1],
                                    _p(k_cache), _p(v_cache)))


def act_quant_i8(x: np.ndarray):
    """One int8 word per value -> (xq int8 [rows,K], xd f32 [rows,K/32])."""
    x = _c(x, np.float32)
    rows, k = x.shape
    xq = np.empty((rows, k), np.int8)
    xd = np.empty((rows, k // QK), np.float32)
    _load().orc_act_quant_i8(_p(x), rows, k, _p(xq), _p(xd))
    return xq, xd


def act_quant_i8x2(x: np.ndarray):
    """Two-word 14-bit split -> (xh int8, xl int8, xd f32)."""
    x = _c(x, np.float32)
    rows, k = x.shape
    xh = np.empty((rows, k), np.int8)
    xl = np.empty((rows, k), np.int8)
    xd = np.empty((rows, k // QK), np.float32)
    _load().orc_act_quant_i8x2(_p(x), rows, k, _p(xh), _p(xl), _p(xd))
    return xh, xl, xd


def block_dots(q: np.ndarray, xh: np.ndarray, xl: np.ndarray | None = None):
    """Per-block int32 dots -> isum int32 [rows, N, K/32]."""
    q = _c(q, np.int8)
    xh = _c(xh, np.int8)
    if xl is not None:
        xl = _c(xl, np.int8)
    n, k = q.shape
    rows = xh.shape[0]
    isum = np.empty((rows, n, k // QK), np.int32)
    _load().orc_block_dots(_p(q), _p(xh), _p(xl), n, k, rows, _p(isum))
    return isum


def proj_q(q, s, xh, xl, xd):
    """Modes one-word (xl None) / two-word projection -> (y f32 [rows,N], norm f64)."""
    q = _c(q, np.int8)
    s = _c(s, np.uint16)
    xh = _c(xh, np.int8)
    if xl is not None:
        xl = _c(xl, np.int8)
    xd = _c(xd, np.float32)
    n, k = q.shape
    rows = xh.shape[0]
    y = np.empty((rows, n), np.float32)
    norm = np.empty((rows, n), np.float64)
    _load().orc_proj_q(_p(q), _p(s), _p(xh), _p(xl), _p(xd), n, k, rows, _p(y), _p(norm))
    return y, norm


def proj_f64(q, s, x):
    """f32 activations, f64 sums -> (y f64 [rows,N], norm f64)."""
    q = _c(q, np.int8)
    s = _c(s, np.uint16)
    x = _c(x, np.float32)
    n, k = q.shape
    rows = x.shape[0]
    y = np.empty((rows, n), np.float64)
    norm = np.empty((rows, n), np.float64)
    _load().orc_proj_f64(_p(q), _p(s), _p(x), n, k, rows, _p(y), _p(norm))
    return y, norm


def argmax(logits: np.ndarray):
    """Row arg-max with the lowest index on ties -> (tok int32, best value).
    NaN logits are no candidates; a row of NaN only gives index 0, value NaN."""
    logits = np.ascontiguousarray(logits)
    rows, n = logits.shape
    tok = np.empty(rows, np.int32)
    if logits.dtype == np.float32:
        best = np.empty(rows, np.float32)
        _load().orc_argmax_f32(_p(logits), rows, n, _p(tok), _p(best))
    elif logits.dtype == np.float64:
        best = np.empty(rows, np.float64)
        _load().orc_argmax_f64(_p(logits), rows, n, _p(tok), _p(best))
    else:
        raise TypeError("logits must be f32 or f64")
    return tok, best


# Relative distance from an f32 rounding boundary within which the RMS scale r
# of a row is a "near tie": the oracle's own sequential f64 sum of squares is
# accurate to about 2^-42 relative at K <= 16384, and the library evaluates r
# to about 2^-44, so either may round r to the other f32 neighbour there.
NEAR_TIE_REL = 2.0 ** -40


def near_tie(r, rel: float = NEAR_TIE_REL) -> np.ndarray:
    """Per row: whether the f64 RMS scale r lies within rel * r of an f32
    rounding boundary (see orc_near_tie)."""
    lib = _load()
    rr = np.atleast_1d(np.asarray(r, dtype=np.float64))
    return np.array([bool(lib.orc_near_tie(float(v), float(rel))) for v in rr], dtype=bool)


# ----------------------------------------------------------------- compositions
# Mode names follow the lane's CudaKnobs: "f32" (f32 activations, f64 sums),
# "i8" (one int8 word), "i8x2" (two-word ~14-bit).

def quantize(mode: str, x: np.ndarray):
    """Producer output for a mode: f32 -> (x,), i8 -> (xq, xd), i8x2 -> (xh, xl, xd)."""
    if mode == "f32":
        return (np.ascontiguousarray(x, dtype=np.float32),)
    if mode == "i8":
        return act_quant_i8(x)
    if mode == "i8x2":
        return act_quant_i8x2(x)
    raise ValueError(mode)


def project(mode: str, q, s, act):
    """Projection of an already-quantised activation tuple (see quantize)."""
    if mode == "f32":
        return proj_f64(q, s, act[0])
    if mode == "i8":
        xq, xd = act
        return proj_q(q, s, xq, None, xd)
    if mode == "i8x2":
        xh, xl, xd = act
        return proj_q(q, s, xh, xl, xd)
    raise ValueError(mode)


def head_argmax(mode: str, q, s, act):
    """LM head product followed by the row arg-max -> (tok, best, logits)."""
    y, _ = project(mode, q, s, act)
    tok, best = argmax(y)
    return tok, best, y
