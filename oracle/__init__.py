"""CPU oracle for the h3fp4 NVFP4 linear path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library (``audio_dit_gb300``) never
imports it and shares no code with it.

The arithmetic lives in ``h3fp4_oracle.c`` (strict IEEE C, float64 GEMM); this
module compiles it with gcc on first use and marshals numpy arrays through
ctypes.  See the header of ``h3fp4_oracle.c`` for the passages each function
follows and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "h3fp4_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liborc_h3fp4.so")
CFLAGS = ["-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
          "-fPIC", "-shared", "-Wall"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (strict fp32, no contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class LinearArgs(C.Structure):
    _fields_ = [
        ("a_codes", C.c_void_p), ("a_sf", C.c_void_p), ("a_gs", C.c_float),
        ("w_codes", C.c_void_p), ("w_sf", C.c_void_p), ("w_gs", C.c_float),
        ("M", C.c_int64), ("N", C.c_int64), ("K", C.c_int64),
        ("bias", C.c_void_p), ("gate", C.c_void_p), ("resid", C.c_void_p),
        ("seg_off", C.c_void_p), ("nseg", C.c_int),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            i64, f32, f64, vp = C.c_int64, C.c_float, C.c_double, C.c_void_p
            sig = {
                "orc_bf16_from_float": (C.c_uint16, [f32]),
                "orc_bf16_to_float": (f32, [C.c_uint16]),
                "orc_e2m1_decode": (f64, [C.c_uint8]),
                "orc_e2m1_encode": (C.c_uint8, [f32]),
                "orc_e4m3_decode": (f64, [C.c_uint8]),
                "orc_e4m3_encode": (C.c_uint8, [f32]),
                "orc_e2m1_encode_array": (None, [vp, i64, vp]),
                "orc_e4m3_encode_array": (None, [vp, i64, vp]),
                "orc_sf_cols4": (i64, [i64]),
                "orc_sf_bytes": (i64, [i64, i64]),
                "orc_sf_offset": (i64, [i64, i64, i64]),
                "orc_modulate": (None, [vp, i64, i64, vp, vp, vp, C.c_int, vp]),
                "orc_amax": (f32, [vp, i64]),
                "orc_global_scale": (f32, [f32]),
                "orc_quantize_block": (C.c_uint8, [vp, f32, vp]),
                "orc_quantize": (None, [vp, i64, i64, vp, vp, vp, C.c_int, C.c_int, vp, vp, vp]),
                "orc_dequantize": (None, [vp, vp, f32, i64, i64, vp]),
                "orc_linear_points": (None, [C.POINTER(LinearArgs), vp, i64, vp, vp]),
                "orc_linear_full": (None, [C.POINTER(LinearArgs), vp, vp]),
                "orc_gemm_f64": (None, [vp, vp, i64, i64, i64, vp]),
                "orc_num_threads": (C.c_int, []),
                "orc_swiglu_bf16": (C.c_uint16, [C.c_uint16, C.c_uint16]),
                "orc_swiglu_rows": (None, [vp, i64, i64, vp]),
                "orc_silu_mul_f64": (None, [vp, vp, i64, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalars

def bf16_from_float(f: float) -> int:
    return int(lib().orc_bf16_from_float(f))


def bf16_to_float(h: int) -> float:
    return float(lib().orc_bf16_to_float(h))


def e2m1_decode(c: int) -> float:
    return float(lib().orc_e2m1_decode(c))


def e2m1_encode(f: float) -> int:
    return int(lib().orc_e2m1_encode(f))


def e4m3_decode(c: int) -> float:
    return float(lib().orc_e4m3_decode(c))


def e4m3_encode(f: float) -> int:
    return int(lib().orc_e4m3_encode(f))


def global_scale(amax: float) -> float:
    return float(lib().orc_global_scale(amax))


def sf_bytes(rows: int, K: int) -> int:
    return int(lib().orc_sf_bytes(rows, K))


def sf_offset(r: int, c: int, K: int) -> int:
    return int(lib().orc_sf_offset(r, c, K))


def num_threads() -> int:
    return int(lib().orc_num_threads())


# ---------------------------------------------------------------- arrays

def e2m1_encode_array(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e2m1_encode_array(_p(x), x.size, _p(out))
    return out


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def quantize_block(m16: np.ndarray, s_g: float):
    """One 16-element block -> (E4M3 scale code, 16 E2M1 codes)."""
    m16 = _c(m16, np.float32)
    assert m16.size == 16
    q = np.empty(16, np.uint8)
    S = lib().orc_quantize_block(_p(m16), s_g, _p(q))
    return int(S), q


def _segs(seg_off, rows):
    if seg_off is None:
        seg_off = [0, rows]
    so = np.ascontiguousarray(seg_off, dtype=np.int64)
    return so, len(so) - 1


def modulate(x_bf16, shift=None, scale=None, seg_off=None):
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    so, nseg = _segs(seg_off, M)
    out = np.empty_like(x)
    lib().orc_modulate(_p(x), M, K, _p(_c(shift, np.float32)), _p(_c(scale, np.float32)),
                       _p(so), nseg, _p(out))
    return out


def amax(m_bf16) -> float:
    m = _c(m_bf16, np.uint16)
    return float(lib().orc_amax(_p(m), m.size))


def quantize(x_bf16, shift=None, scale=None, seg_off=None, gscale=None):
    """Quantise a [rows, K] bf16 (uint16 bit pattern) operand.

    Returns (codes uint8 [rows, K/2], sf uint8 [sf_bytes], global scale float).
    ``gscale`` given -> used as-is (the caller-supplied global scale mode).
    """
    x = _c(x_bf16, np.uint16)
    rows, K = x.shape
    assert K % 16 == 0
    so, nseg = _segs(seg_off, rows)
    codes = np.empty((rows, K // 2), np.uint8)
    sf = np.empty(sf_bytes(rows, K), np.uint8)
    gs = np.array([0.0 if gscale is None else gscale], np.float32)
    lib().orc_quantize(_p(x), rows, K, _p(_c(shift, np.float32)), _p(_c(scale, np.float32)),
                       _p(so), nseg, 0 if gscale is None else 1, _p(gs), _p(codes), _p(sf))
    return codes, sf, float(gs[0])


def dequantize(codes, sf, gscale, rows, K) -> np.ndarray:
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    out = np.empty((rows, K), np.float64)
    lib().orc_dequantize(_p(codes), _p(sf), gscale, rows, K, _p(out))
    return out


def _linear_args(a, w, M, N, K, bias, gate, resid, seg_off, keep):
    (a_codes, a_sf, a_gs), (w_codes, w_sf, w_gs) = a, w
    so, nseg = _segs(seg_off, M)
    arrs = [_c(a_codes, np.uint8), _c(a_sf, np.uint8), _c(w_codes, np.uint8), _c(w_sf, np.uint8),
            _c(bias, np.uint16), _c(gate, np.float32), _c(resid, np.uint16), so]
    keep.extend(arrs)
    return LinearArgs(_p(arrs[0]), _p(arrs[1]), a_gs, _p(arrs[2]), _p(arrs[3]), w_gs,
                      M, N, K, _p(arrs[4]), _p(arrs[5]), _p(arrs[6]), _p(arrs[7]), nseg)


def linear_full(a, w, M, N, K, bias=None, gate=None, resid=None, seg_off=None):
    """Every output of out = R + g*(alpha*A_q W_q^T + b) in float64, with its bound.

    a, w: (codes, sf, gscale) triples from :func:`quantize`.
    """
    keep = []
    args = _linear_args(a, w, M, N, K, bias, gate, resid, seg_off, keep)
    out = np.empty((M, N), np.float64)
    bound = np.empty((M, N), np.float64)
    lib().orc_linear_full(C.byref(args), _p(out), _p(bound))
    return out, bound


def linear_points(a, w, M, N, K, points, bias=None, gate=None, resid=None, seg_off=None):
    """Selected outputs (points: int64 [n, 2] of (m, n)) and their bounds."""
    keep = []
    args = _linear_args(a, w, M, N, K, bias, gate, resid, seg_off, keep)
    pts = np.ascontiguousarray(points, dtype=np.int64)
    out = np.empty(len(pts), np.float64)
    bound = np.empty(len(pts), np.float64)
    lib().orc_linear_points(C.byref(args), _p(pts), len(pts), _p(out), _p(bound))
    return out, bound


def swiglu_bf16(g: int, u: int) -> int:
    """bf16(silu(g) * u) for bf16 bit patterns g, u (gate and up FC1 outputs)."""
    return int(lib().orc_swiglu_bf16(g, u))


def swiglu_rows(y_bf16) -> np.ndarray:
    """SwiGLU over an FC1 output in the 256-column [gate 128 | up 128] group
    layout: y uint16 [rows, 2H] -> h uint16 [rows, H]."""
    y = _c(y_bf16, np.uint16)
    rows, n2 = y.shape
    assert n2 % 256 == 0
    h = np.empty((rows, n2 // 2), np.uint16)
    lib().orc_swiglu_rows(_p(y), rows, n2 // 2, _p(h))
    return h


def silu_mul_f64(g, u) -> np.ndarray:
    """silu(g) * u in float64 for float64 arrays g, u (no bf16 rounding)."""
    g = _c(g, np.float64).ravel()
    u = _c(u, np.float64).ravel()
    assert g.shape == u.shape
    out = np.empty(g.size, np.float64)
    lib().orc_silu_mul_f64(_p(g), _p(u), g.size, _p(out))
    return out


def gemm_f64(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    a = _c(a, np.float64)
    w = _c(w, np.float64)
    M, K = a.shape
    N = w.shape[0]
    c = np.empty((M, N), np.float64)
    lib().orc_gemm_f64(_p(a), _p(w), M, N, K, _p(c))
    return c
