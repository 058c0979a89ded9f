"""CPU oracle for the small-M NVFP4 W4A4 linear -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never loads it, and it shares
no code with the CUDA library: the arithmetic lives in ``nvfp4_oracle.c``
(plain C, FP32 quantisation decisions, FP64 accumulation), which this module
compiles with gcc on first use and calls through ctypes.

What each function follows is stated in ``nvfp4_oracle.c``'s header: the
operation is the W4A4 decode linear of "ReSET: Accurate Latency-Critical NVFP4
Reasoning via Step-Aware Temperature Scaling" (abstract; README "Core
components" item 2), with the NVFP4 bit formats read as OCP FP4 E2M1 and FP8
E4M3 with one E4M3 scale per 16 elements and an FP32 tensor scale.

Pins: every function here is checked against values fixed by something other
than itself (closed forms, a library float8 decode, brute force, invariants)
in ``tests/test_oracle_pins.py``.  Parity is pinned for all functions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile ``nvfp4_oracle.c`` into ``liboracle.so`` (gcc, IEEE FP32, no contraction)."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_e2m1_value.argtypes = [ctypes.c_int]
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_int]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_encode.restype = ctypes.c_int
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_int
        lib.oracle_amax.argtypes = [_f32p, _i64]
        lib.oracle_amax.restype = ctypes.c_float
        lib.oracle_global_scale.argtypes = [_f32p, _i64]
        lib.oracle_global_scale.restype = ctypes.c_float
        lib.oracle_quantize.argtypes = [_f32p, _i64, _i64, ctypes.c_float, _u8p, _u8p]
        lib.oracle_quantize.restype = None
        lib.oracle_pack_weight.argtypes = [_f32p, _i64, _i64, _u8p, _u8p, _f32p]
        lib.oracle_pack_weight.restype = None
        lib.oracle_dequantize.argtypes = [_u8p, _u8p, ctypes.c_float, _i64, _i64, _f64p]
        lib.oracle_dequantize.restype = None
        lib.oracle_gemm.argtypes = [_u8p, _u8p, ctypes.c_float, _u8p, _u8p, ctypes.c_float,
                                    _i64, _i64, _i64, _f64p]
        lib.oracle_gemm.restype = None
        lib.oracle_gemm_sampled.argtypes = [_u8p, _u8p, ctypes.c_float, _u8p, _u8p,
                                            ctypes.c_float, _i64, _i64p, _i64p, _i64, _f64p]
        lib.oracle_gemm_sampled.restype = None
        lib.oracle_bf16_widen.argtypes = [_u16p, _i64, _f32p]
        lib.oracle_bf16_widen.restype = None
        lib.oracle_bf16_round.argtypes = [_f32p, _i64, _u16p]
        lib.oracle_bf16_round.restype = None
        _lib = lib
        return lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


# ---- element formats --------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e2m1_encode(v: float) -> int:
    return _load().oracle_e2m1_encode(float(v))


def e4m3_encode(s: float) -> int:
    return _load().oracle_e4m3_encode(float(s))


# ---- tensors -----------------------------------------------------------------

def amax(t) -> np.float32:
    t = _f32(t).reshape(-1)
    return np.float32(_load().oracle_amax(t, t.size))


def global_scale(t) -> np.float32:
    """g = amax(|t|) / (6 * 448) in FP32."""
    t = _f32(t).reshape(-1)
    return np.float32(_load().oracle_global_scale(t, t.size))


def quantize(t, g) -> tuple[np.ndarray, np.ndarray]:
    """Quantise rows of ``t`` [rows, k] with tensor scale ``g``.

    Returns (q uint8 [rows, k/2], s uint8 [rows, k/16])."""
    t = _f32(t)
    rows, k = t.shape
    if k % 16:
        raise ValueError("k must be a multiple of 16")
    q = np.zeros((rows, k // 2), np.uint8)
    s = np.zeros((rows, k // 16), np.uint8)
    _load().oracle_quantize(t, rows, k, float(np.float32(g)), q, s)
    return q, s


def pack_weight(w) -> tuple[np.ndarray, np.ndarray, np.float32]:
    """Weight packing: (wq [n, k/2], ws [n, k/16], gw = amax/2688)."""
    w = _f32(w)
    n, k = w.shape
    if k % 16:
        raise ValueError("k must be a multiple of 16")
    q = np.zeros((n, k // 2), np.uint8)
    s = np.zeros((n, k // 16), np.uint8)
    g = np.zeros(1, np.float32)
    _load().oracle_pack_weight(w, n, k, q, s, g)
    return q, s, np.float32(g[0])


def dequantize(q, s, g) -> np.ndarray:
    q = _u8(q)
    s = _u8(s)
    rows = q.shape[0]
    k = q.shape[1] * 2
    out = np.zeros((rows, k), np.float64)
    _load().oracle_dequantize(q, s, float(np.float32(g)), rows, k, out)
    return out


def gemm(xq, xs, gx, wq, ws, gw) -> np.ndarray:
    """FP64 y[m, n] from the packed operands."""
    xq, xs, wq, ws = _u8(xq), _u8(xs), _u8(wq), _u8(ws)
    m, n, k = xq.shape[0], wq.shape[0], xq.shape[1] * 2
    if wq.shape[1] * 2 != k:
        raise ValueError("K mismatch")
    y = np.zeros((m, n), np.float64)
    _load().oracle_gemm(xq, xs, float(np.float32(gx)), wq, ws, float(np.float32(gw)),
                        m, n, k, y)
    return y


def gemm_sampled(xq, xs, gx, wq, ws, gw, ms, ns) -> np.ndarray:
    """FP64 y at the (ms[t], ns[t]) positions only."""
    xq, xs, wq, ws = _u8(xq), _u8(xs), _u8(wq), _u8(ws)
    k = xq.shape[1] * 2
    ms = np.ascontiguousarray(ms, np.int64)
    ns = np.ascontiguousarray(ns, np.int64)
    y = np.zeros(ms.size, np.float64)
    _load().oracle_gemm_sampled(xq, xs, float(np.float32(gx)), wq, ws, float(np.float32(gw)),
                                k, ms, ns, ms.size, y)
    return y


# ---- BF16 (production activation / output dtype) ----------------------------

def bf16_to_f32(bits) -> np.ndarray:
    """BF16 bit patterns (uint16 array) -> FP32 values, exact."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    _load().oracle_bf16_widen(b.reshape(-1), b.size, out.reshape(-1))
    return out


def f32_to_bf16(v) -> np.ndarray:
    """FP32 values -> BF16 bit patterns, round to nearest, ties to even."""
    f = _f32(v)
    out = np.empty(f.shape, dtype=np.uint16)
    _load().oracle_bf16_round(f.reshape(-1), f.size, out.reshape(-1))
    return out

