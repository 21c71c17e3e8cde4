"""CPU oracle for the fused 4-bit block-quantized GEMV (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (``skinny_gemm_q4_gb300``)
never imports it, and the two share no code: the oracle is plain C in
``oracle.c`` (decode each block in float64, round once to float32, then a
float64 dot in increasing k), wrapped here with ``ctypes``.

The shared library is compiled with gcc on first use (or by ``build()``) into
``oracle/_build/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q4_K = 12
Q5_K = 13
Q6_K = 14
NVFP4 = 256
FP8 = 257

BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "oracle.c")]
_HDR = os.path.join(_HERE, "oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags only: it runs on x86-64
    and on aarch64).  Returns the path of the shared library."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(p) for p in _SRC + [_HDR])
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add contraction, so every float64
    # operation rounds exactly as written.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp] + _SRC + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, f32, i32 = ctypes.c_int64, ctypes.c_float, ctypes.c_int
        vp = ctypes.c_void_p
        lib.or_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.or_f16_to_f64.restype = ctypes.c_double
        lib.or_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_to_f64.restype = ctypes.c_double
        lib.or_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.or_e2m1_to_f64.restype = ctypes.c_double
        lib.or_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.or_bf16_to_f64.restype = ctypes.c_double
        lib.or_row_bytes.argtypes = [i32, i64]
        lib.or_row_bytes.restype = i64
        lib.or_unpack_scale_min.argtypes = [vp, i32, vp, vp]
        lib.or_unpack_scale_min.restype = None
        lib.or_dequant_rows.argtypes = [i32, vp, vp, f32, i64, i64, vp, i64, vp]
        lib.or_dequant_rows.restype = i32
        lib.or_qgemv_rows.argtypes = [i32, vp, vp, f32, i64, i64, vp, i64, vp, i64,
                                      vp, vp, vp, vp]
        lib.or_qgemv_rows.restype = i32
        lib.or_silu.argtypes = [ctypes.c_double]
        lib.or_silu.restype = ctypes.c_double
        lib.or_swiglu.argtypes = [vp, vp, i64, vp]
        lib.or_swiglu.restype = None
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def _bytes(a):
    """The raw bytes of an array (FP8 bf16 scales may come as uint16 bits)."""
    a = np.ascontiguousarray(a)
    return a.view(np.uint8) if a.dtype.itemsize > 1 else a.astype(np.uint8, copy=False)


def _f16bits(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    return np.ascontiguousarray(a, dtype=np.uint16)


def row_bytes(qtype: int, K: int) -> int:
    return int(_load().or_row_bytes(qtype, K))


def f16_to_f64(bits: int) -> float:
    return _load().or_f16_to_f64(bits)


def e4m3_to_f64(code: int) -> float:
    return _load().or_e4m3_to_f64(code)


def e2m1_to_f64(code: int) -> float:
    return _load().or_e2m1_to_f64(code)


def bf16_to_f64(bits: int) -> float:
    return _load().or_bf16_to_f64(bits)


def unpack_scale_min(scales12, s: int):
    """(sc, m) of sub-block s from the 12 packed bytes of a Q4_K/Q5_K block."""
    b = _u8(scales12)
    sc = ctypes.c_int()
    m = ctypes.c_int()
    _load().or_unpack_scale_min(_ptr(b), s, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def dequantize(qtype: int, w, M: int, K: int, scales=None, global_scale: float = 1.0,
               rows=None) -> np.ndarray:
    """Decode W (packed bytes, row-major) to float32 [len(rows) or M][K]."""
    w = _u8(w)
    sc = None if scales is None else _bytes(scales)
    if rows is None:
        nrows, rptr, ra = M, None, None
    else:
        ra = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rptr = ra.size, _ptr(ra)
    out = np.empty((nrows, K), dtype=np.float32)
    rc = _load().or_dequant_rows(qtype, _ptr(w), _ptr(sc), global_scale, M, K, rptr,
                                 nrows, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle dequantize failed (rc={rc})")
    return out


def qgemv(qtype: int, w, M: int, K: int, x, scales=None, global_scale: float = 1.0,
          residual=None, rows=None):
    """The whole path on selected rows: y, mag (float64 [N][len(rows)])."""
    w = _u8(w)
    sc = None if scales is None else _bytes(scales)
    xb = _f16bits(x).reshape(-1, K)
    N = xb.shape[0]
    if rows is None:
        nrows, rptr, ra = M, None, None
    else:
        ra = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rptr = ra.size, _ptr(ra)
    rb = None if residual is None else _f16bits(residual).reshape(N, M)
    y = np.empty((N, nrows), dtype=np.float64)
    mag = np.empty((N, nrows), dtype=np.float64)
    scratch = np.empty(K, dtype=np.float32)
    rc = _load().or_qgemv_rows(qtype, _ptr(w), _ptr(sc), global_scale, M, K, rptr, nrows,
                               _ptr(xb), N, _ptr(rb), _ptr(y), _ptr(mag), _ptr(scratch))
    if rc != 0:
        raise ValueError(f"oracle qgemv failed (rc={rc})")
    return y, mag


def silu(v: float) -> float:
    """silu(v) = v / (1 + exp(-v)) in float64 (reflex-llm "docs/kernels.md",
    SwiGLU section)."""
    return float(_load().or_silu(float(v)))


def swiglu(g, u) -> np.ndarray:
    """h = silu(g) * u elementwise in float64 (g, u: the oracle's float64
    gate and up products for the same x)."""
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    if g.shape != u.shape:
        raise ValueError("gate and up shapes differ")
    h = np.empty_like(g)
    _load().or_swiglu(_ptr(g), _ptr(u), g.size, _ptr(h))
    return h


def qgemv_swiglu(qtype_g: int, wg, qtype_u: int, wu, M: int, K: int, x, rows=None,
                 scales_g=None, gscale_g: float = 1.0, scales_u=None, gscale_u: float = 1.0):
    """The fused pair: h = silu(x.Wg^T) * (x.Wu^T) on selected rows, plus
    both products and their magnitudes: (h, g, mag_g, u, mag_u), float64
    [N][len(rows)]."""
    g, mg = qgemv(qtype_g, wg, M, K, x, scales=scales_g, global_scale=gscale_g, rows=rows)
    u, mu = qgemv(qtype_u, wu, M, K, x, scales=scales_u, global_scale=gscale_u, rows=rows)
    return swiglu(g, u), g, mg, u, mu
