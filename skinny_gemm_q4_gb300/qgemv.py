"""Thin ctypes binding of the qgemv C ABI (include/qgemv.h).

Argument marshalling only: every step of the product runs in the CUDA library
``_build/libqgemv.so``.  If the library is missing this module raises; there
is no CPU or PyTorch fallback.

The module-level functions carry the C names and take raw pointers/ints.
``QGemv`` is a convenience wrapper that takes torch CUDA tensors, keeps the
borrowed weight tensors alive and passes ``torch.cuda.current_stream()``.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libqgemv.so")

Q4_K = 12
Q5_K = 13
Q6_K = 14
NVFP4_W4A16 = 256
FP8_E4M3 = 257

OUT_F16 = 0
OUT_F32 = 1

FLAG_FORCE_REFERENCE = 1
FLAG_DEBUG_SYNC = 2
FLAG_NO_FALLBACK = 4
FLAG_MMA_SYNC_PREFILL = 8

OK = 0
STATUS_NAMES = {0: "QG_OK", -1: "QG_EINVAL", -2: "QG_EUNSUPPORTED", -3: "QG_EALIGN",
                -4: "QG_ECUDA", -5: "QG_ENOMEM", -6: "QG_EFAULT_INJECTED"}

#: every symbol include/qgemv.h declares
EXPORTS = ["qgemv_create", "qgemv_run", "qgemv_run_add", "qgemv_pair_run", "qgemv_triple_run",
           "qgemv_run_host", "qgemv_dequantize", "qgemv_destroy", "qgemv_last_error",
           "qgemv_row_bytes", "qgemv_plan_info", "qgemv_describe", "qgemv_device_status",
           "qgemv_run_noalloc", "qgemv_pair_swiglu_run", "qgemv_chain_create",
           "qgemv_chain_run", "qgemv_chain_status", "qgemv_chain_destroy",
           "qgemv_chain_run_host"]

CHAIN_PERSISTENT = 1

CALL_RUN = 0
CALL_RUN_ADD = 1
CALL_PAIR = 2
CALL_TRIPLE = 3


class QgOpts(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_uint32), ("max_tokens", ctypes.c_int32)]


class QgCall(ctypes.Structure):
    """struct qg_call (one call of a decode chain)."""
    _fields_ = [("kind", ctypes.c_int32), ("out_dtype", ctypes.c_int32), ("N", ctypes.c_int64),
                ("h", ctypes.c_void_p * 3), ("x", ctypes.c_void_p),
                ("residual", ctypes.c_void_p), ("y", ctypes.c_void_p * 3)]


class QgemvError(RuntimeError):
    def __init__(self, status: int, what: str, message: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqgemv.so (built by ``skinny_gemm_q4_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is not built; run "
                           "`python -m skinny_gemm_q4_gb300.build` first")
    lib = ctypes.CDLL(path)
    vp, i64, i32, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
    lib.qgemv_create.argtypes = [ctypes.POINTER(vp), c_int, i64, i64, vp, vp, ctypes.c_float,
                                 ctypes.POINTER(QgOpts)]
    lib.qgemv_run.argtypes = [vp, vp, i64, vp, c_int, vp]
    lib.qgemv_run_add.argtypes = [vp, vp, i64, vp, vp, vp]
    lib.qgemv_pair_run.argtypes = [vp, vp, vp, i64, vp, vp, c_int, vp]
    lib.qgemv_triple_run.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, c_int, vp]
    lib.qgemv_run_host.argtypes = [vp, vp, i64, vp, c_int, vp]
    lib.qgemv_dequantize.argtypes = [vp, vp, vp]
    lib.qgemv_destroy.argtypes = [vp]
    lib.qgemv_destroy.restype = None
    lib.qgemv_last_error.argtypes = []
    lib.qgemv_last_error.restype = ctypes.c_char_p
    lib.qgemv_row_bytes.argtypes = [c_int, i64]
    lib.qgemv_row_bytes.restype = i64
    lib.qgemv_plan_info.argtypes = [vp, i64, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                    ctypes.POINTER(i32)]
    lib.qgemv_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), c_int]
    lib.qgemv_describe.argtypes = []
    lib.qgemv_describe.restype = ctypes.c_char_p
    lib.qgemv_run_noalloc.argtypes = [c_int, i64, i64, vp, vp, ctypes.c_float, vp, i64, vp, c_int,
                                      vp]
    lib.qgemv_pair_swiglu_run.argtypes = [vp, vp, vp, i64, vp, c_int, vp]
    lib.qgemv_chain_create.argtypes = [ctypes.POINTER(vp), ctypes.c_uint32]
    lib.qgemv_chain_run.argtypes = [vp, ctypes.POINTER(QgCall), i32, vp]
    lib.qgemv_chain_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), c_int]
    sz = ctypes.c_size_t
    lib.qgemv_chain_run_host.argtypes = [vp, ctypes.POINTER(QgCall), i32, vp, vp, sz, vp, vp, sz,
                                         vp]
    lib.qgemv_chain_destroy.argtypes = [vp]
    lib.qgemv_chain_destroy.restype = None
    for name in ("qgemv_create", "qgemv_run", "qgemv_run_add", "qgemv_pair_run",
                 "qgemv_triple_run", "qgemv_run_host", "qgemv_dequantize", "qgemv_plan_info",
                 "qgemv_device_status", "qgemv_run_noalloc", "qgemv_pair_swiglu_run",
                 "qgemv_chain_create", "qgemv_chain_run", "qgemv_chain_status",
                 "qgemv_chain_run_host"):
        getattr(lib, name).restype = c_int
    _lib = lib
    return lib


# ----------------------------------------------------------- C-named calls

def qgemv_last_error() -> str:
    return load().qgemv_last_error().decode()


def _check(status: int, what: str):
    if status != OK:
        raise QgemvError(status, what, qgemv_last_error())


def qgemv_row_bytes(qtype: int, K: int) -> int:
    return int(load().qgemv_row_bytes(qtype, K))


def qgemv_describe() -> str:
    return load().qgemv_describe().decode()


def qgemv_create(qtype: int, M: int, K: int, w_ptr: int, scales_ptr: int = 0,
                 global_scale: float = 1.0, flags: int = 0, max_tokens: int = 0) -> int:
    h = ctypes.c_void_p()
    opts = QgOpts(flags, max_tokens)
    _check(load().qgemv_create(ctypes.byref(h), qtype, M, K, w_ptr or None, scales_ptr or None,
                               global_scale, ctypes.byref(opts)), "qgemv_create")
    return h.value


def qgemv_destroy(h: int):
    if h:
        load().qgemv_destroy(h)


def qgemv_run(h, x_ptr, N, y_ptr, ydt, stream):
    _check(load().qgemv_run(h, x_ptr, N, y_ptr, ydt, stream), "qgemv_run")


def qgemv_run_add(h, x_ptr, N, res_ptr, y_ptr, stream):
    _check(load().qgemv_run_add(h, x_ptr, N, res_ptr, y_ptr, stream), "qgemv_run_add")


def qgemv_pair_run(a, b, x_ptr, N, ya, yb, ydt, stream):
    _check(load().qgemv_pair_run(a, b, x_ptr, N, ya, yb, ydt, stream), "qgemv_pair_run")


def qgemv_triple_run(a, b, c, x_ptr, N, ya, yb, yc, ydt, stream):
    _check(load().qgemv_triple_run(a, b, c, x_ptr, N, ya, yb, yc, ydt, stream),
           "qgemv_triple_run")


def qgemv_pair_swiglu_run(gate, up, x_ptr, N, h_ptr, hdt, stream):
    _check(load().qgemv_pair_swiglu_run(gate, up, x_ptr, N, h_ptr, hdt, stream),
           "qgemv_pair_swiglu_run")


def qgemv_run_host(h, x_host_ptr, N, y_host_ptr, ydt, stream):
    _check(load().qgemv_run_host(h, x_host_ptr, N, y_host_ptr, ydt, stream), "qgemv_run_host")


def qgemv_dequantize(h, w_out_ptr, stream):
    _check(load().qgemv_dequantize(h, w_out_ptr, stream), "qgemv_dequantize")


def qgemv_plan_info(h, N):
    ks, rows, launches = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load().qgemv_plan_info(h, N, ctypes.byref(ks), ctypes.byref(rows),
                                  ctypes.byref(launches)), "qgemv_plan_info")
    return ks.value, rows.value, launches.value


def qgemv_device_status(h, clear: bool = False) -> int:
    """The handle's device error word (h = None: qgemv_run_noalloc's, on the
    current device)."""
    w = ctypes.c_uint32()
    _check(load().qgemv_device_status(h, ctypes.byref(w), 1 if clear else 0),
           "qgemv_device_status")
    return w.value


def qgemv_run_noalloc(qtype, M, K, w_ptr, scales_ptr, global_scale, x_ptr, N, y_ptr, ydt,
                      stream):
    """Allocation-free product (no handle; scratch in a fixed device array)."""
    _check(load().qgemv_run_noalloc(qtype, M, K, w_ptr or None, scales_ptr or None, global_scale,
                                    x_ptr or None, N, y_ptr or None, ydt, stream),
           "qgemv_run_noalloc")


def qgemv_chain_create(flags: int = 0) -> int:
    c = ctypes.c_void_p()
    _check(load().qgemv_chain_create(ctypes.byref(c), flags), "qgemv_chain_create")
    return c.value


def qgemv_chain_run(c, calls, stream):
    """calls: a QgCall array (see make_calls)."""
    _check(load().qgemv_chain_run(c, calls, len(calls), stream), "qgemv_chain_run")


def qgemv_chain_run_host(c, calls, in_host, in_dev, in_bytes, out_dev, out_host, out_bytes,
                         stream):
    """One step with host inputs and outputs (raw pointers); synchronizes."""
    _check(load().qgemv_chain_run_host(c, calls, len(calls), in_host or None, in_dev or None,
                                       in_bytes, out_dev or None, out_host or None, out_bytes,
                                       stream), "qgemv_chain_run_host")


def qgemv_chain_status(c, clear: bool = False) -> int:
    w = ctypes.c_uint32()
    _check(load().qgemv_chain_status(c, ctypes.byref(w), 1 if clear else 0), "qgemv_chain_status")
    return w.value


def qgemv_chain_destroy(c):
    if c:
        load().qgemv_chain_destroy(c)


def make_calls(specs):
    """QgCall array from (kind, handles, x_ptr, N, ys, out_dtype, residual_ptr)
    tuples (raw pointers and handle values)."""
    arr = (QgCall * len(specs))()
    for i, (kind, hs, x, N, ys, odt, res) in enumerate(specs):
        c = arr[i]
        c.kind, c.out_dtype, c.N, c.x, c.residual = kind, odt, N, x, res or None
        for j, h in enumerate(hs):
            c.h[j] = h
        for j, y in enumerate(ys):
            c.y[j] = y
    return arr


# ----------------------------------------------------- torch convenience

def _stream_ptr(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class QGemv:
    """One weight matrix on the device (borrowed torch uint8 tensors)."""

    def __init__(self, qtype: int, M: int, K: int, w, scales=None, global_scale: float = 1.0,
                 flags: int = 0, max_tokens: int = 0):
        self.qtype, self.M, self.K = qtype, M, K
        self._w, self._scales = w, scales      # keep the borrowed buffers alive
        self.h = qgemv_create(qtype, M, K, w.data_ptr(),
                              scales.data_ptr() if scales is not None else 0,
                              global_scale, flags, max_tokens)

    def close(self):
        if getattr(self, "h", None):
            qgemv_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _y(self, N, out_f32, y):
        import torch
        if y is None:
            y = torch.empty((N, self.M), dtype=torch.float32 if out_f32 else torch.float16,
                            device=self._w.device)
        return y

    def run(self, x, y=None, out_f32: bool = False, stream=None):
        N = x.shape[0]
        y = self._y(N, out_f32, y)
        qgemv_run(self.h, x.data_ptr(), N, y.data_ptr(), OUT_F32 if out_f32 else OUT_F16,
                  _stream_ptr(stream))
        return y

    def run_add(self, x, residual, y=None, stream=None):
        N = x.shape[0]
        y = self._y(N, False, y)
        qgemv_run_add(self.h, x.data_ptr(), N, residual.data_ptr(), y.data_ptr(),
                      _stream_ptr(stream))
        return y

    def dequantize(self, stream=None):
        import torch
        w = torch.empty((self.M, self.K), dtype=torch.float32, device=self._w.device)
        qgemv_dequantize(self.h, w.data_ptr(), _stream_ptr(stream))
        return w

    def run_host(self, x_host, y_host, out_f32: bool = False, stream=None):
        qgemv_run_host(self.h, x_host.data_ptr(), x_host.shape[0], y_host.data_ptr(),
                       OUT_F32 if out_f32 else OUT_F16, _stream_ptr(stream))
        return y_host

    def plan_info(self, N: int):
        return qgemv_plan_info(self.h, N)

    def device_status(self, clear: bool = False) -> int:
        return qgemv_device_status(self.h, clear)


def pair_run(a: QGemv, b: QGemv, x, out_f32: bool = False, stream=None):
    N = x.shape[0]
    ya, yb = a._y(N, out_f32, None), b._y(N, out_f32, None)
    qgemv_pair_run(a.h, b.h, x.data_ptr(), N, ya.data_ptr(), yb.data_ptr(),
                   OUT_F32 if out_f32 else OUT_F16, _stream_ptr(stream))
    return ya, yb


def triple_run(a: QGemv, b: QGemv, c: QGemv, x, out_f32: bool = False, stream=None):
    N = x.shape[0]
    ya, yb, yc = a._y(N, out_f32, None), b._y(N, out_f32, None), c._y(N, out_f32, None)
    qgemv_triple_run(a.h, b.h, c.h, x.data_ptr(), N, ya.data_ptr(), yb.data_ptr(),
                     yc.data_ptr(), OUT_F32 if out_f32 else OUT_F16, _stream_ptr(stream))
    return ya, yb, yc


def pair_swiglu_run(gate: QGemv, up: QGemv, x, out_f32: bool = False, stream=None):
    """h = silu(x . gate^T) * (x . up^T), one launch."""
    N = x.shape[0]
    h = gate._y(N, out_f32, None)
    qgemv_pair_swiglu_run(gate.h, up.h, x.data_ptr(), N, h.data_ptr(),
                          OUT_F32 if out_f32 else OUT_F16, _stream_ptr(stream))
    return h


class Chain:
    """A decode chain: consecutive calls in one persistent launch where the
    library can, with the results of issuing them one by one."""

    def __init__(self, flags: int = 0):
        self.c = qgemv_chain_create(flags)

    def run(self, calls, stream=None):
        """calls: QgCall array from make_calls (reusable across runs)."""
        qgemv_chain_run(self.c, calls, _stream_ptr(stream))

    def status(self, clear: bool = False) -> int:
        return qgemv_chain_status(self.c, clear)

    def close(self):
        if getattr(self, "c", None):
            qgemv_chain_destroy(self.c)
            self.c = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
