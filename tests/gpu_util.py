"""Helpers shared by the GPU tests: upload seeded inputs, run through the
C ABI, compare with the CPU oracle under the stated tolerance."""
from __future__ import annotations

import numpy as np

import oracle
from skinny_gemm_q4_gb300 import qgemv as qg
from skinny_gemm_q4_gb300 import synth

#: |y - y_ref| <= REL * sum_k |w x| (+ |residual|) + ABS   (fp32 output)
REL = 1e-3
ABS = 1e-5


def torch():
    import torch as t
    return t


def make_matrix(qtype, M, K, seed=0, stream=None, device="cuda", flags=0):
    """(QGemv handle, host bytes, host scales, global scale)."""
    t = torch()
    w, sc, g = synth.weights(qtype, M, K, seed=seed, stream=qtype if stream is None else stream)
    wd = t.from_numpy(np.ascontiguousarray(w)).to(device)
    sd = None if sc is None else t.from_numpy(np.ascontiguousarray(sc).view(np.uint8)).to(device)
    h = qg.QGemv(qtype, M, K, wd, sd, g, flags=flags)
    return h, w, sc, g


def to_dev(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a)).cuda()


def check_close(y_gpu, y_ref, mag, fp16_out=False, what=""):
    """Element-wise acceptance test; returns the worst ratio err / bound."""
    y = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = REL * mag + ABS
    if fp16_out:
        # plus the final rounding of the result to fp16 (half an ulp)
        bound = bound + np.maximum(np.abs(y_ref) * 2.0 ** -11, 2.0 ** -25)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
            f"gpu={y[tuple(i)]!r} ref={y_ref[tuple(i)]!r} mag={mag[tuple(i)]!r}")
    return float(np.max(err / bound))


def canon(a):
    a = np.array(a, dtype=np.float32, copy=True)
    a[a == 0] = 0.0
    return a


def swiglu_bound(g_ref, mag_g, u_ref, mag_u, fp16_out=False):
    """Bound on |h_gpu - h_ref| for h = silu(g) * u, derived from the product
    tolerance: |g_gpu - g_ref| <= e_g = REL mag_g + ABS (likewise u), silu is
    1.1-Lipschitz (max |silu'| = 1.0998), so
      |h_gpu - h_ref| <= (|silu(g_ref)| + 1.1 e_g) e_u + 1.1 |u_ref| e_g
                         + 2^-20 (|silu(g_ref)| + 1.1 e_g)(|u_ref| + e_u)
    (the last term: fp32 expf, add, divide and multiply, a few ulps), plus half
    an fp16 ulp of the result for fp16 output."""
    g_ref = np.asarray(g_ref, dtype=np.float64)
    u_ref = np.asarray(u_ref, dtype=np.float64)
    e_g = REL * mag_g + ABS
    e_u = REL * mag_u + ABS
    with np.errstate(over="ignore"):
        sg = np.abs(g_ref / (1.0 + np.exp(-g_ref)))
    b = (sg + 1.1 * e_g) * e_u + 1.1 * np.abs(u_ref) * e_g
    b = b + 2.0 ** -20 * (sg + 1.1 * e_g) * (np.abs(u_ref) + e_u)
    if fp16_out:
        h = sg * np.abs(u_ref)
        b = b + np.maximum(h * 2.0 ** -11, 2.0 ** -25)
    return b


def check_swiglu(h_gpu, h_ref, bound, what="", fp16_out=False):
    h = np.asarray(h_gpu, dtype=np.float64)
    h_ref = np.asarray(h_ref, dtype=np.float64)
    if fp16_out:
        # fp16 round-to-nearest overflows to +-inf from |v| >= 65520: compare
        # both sides saturated at that threshold
        top = 65520.0
        h = np.where(np.isinf(h), np.sign(h) * top, h)
        h_ref = np.clip(h_ref, -top, top)
    err = np.abs(h - h_ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside the SwiGLU bound; first "
                             f"at {tuple(i)}: gpu={h[tuple(i)]!r} ref={h_ref[tuple(i)]!r} "
                             f"bound={bound[tuple(i)]!r}")
    return float(np.max(err / bound))
