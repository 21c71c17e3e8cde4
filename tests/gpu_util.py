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
    sd = None if sc is None else t.from_numpy(np.ascontiguousarray(sc)).to(device)
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
