"""The allocation-free entry point (qgemv_run_noalloc) against qgemv_run.

For callers that cannot allocate device memory while they run, the library
offers a handle-free product whose scratch is a fixed array inside the
library.  This file is collected last so that a run stopping at the first
failure has run every other test before it.  Two calls in a row share the
array; each must still match the handle-based qgemv_run within the parity
tolerance (and in fact bit for bit: same arithmetic and plan)."""
import ctypes

import numpy as np
import pytest

import oracle
from gpu_util import check_close, make_matrix, to_dev, torch
from skinny_gemm_q4_gb300 import qgemv as qg
from skinny_gemm_q4_gb300 import synth

pytestmark = pytest.mark.gpu

ORTYPE = {qg.Q4_K: oracle.Q4_K, qg.Q5_K: oracle.Q5_K, qg.Q6_K: oracle.Q6_K,
          qg.NVFP4_W4A16: oracle.NVFP4}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from skinny_gemm_q4_gb300 import build
    build.build()
    assert torch().cuda.is_available()


def _noalloc(h, x, N, y, out_f32):
    t = torch()
    qg.qgemv_run_noalloc(h.qtype, h.M, h.K, h._w.data_ptr(),
                         h._scales.data_ptr() if h._scales is not None else 0, h._gscale,
                         x.data_ptr(), N, y.data_ptr(), qg.OUT_F32 if out_f32 else qg.OUT_F16,
                         t.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("qtype,M,K,N", [(qg.Q4_K, 4096, 2560, 20), (qg.Q6_K, 1024, 9728, 40),
                                         (qg.NVFP4_W4A16, 2048, 5120, 9),
                                         (qg.Q5_K, 640, 2560, 3)])
def test_noalloc_matches_run_on_two_calls_in_a_row(qtype, M, K, N):
    t = torch()
    h, w, sc, g = make_matrix(qtype, M, K, seed=21)
    h._gscale = g
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(1).integers(0, M, 48)]))
    xs = [synth.activations(N, K, seed=22 + i) for i in range(2)]
    outs = []
    for x in xs:                                   # two calls back to back, shared scratch
        y = t.empty((N, M), dtype=t.float32, device="cuda")
        _noalloc(h, to_dev(x), N, y, True)
        outs.append(y)
    t.cuda.synchronize()
    for x, y in zip(xs, outs):
        ref = h.run(to_dev(x), out_f32=True)
        t.cuda.synchronize()
        _, mag = oracle.qgemv(ORTYPE[qtype], w, M, K, x, scales=sc, global_scale=g, rows=rows)
        check_close(y.cpu().numpy()[:, rows], ref.cpu().numpy()[:, rows].astype(np.float64), mag,
                    what="noalloc vs qgemv_run")
        assert t.equal(y, ref)


def test_noalloc_rejects_oversized_k_without_touching_the_gpu():
    lib = qg.load()
    f = lib.qgemv_run_noalloc
    f.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_float, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_void_p]
    f.restype = ctypes.c_int
    st = f(qg.Q4_K, 16, 1 << 20, 4096, None, 1.0, 4096, 1, 4096, qg.OUT_F16, None)
    assert st == -2 and "2 MiB" in qg.qgemv_last_error()
