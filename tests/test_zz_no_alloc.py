"""The allocation-free entry point (qgemv_run_noalloc) against the oracle and
against qgemv_run.

Some callers cannot allocate device memory while they run (a serving runtime
that owns all device memory in its own pool, a library that must keep its
footprint fixed), so the library offers a handle-free product whose scratch
is a fixed array inside the library.  This file is collected last so that a
run stopping at the first failure has run every other test before it.  Two
calls in a row share the array; each must match the CPU oracle within the
parity tolerance and qgemv_run bit for bit (same plan and kernels), and its
error word must stay clear.  (The argument checks, which run before the
device is touched, are tested on the host in test_abi_host.py.)"""
import numpy as np
import pytest

import oracle
from gpu_util import check_close, make_matrix, to_dev, torch
from skinny_gemm_q4_gb300 import qgemv as qg
from skinny_gemm_q4_gb300 import synth

pytestmark = pytest.mark.gpu

ORTYPE = {qg.Q4_K: oracle.Q4_K, qg.Q5_K: oracle.Q5_K, qg.Q6_K: oracle.Q6_K,
          qg.NVFP4_W4A16: oracle.NVFP4, qg.FP8_E4M3: oracle.FP8}


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
                                         (qg.FP8_E4M3, 1000, 5120, 12),
                                         (qg.Q5_K, 640, 2560, 3), (qg.Q4_K, 9728, 2560, 1),
                                         (qg.Q6_K, 2560, 9728, 1)])
def test_noalloc_matches_oracle_and_run_on_two_calls_in_a_row(qtype, M, K, N):
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
    assert qg.qgemv_device_status(None) == 0
    for x, y in zip(xs, outs):
        yref, mag = oracle.qgemv(ORTYPE[qtype], w, M, K, x, scales=sc, global_scale=g, rows=rows)
        check_close(y.cpu().numpy()[:, rows], yref, mag, what="noalloc vs oracle")
        # N >= 33 K-quant calls of a default handle run on the tcgen05 engine;
        # the allocation-free entry stays on the mma.sync kernels
        hr = h
        if N >= 33 and qtype in (qg.Q4_K, qg.Q5_K, qg.Q6_K):
            hr = qg.QGemv(qtype, M, K, h._w, h._scales, g, flags=qg.FLAG_MMA_SYNC_PREFILL)
        ref = hr.run(to_dev(x), out_f32=True)
        t.cuda.synchronize()
        check_close(y.cpu().numpy()[:, rows], ref.cpu().numpy()[:, rows].astype(np.float64), mag,
                    what="noalloc vs qgemv_run")
        assert t.equal(y, ref)


def test_noalloc_q4k_prefill_chunk_keeps_the_mma_sync_bits():
    """Q4_K at N = 40: qgemv_run_noalloc stays on the mma.sync kernels, so it
    equals a handle created with QG_FLAG_MMA_SYNC_PREFILL bit for bit and the
    default handle (tcgen05 engine) within the tolerance."""
    t = torch()
    M, K, N = 3000, 2560, 40
    h, w, sc, g = make_matrix(qg.Q4_K, M, K, seed=23)
    h._gscale = g
    hm = qg.QGemv(qg.Q4_K, M, K, h._w, flags=qg.FLAG_MMA_SYNC_PREFILL)
    x = synth.activations(N, K, seed=24, duplicate_rows=True)
    xd = to_dev(x)
    y = t.empty((N, M), dtype=t.float32, device="cuda")
    _noalloc(h, xd, N, y, True)
    ym = hm.run(xd, out_f32=True)
    yd = h.run(xd, out_f32=True)
    t.cuda.synchronize()
    assert t.equal(y, ym)
    rows = np.arange(0, M, 7)
    yref, mag = oracle.qgemv(oracle.Q4_K, w, M, K, x, rows=rows)
    check_close(y.cpu().numpy()[:, rows], yref, mag, what="noalloc N=40 vs oracle")
    check_close(yd.cpu().numpy()[:, rows], yref, mag, what="default handle N=40 vs oracle")
    assert qg.qgemv_device_status(None) == 0
