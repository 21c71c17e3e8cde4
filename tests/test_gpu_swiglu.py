"""Fused gate/up pair with the SwiGLU epilogue (reflex-llm "docs/kernels.md",
SwiGLU section: output = silu(gate) x up) through the C ABI, against the CPU
oracle (silu in float64 of the float64 products) under a tolerance derived
from the product tolerance, and bit-exact properties: the rows of an N-row
call equal one-row calls (N = 1..32), and h is silu(g) * u of exactly the
values a plain pair call returns."""
import numpy as np
import pytest

import oracle
from gpu_util import check_swiglu, make_matrix, swiglu_bound, to_dev, torch
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


def _pair(qtype, M, K, seed, flags=0):
    hg, wg, sg, gg = make_matrix(qtype, M, K, seed=seed, stream=qtype, flags=flags)
    hu, wu, su, gu = make_matrix(qtype, M, K, seed=seed, stream=qtype + 1000, flags=flags)
    return (hg, wg, sg, gg), (hu, wu, su, gu)


def _ref(qtype, gate, up, M, K, x, rows):
    (_, wg, sg, gg), (_, wu, su, gu) = gate, up
    return oracle.qgemv_swiglu(ORTYPE[qtype], wg, ORTYPE[qtype], wu, M, K, x, rows=rows,
                               scales_g=sg, gscale_g=gg, scales_u=su, gscale_u=gu)


# (9728, 2560): the decode layer's gate/up shape (K split 2); the others hit
# K splits of 1, 2 and 8 (the SwiGLU exchange with and without cluster
# ranks) and every format.
SHAPES = [(qg.Q4_K, 9728, 2560), (qg.Q4_K, 300, 2560), (qg.Q5_K, 130, 4096),
          (qg.Q6_K, 200, 2560), (qg.NVFP4_W4A16, 150, 5120), (qg.Q4_K, 2000, 256),
          (qg.Q5_K, 700, 512), (qg.FP8_E4M3, 260, 2560)]


@pytest.mark.parametrize("qtype,M,K", SHAPES)
@pytest.mark.parametrize("N", [1, 3, 8, 13, 32, 40])
def test_swiglu_pair_matches_oracle(qtype, M, K, N):
    t = torch()
    gate, up = _pair(qtype, M, K, seed=31)
    x = synth.activations(N, K, seed=31, duplicate_rows=True)
    rows = np.arange(M) if M <= 2000 else np.unique(
        np.concatenate([[0, M - 1], np.random.default_rng(2).integers(0, M, 300)]))
    href, g, mg, u, mu = _ref(qtype, gate, up, M, K, x, rows)
    xd = to_dev(x)
    h32 = qg.pair_swiglu_run(gate[0], up[0], xd, out_f32=True)
    h16 = qg.pair_swiglu_run(gate[0], up[0], xd, out_f32=False)
    t.cuda.synchronize()
    check_swiglu(h32.cpu().numpy()[:, rows], href, swiglu_bound(g, mg, u, mu),
                 what=f"swiglu fp32 {qtype} {M}x{K} N={N}")
    check_swiglu(h16.float().cpu().numpy()[:, rows], href,
                 swiglu_bound(g, mg, u, mu, fp16_out=True), what=f"swiglu fp16 {qtype} N={N}",
                 fp16_out=True)
    # fp16 output is the fp32 result rounded once
    assert np.array_equal(h16.cpu().numpy(), h32.half().cpu().numpy())
    # h is silu(g) * u of the pair call's own fp32 values (same products, fp32
    # epilogue); the SwiGLU pair keeps Q4_K prefill chunks on the mma.sync
    # kernels, so compare with a pair that does too
    pg = qg.QGemv(qtype, M, K, gate[0]._w, gate[0]._scales, gate[3],
                  flags=qg.FLAG_MMA_SYNC_PREFILL)
    pu = qg.QGemv(qtype, M, K, up[0]._w, up[0]._scales, up[3], flags=qg.FLAG_MMA_SYNC_PREFILL)
    ga, ua = qg.pair_run(pg, pu, xd, out_f32=True)
    hh = (ga / (1.0 + t.exp(-ga))) * ua
    assert t.allclose(h32, hh, rtol=2.0 ** -19, atol=1e-30)
    assert gate[0].device_status() == 0 and up[0].device_status() == 0


@pytest.mark.parametrize("qtype,M,K", [(qg.Q4_K, 9728, 2560), (qg.Q6_K, 200, 2560),
                                       (qg.NVFP4_W4A16, 150, 5120)])
def test_swiglu_pair_row_invariance_twins(qtype, M, K):
    """An N-row SwiGLU call equals N one-row calls bit for bit, N = 2..32."""
    t = torch()
    gate, up = _pair(qtype, M, K, seed=32)
    x = to_dev(synth.activations(32, K, seed=32, duplicate_rows=True))
    one = t.cat([qg.pair_swiglu_run(gate[0], up[0], x[n:n + 1], out_f32=True)
                 for n in range(32)]).cpu().numpy()
    for N in range(2, 33):
        hN = qg.pair_swiglu_run(gate[0], up[0], x[:N], out_f32=True).cpu().numpy()
        assert np.array_equal(hN.view(np.uint32), one[:N].view(np.uint32)), f"N={N}"
    assert np.array_equal(one[2], one[0])


def test_swiglu_reference_path_and_errors():
    """QG_FLAG_FORCE_REFERENCE runs the reference SwiGLU kernel (within the
    same bound); mismatched handles are rejected before any launch."""
    t = torch()
    M, K, N = 130, 2560, 5
    gate, up = _pair(qg.Q4_K, M, K, seed=33, flags=qg.FLAG_FORCE_REFERENCE)
    x = synth.activations(N, K, seed=33)
    href, g, mg, u, mu = _ref(qg.Q4_K, gate, up, M, K, x, np.arange(M))
    h = qg.pair_swiglu_run(gate[0], up[0], to_dev(x), out_f32=True)
    t.cuda.synchronize()
    check_swiglu(h.cpu().numpy(), href, swiglu_bound(g, mg, u, mu), what="reference swiglu")
    other, _, _, _ = make_matrix(qg.Q4_K, M + 1, K, seed=34)
    with pytest.raises(qg.QgemvError) as e:
        qg.pair_swiglu_run(gate[0], other, to_dev(x))
    assert e.value.status == -1
    q6, _, _, _ = make_matrix(qg.Q6_K, M, K, seed=35)
    with pytest.raises(qg.QgemvError) as e:
        qg.pair_swiglu_run(gate[0], q6, to_dev(x))
    assert e.value.status == -2
