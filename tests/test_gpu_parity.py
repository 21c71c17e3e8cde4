"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element
by element, on seeded inputs that span several tiles, K-split ranks and ragged
row tails; bit-exact checks where the arithmetic is exact."""
import numpy as np
import pytest

import oracle
from gpu_util import canon, check_close, make_matrix, to_dev, torch
from skinny_gemm_q4_gb300 import qgemv as qg
from skinny_gemm_q4_gb300 import synth

pytestmark = pytest.mark.gpu

TYPES = [qg.Q4_K, qg.Q5_K, qg.Q6_K, qg.NVFP4_W4A16, qg.FP8_E4M3]
ORTYPE = {qg.Q4_K: oracle.Q4_K, qg.Q5_K: oracle.Q5_K, qg.Q6_K: oracle.Q6_K,
          qg.NVFP4_W4A16: oracle.NVFP4, qg.FP8_E4M3: oracle.FP8}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from skinny_gemm_q4_gb300 import build
    build.build()
    t = torch()
    assert t.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("M,K", [(37, 768), (130, 2560), (1030, 9728)])
@pytest.mark.parametrize("flags", [0, qg.FLAG_FORCE_REFERENCE], ids=["product_decoders", "reference"])
def test_dequantize_bit_exact(qtype, M, K, flags):
    """qgemv_dequantize runs the product kernels' own decoders (and, with
    FORCE_REFERENCE, the simple per-element reference decoder): every weight
    equals the oracle's bit for bit (after -0 -> +0)."""
    h, w, sc, g = make_matrix(qtype, M, K, seed=3, flags=flags)
    wd = h.dequantize()
    torch().cuda.synchronize()
    ref = oracle.dequantize(ORTYPE[qtype], w, M, K, scales=sc, global_scale=g)
    got = canon(wd.cpu().numpy())
    assert np.array_equal(got.view(np.uint32), canon(ref).view(np.uint32))


# Shapes and one-hot chunk sizes that reach every mma.sync product kernel:
# chunk 1 -> the N = 1 variant of the N <= 8 kernel; chunk 8 -> the N <= 8
# kernel (Q6_K, NVFP4, and Q4_K/Q5_K above 4096 rows) or qg_sk_kernel with x
# staged inside (Q4_K/Q5_K up to 4096 rows); chunks 16 and 32 -> qg_sk_kernel
# after the staging launch (2 and 4 column groups).
ONE_HOT = [(qg.Q4_K, 150, 1024), (qg.Q4_K, 4100, 512), (qg.Q5_K, 96, 768),
           (qg.Q5_K, 4100, 512), (qg.Q6_K, 150, 1024), (qg.NVFP4_W4A16, 150, 1024),
           (qg.FP8_E4M3, 150, 1024), (qg.FP8_E4M3, 4100, 512)]


@pytest.mark.parametrize("qtype,M,K", ONE_HOT)
@pytest.mark.parametrize("chunk", [1, 8, 16, 32])
def test_mma_sync_one_hot_is_the_exact_weight(qtype, M, K, chunk):
    """x = e_k for every k, in calls of `chunk` rows: each mma.sync kernel
    returns w[m][k] bit for bit (one exact product, the fold's single
    rounding), so its decoders equal the oracle's dequantization."""
    t = torch()
    h, w, sc, g = make_matrix(qtype, M, K, seed=4, flags=qg.FLAG_MMA_SYNC_PREFILL)
    x = to_dev(np.eye(K, dtype=np.float16))
    y = t.cat([h.run(x[i:i + chunk], out_f32=True) for i in range(0, K, chunk)])
    t.cuda.synchronize()
    ref = oracle.dequantize(ORTYPE[qtype], w, M, K, scales=sc, global_scale=g)
    assert np.array_equal(canon(y.cpu().numpy()).view(np.uint32), canon(ref.T).view(np.uint32))
    assert h.device_status() == 0


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("N", [1, 5, 16, 40])
def test_large_magnitude_x(qtype, N):
    """x far outside N(0, 1): rows scaled by 2^8, 2^10, 2^12 and sub-blocks of
    32 equal values near the fp16 limit (|sum| up to 32 * 65504, past the fp16
    range, which the Q4_K/Q5_K min term's sub-block sums must still carry).
    fp32 output within the tolerance; power-of-two scaling stays exact."""
    M = 300
    K = 5120 if qtype in (qg.NVFP4_W4A16, qg.FP8_E4M3) else 2560
    h, w, sc, g = make_matrix(qtype, M, K, seed=11)
    base = synth.activations(N, K, seed=11).astype(np.float32)
    x = base * (2.0 ** (8 + 2 * (np.arange(N) % 3)))[:, None]
    x[0, 96:128] = 60000.0
    x[-1, 0:32] = -65504.0
    x[-1, 2048:2080] = 65504.0
    x = x.astype(np.float16)
    assert np.isfinite(x).all()
    yref, mag = oracle.qgemv(ORTYPE[qtype], w, M, K, x, scales=sc, global_scale=g)
    y = h.run(to_dev(x), out_f32=True).cpu().numpy()
    check_close(y, yref, mag, what=f"large x {qtype} N={N}")
    xs = base.astype(np.float16)
    y1 = h.run(to_dev(xs), out_f32=True).cpu().numpy()
    y256 = h.run(to_dev((xs.astype(np.float32) * 256).astype(np.float16)), out_f32=True).cpu().numpy()
    # Exact scaling needs every nonzero sub-block sum of x at |S| >= 2^-9 (the
    # Q4_K/Q5_K min term splits S = 32 hi + lo with hi an fp16 normal there).
    S = np.abs(xs.astype(np.float64).reshape(N, K // 32, 32).sum(-1))
    ok = ((S == 0) | (S >= 2.0 ** -9)).all(axis=1)
    if qtype in (qg.Q6_K, qg.NVFP4_W4A16, qg.FP8_E4M3):
        ok[:] = True
    assert ok.any()
    assert np.array_equal(y256[ok], 256 * y1[ok])
    assert h.device_status() == 0


@pytest.mark.parametrize("qtype", TYPES)
def test_fast_path_one_hot_is_the_exact_weight(qtype):
    """K = 256, x = e_k for all 256 k (two token chunks of 128; the tcgen05
    engine for the K-quants): the fast product returns w[m][k] bit for bit (a
    single exact product, one final rounding), so the fast decoders equal the
    oracle's dequantization.  Q6_K on the tcgen05 engine rounds s * (q - 32)
    once to fp16 where it needs 12 significant bits (|s (q - 32)| > 2048):
    there the weight is within 2^-11 of the oracle's, everywhere else exact;
    its mma.sync kernels stay exact."""
    M, K = 21, 256
    h, w, sc, g = make_matrix(qtype, M, K, seed=4)
    x = np.eye(K, dtype=np.float16)
    y = h.run(to_dev(x), out_f32=True)
    torch().cuda.synchronize()
    ref = oracle.dequantize(ORTYPE[qtype], w, M, K, scales=sc, global_scale=g)
    yc = canon(y.cpu().numpy())
    if qtype != qg.Q6_K:
        assert np.array_equal(yc.view(np.uint32), canon(ref.T).view(np.uint32))
        return
    rt = ref.T.astype(np.float64)
    err = np.abs(yc.astype(np.float64) - rt)
    assert (err <= np.abs(rt) * 2.0 ** -11).all()
    assert (err == 0).mean() > 0.9
    hm, _, _, _ = make_matrix(qtype, M, K, seed=4, flags=qg.FLAG_MMA_SYNC_PREFILL)
    ym = canon(hm.run(to_dev(x), out_f32=True).cpu().numpy())
    assert np.array_equal(ym.view(np.uint32), canon(ref.T).view(np.uint32))


CASES = [
    (qg.Q4_K, 300, 2560), (qg.Q4_K, 77, 4096),
    (qg.Q5_K, 130, 4096), (qg.Q5_K, 64, 1536),
    (qg.Q6_K, 200, 2560), (qg.Q6_K, 45, 9728),
    (qg.NVFP4_W4A16, 150, 5120), (qg.NVFP4_W4A16, 33, 768),
    (qg.FP8_E4M3, 150, 5120), (qg.FP8_E4M3, 300, 768), (qg.FP8_E4M3, 33, 2560),
]


@pytest.mark.parametrize("qtype,M,K", CASES)
@pytest.mark.parametrize("N", [1, 3, 8, 13, 32, 40])
def test_product_matches_oracle(qtype, M, K, N):
    h, w, sc, g = make_matrix(qtype, M, K, seed=5)
    x = synth.activations(N, K, seed=5, duplicate_rows=True)
    yref, mag = oracle.qgemv(ORTYPE[qtype], w, M, K, x, scales=sc, global_scale=g)
    xd = to_dev(x)
    y32 = h.run(xd, out_f32=True)
    y16 = h.run(xd, out_f32=False)
    torch().cuda.synchronize()
    check_close(y32.cpu().numpy(), yref, mag, what=f"fp32 {qtype} {M}x{K} N={N}")
    check_close(y16.float().cpu().numpy(), yref, mag, fp16_out=True,
                what=f"fp16 {qtype} {M}x{K} N={N}")
    # fp16 output is the fp32 result rounded once
    assert np.array_equal(y16.cpu().numpy(), y32.half().cpu().numpy())


@pytest.mark.parametrize("qtype,M,K", [(qg.Q4_K, 9728, 2560), (qg.Q4_K, 4096, 2560),
                                       (qg.Q4_K, 2560, 4096), (qg.Q4_K, 1024, 2560),
                                       (qg.Q5_K, 2560, 9728),
                                       (qg.Q6_K, 1024, 2560), (qg.Q6_K, 2560, 9728),
                                       (qg.NVFP4_W4A16, 7168, 5120),
                                       (qg.NVFP4_W4A16, 27648, 5120),
                                       (qg.NVFP4_W4A16, 5120, 27648),
                                       (qg.FP8_E4M3, 7168, 5120), (qg.FP8_E4M3, 2560, 9728)])
def test_row_invariance_twins(qtype, M, K):
    """TandemLLM verify-twin rule: an N-row call equals N one-row calls bit
    for bit, N = 2..32, with rows that share inputs."""
    # N >= 33 Q4_K calls default to the tcgen05 engine (tolerance only); the
    # mma.sync prefill path is the one that keeps the N <= 32 bits
    h, w, sc, g = make_matrix(qtype, M, K, seed=6, flags=qg.FLAG_MMA_SYNC_PREFILL)
    x = synth.activations(32, K, seed=6, duplicate_rows=True)
    xd = to_dev(x)
    singles = [h.run(xd[n:n + 1], out_f32=True) for n in range(32)]
    one = torch().cat(singles).cpu().numpy()
    for N in range(2, 33):
        yN = h.run(xd[:N], out_f32=True).cpu().numpy()
        assert np.array_equal(yN.view(np.uint32), one[:N].view(np.uint32)), f"N={N}"
    # duplicated inputs give duplicated outputs
    assert np.array_equal(one[2], one[0])
    # N >= 33 (next chunking regime) keeps the same bits too on the mma.sync path
    y40 = h.run(to_dev(np.concatenate([x, x[:8]])), out_f32=True).cpu().numpy()
    assert np.array_equal(y40[:32].view(np.uint32), one.view(np.uint32))
    assert h.device_status() == 0


TC_SHAPES = [(qg.Q4_K, 9728, 2560), (qg.Q4_K, 300, 2560), (qg.Q4_K, 77, 4096),
             (qg.Q5_K, 130, 4096), (qg.Q6_K, 2560, 9728), (qg.Q6_K, 200, 2560),
             (qg.Q6_K, 45, 9728)]


@pytest.mark.parametrize("qtype,M,K", TC_SHAPES)
@pytest.mark.parametrize("N", [33, 40, 64, 100, 128, 200])
def test_tcgen05_prefill_engine(qtype, M, K, N):
    """tcgen05 / tensor-memory engine, the default for K-quant prefill chunks
    (N >= 33): within the tolerance of the oracle, duplicated rows
    bit-identical, fp16 output the fp32 result rounded once, residual variant
    and fused pair; QG_FLAG_MMA_SYNC_PREFILL selects the mma.sync kernels."""
    t = torch()
    w, sc, g = synth.weights(qtype, M, K, seed=21, stream=qtype)
    wd = t.from_numpy(np.ascontiguousarray(w)).cuda()
    h = qg.QGemv(qtype, M, K, wd)
    ks, rows, launches = h.plan_info(N)
    assert rows == 128 and launches == 2 * ((N + 127) // 128)
    assert 1 <= ks <= 8 and ks <= K // 256
    hm = qg.QGemv(qtype, M, K, wd, flags=qg.FLAG_MMA_SYNC_PREFILL)
    ym = hm.run(to_dev(synth.activations(N, K, seed=21, duplicate_rows=True)), out_f32=True)
    x = synth.activations(N, K, seed=21, duplicate_rows=True)
    rows_chk = np.unique(np.concatenate([np.arange(min(M, 64)), np.arange(M - min(M, 64), M),
                                         np.random.default_rng(N).integers(0, M, 200)]))
    yref, mag = oracle.qgemv(ORTYPE[qtype], w, M, K, x, rows=rows_chk)
    xd = to_dev(x)
    y32 = h.run(xd, out_f32=True)
    y16 = h.run(xd, out_f32=False)
    check_close(y32.cpu().numpy()[:, rows_chk], yref, mag, what=f"tcgen05 {qtype} {M}x{K} N={N}")
    check_close(ym.cpu().numpy()[:, rows_chk], yref, mag,
                what=f"mma.sync prefill {qtype} {M}x{K} N={N}")
    assert np.array_equal(y16.cpu().numpy(), y32.half().cpu().numpy())
    yc = y32.cpu().numpy()
    assert np.array_equal(yc[2].view(np.uint32), yc[0].view(np.uint32))  # row 2 repeats row 0
    r = synth.residual(N, M, seed=21)
    ya = h.run_add(xd, to_dev(r)).float().cpu().numpy()
    yref_a, mag_a = oracle.qgemv(ORTYPE[qtype], w, M, K, x, residual=r, rows=rows_chk)
    check_close(ya[:, rows_chk], yref_a, mag_a, fp16_out=True, what="tcgen05 run_add")
    # the pair call: one launch over both matrices (its K split follows the
    # launch's row tiles, so the bits may differ from a single call's; prefill
    # chunks have no twin contract), each within the tolerance
    h2 = qg.QGemv(qtype, M, K, wd)
    pa, pb = qg.pair_run(h, h2, xd, out_f32=True)
    check_close(pa.cpu().numpy()[:, rows_chk], yref, mag, what="tcgen05 pair a")
    check_close(pb.cpu().numpy()[:, rows_chk], yref, mag, what="tcgen05 pair b")
    assert np.array_equal(pa.cpu().numpy().view(np.uint32), pb.cpu().numpy().view(np.uint32))
    assert h.device_status() == 0 and h2.device_status() == 0


TC_EDGE = [  # (M, K, N, max_tokens): one row, one super-block, token chunks, ragged tails
    (1, 256, 40, 0), (1, 2560, 33, 0), (17, 256, 129, 0), (130, 1024, 70, 32),
    (129, 768, 47, 0), (255, 512, 200, 64),
]


@pytest.mark.parametrize("qtype", [qg.Q4_K, qg.Q5_K, qg.Q6_K])
@pytest.mark.parametrize("M,K,N,mt", TC_EDGE)
def test_tcgen05_edge_shapes(qtype, M, K, N, mt):
    """The tcgen05 engine on degenerate and ragged shapes: a single row, a
    single super-block (one K slice), 129 rows (a one-row second tile),
    token chunks of max_tokens and a ragged last chunk; within the tolerance
    of the oracle, duplicated rows bit-identical."""
    t = torch()
    w, sc, g = synth.weights(qtype, M, K, seed=31, stream=qtype)
    wd = t.from_numpy(np.ascontiguousarray(w)).cuda()
    h = qg.QGemv(qtype, M, K, wd, max_tokens=mt)
    x = synth.activations(N, K, seed=31, duplicate_rows=True)
    y = h.run(to_dev(x), out_f32=True).cpu().numpy()
    yref, mag = oracle.qgemv(ORTYPE[qtype], w, M, K, x)
    check_close(y, yref, mag, what=f"tcgen05 edge {qtype} {M}x{K} N={N} max_tokens={mt}")
    assert np.array_equal(y[2].view(np.uint32), y[0].view(np.uint32))
    assert h.device_status() == 0


@pytest.mark.parametrize("qtype", [qg.Q4_K, qg.Q6_K, qg.NVFP4_W4A16, qg.FP8_E4M3])
def test_sign_and_power_of_two_scaling_exact(qtype):
    M, K = 96, 2560 if qtype not in (qg.NVFP4_W4A16, qg.FP8_E4M3) else 5120
    h, w, sc, g = make_matrix(qtype, M, K, seed=7)
    x = synth.activations(5, K, seed=7)
    y = h.run(to_dev(x), out_f32=True).cpu().numpy()
    yn = h.run(to_dev(-x), out_f32=True).cpu().numpy()
    y4 = h.run(to_dev((x.astype(np.float32) * 4).astype(np.float16)), out_f32=True).cpu().numpy()
    assert np.array_equal(yn, -y)
    assert np.array_equal(y4, 4 * y)


def test_q4k_all_q_zero_min_term():
    """All q = 0 with uniform mins: y = -dmin * m * sum(x) (within tolerance)."""
    from packers import pack_q4k_block
    M, K, N = 64, 2560, 4
    blk = pack_q4k_block(0.01171875, 0.0078125, [17] * 8, [37] * 8, np.zeros(256, dtype=np.int64))
    w = np.tile(blk, (M, K // 256))
    t = torch()
    h = qg.QGemv(qg.Q4_K, M, K, t.from_numpy(w).cuda())
    x = synth.activations(N, K, seed=8)
    y = h.run(to_dev(x), out_f32=True).cpu().numpy()
    expect = -0.0078125 * 37 * x.astype(np.float64).sum(axis=1)
    mag = 0.0078125 * 37 * np.abs(x.astype(np.float64)).sum(axis=1)
    check_close(y, np.repeat(expect[:, None], M, 1), np.repeat(mag[:, None], M, 1))


@pytest.mark.parametrize("inplace", [False, True])
@pytest.mark.parametrize("M,N", [(2560, 3), (77, 12), (2560, 40)])
def test_run_add_residual(inplace, M, N):
    """Residual added in fp32 before one rounding; M = 77 gives rows whose
    y addresses are not 8-byte aligned (scalar epilogue stores)."""
    K = 4096
    h, w, sc, g = make_matrix(qg.Q4_K, M, K, seed=9)
    x = synth.activations(N, K, seed=9)
    r = synth.residual(N, M, seed=9)
    yref, mag = oracle.qgemv(oracle.Q4_K, w, M, K, x, residual=r)
    rd = to_dev(r)
    y = rd if inplace else torch().empty_like(rd)
    h.run_add(to_dev(x), rd, y)
    check_close(y.float().cpu().numpy(), yref, mag, fp16_out=True, what="run_add")


@pytest.mark.parametrize("N", [5, 12, 40])
def test_pair_and_mixed_triple_equal_separate_calls(N):
    """The fused calls give each matrix the bits of its own call; the triple
    mixes formats and K-slice counts (Q 4096 rows: 4 slices, K/V: 8).  At
    N >= 33 (the tcgen05 engine) a launch's K split follows all its row
    tiles, so there the fused calls are checked against the oracle only
    (prefill chunks have no twin contract)."""
    K = 2560
    a, wa, _, _ = make_matrix(qg.Q4_K, 4096, K, seed=10, stream=1)
    b, wb, _, _ = make_matrix(qg.Q4_K, 1024, K, seed=10, stream=2)
    c, wc, _, _ = make_matrix(qg.Q6_K, 1024, K, seed=10, stream=3)
    x = synth.activations(N, K, seed=10)
    xd = to_dev(x)
    ya, yb, yc = qg.triple_run(a, b, c, xd, out_f32=True)
    for hnd, y, w, t in ((a, ya, wa, oracle.Q4_K), (b, yb, wb, oracle.Q4_K), (c, yc, wc, oracle.Q6_K)):
        sep = hnd.run(xd, out_f32=True)
        assert N >= 33 or torch().equal(y, sep)
        yref, mag = oracle.qgemv(t, w, hnd.M, K, x)
        check_close(y.cpu().numpy(), yref, mag, what="triple")
    p1, w1, _, _ = make_matrix(qg.Q4_K, 9728, K, seed=11, stream=4)
    p2, w2, _, _ = make_matrix(qg.Q4_K, 9728, K, seed=11, stream=5)
    y1, y2 = qg.pair_run(p1, p2, xd)
    assert N >= 33 or (torch().equal(y1, p1.run(xd)) and torch().equal(y2, p2.run(xd)))
    rows = np.arange(0, 9728, 97)
    yref, mag = oracle.qgemv(oracle.Q4_K, w2, 9728, K, x, rows=rows)
    check_close(y2.float().cpu().numpy()[:, rows], yref, mag, fp16_out=True, what="pair")


def test_reference_kernel_and_fallback(monkeypatch):
    M, K, N = 160, 2560, 6
    t = torch()
    w, _, _ = synth.weights(qg.Q4_K, M, K, seed=12, stream=1)
    wd = t.from_numpy(w).cuda()
    x = synth.activations(N, K, seed=12)
    yref, mag = oracle.qgemv(oracle.Q4_K, w, M, K, x)
    ref = qg.QGemv(qg.Q4_K, M, K, wd, flags=qg.FLAG_FORCE_REFERENCE)
    check_close(ref.run(to_dev(x), out_f32=True).cpu().numpy(), yref, mag, what="reference")
    monkeypatch.setenv("QGEMV_FAULT_INJECT", "launch")
    fb = qg.QGemv(qg.Q4_K, M, K, wd)
    y = fb.run(to_dev(x), out_f32=True)
    t.cuda.synchronize()
    assert "reference" in qg.qgemv_last_error()
    check_close(y.cpu().numpy(), yref, mag, what="fallback")
    strict = qg.QGemv(qg.Q4_K, M, K, wd, flags=qg.FLAG_NO_FALLBACK)
    with pytest.raises(qg.QgemvError) as ei:
        strict.run(to_dev(x))
    assert ei.value.status == -6
    monkeypatch.setenv("QGEMV_FAULT_INJECT", "create")
    with pytest.raises(qg.QgemvError) as ei:
        qg.QGemv(qg.Q4_K, M, K, wd)
    assert ei.value.status == -6


def test_run_host_matches_device_path():
    M, K, N = 512, 2560, 4
    h, w, sc, g = make_matrix(qg.Q4_K, M, K, seed=13)
    x = synth.activations(N, K, seed=13)
    t = torch()
    xh = t.from_numpy(x).pin_memory()
    yh = t.empty((N, M), dtype=t.float16).pin_memory()
    h.run_host(xh, yh)
    yd = h.run(to_dev(x))
    t.cuda.synchronize()
    assert t.equal(yh, yd.cpu())


def test_argument_errors_are_statuses():
    M, K = 64, 2560
    h, w, sc, g = make_matrix(qg.Q4_K, M, K, seed=14)
    t = torch()
    x = t.zeros((2, K), dtype=t.float16, device="cuda")
    y = t.zeros((2, M), dtype=t.float16, device="cuda")
    lib = qg.load()
    assert lib.qgemv_run(h.h, x.data_ptr(), 0, y.data_ptr(), 0, None) == -1
    assert lib.qgemv_run(h.h, x.data_ptr() + 2, 1, y.data_ptr(), 0, None) == -3
    assert lib.qgemv_run(h.h, None, 1, y.data_ptr(), 0, None) == -1
    other, _, _, _ = make_matrix(qg.Q4_K, 64, 4096, seed=14)
    assert lib.qgemv_pair_run(h.h, other.h, x.data_ptr(), 1, y.data_ptr(), x.data_ptr(), 0,
                              None) == -1
    kw, rows, launches = h.plan_info(1)
    assert kw == 8 and rows == 16 and launches == 1      # N <= 8: one kernel
    kw, rows, launches = h.plan_info(40)
    assert rows == 128 and launches == 2                 # staging + tcgen05 product
    kw, rows, launches = h.plan_info(16)
    assert kw == 8 and rows == 128 and launches == 2     # staging + product
    kw, rows, launches = h.plan_info(4)
    assert kw == 8 and rows == 128 and launches == 1     # qg_sk_kernel stages x itself
    assert h.device_status() == 0


EDGE = [  # (M, K, N, max_tokens): one row, one super-block, chunked N, ragged tails
    (1, 256, 1, 0), (1, 256, 40, 0), (17, 256, 9, 0), (1, 2560, 33, 0),
    (33, 512, 20, 8), (130, 1024, 70, 32), (5, 768, 3, 1),
]


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("M,K,N,mt", EDGE)
def test_edge_shapes(qtype, M, K, N, mt):
    """Degenerate and ragged shapes: a single row, a single super-block
    (K = 256), N processed in max_tokens chunks, ragged row and token tails.
    Within the tolerance of the oracle, and rows computed in chunks of at
    most 32 equal one-row calls bit for bit."""
    t = torch()
    w, sc, g = synth.weights(qtype, M, K, seed=30, stream=qtype)
    wd = t.from_numpy(np.ascontiguousarray(w)).cuda()
    sd = None if sc is None else t.from_numpy(np.ascontiguousarray(sc)).cuda()
    h = qg.QGemv(qtype, M, K, wd, sd, g, max_tokens=mt,
                 flags=qg.FLAG_MMA_SYNC_PREFILL)
    x = synth.activations(N, K, seed=30, duplicate_rows=True)
    xd = to_dev(x)
    y = h.run(xd, out_f32=True).cpu().numpy()
    yref, mag = oracle.qgemv(ORTYPE[qtype], w, M, K, x, scales=sc, global_scale=g)
    check_close(y, yref, mag, what=f"edge {qtype} {M}x{K} N={N} max_tokens={mt}")
    if N <= 32 or (0 < mt <= 32):
        one = np.concatenate([h.run(xd[n:n + 1], out_f32=True).cpu().numpy() for n in range(N)])
        assert np.array_equal(y.view(np.uint32), one.view(np.uint32))
    assert h.device_status() == 0
