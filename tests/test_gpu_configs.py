"""Parity at the workloads' full sizes, in the launch configuration the bench
times, on sampled outputs the oracle computes one by one."""
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


def _sample_rows(M, n=64, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, n)]))
    return rows


def test_single_small_gemv_all_rows():
    c = synth.CONFIG0
    h, w, _, _ = make_matrix(c["qtype"], c["M"], c["K"], seed=0)
    x = synth.activations(1, c["K"], seed=0)
    y = h.run(to_dev(x))
    yref, mag = oracle.qgemv(oracle.Q4_K, w, c["M"], c["K"], x)
    check_close(y.float().cpu().numpy(), yref, mag, fp16_out=True, what="config0")


def _layer(seed=0):
    mats = {}
    for i, (role, qt, M, K) in enumerate(synth.LAYER):
        mats[role] = make_matrix(qt, M, K, seed=seed, stream=100 + i)
    return mats


@pytest.mark.parametrize("N", [1, 33, 64, 128])
def test_decode_layer_fused_calls(N):
    """One Qwen3-4B-shaped layer as the bench runs it: QKV triple, Wo with the
    residual add, gate/up pair, down."""
    mats = _layer()
    K = 2560
    x = synth.activations(N, K, seed=1)
    xd = to_dev(x)
    q, k, v = (mats[r][0] for r in ("wq", "wk", "wv"))
    yq, yk, yv = qg.triple_run(q, k, v, xd)
    for role, y in (("wq", yq), ("wk", yk), ("wv", yv)):
        h, w, _, _ = mats[role]
        rows = _sample_rows(h.M, seed=2)
        yref, mag = oracle.qgemv(ORTYPE[h.qtype], w, h.M, K, x, rows=rows)
        check_close(y.float().cpu().numpy()[:, rows], yref, mag, fp16_out=True, what=role)
    ho, wo, _, _ = mats["wo"]
    xo = synth.activations(N, 4096, seed=3)
    r = synth.residual(N, 2560, seed=3)
    yo = ho.run_add(to_dev(xo), to_dev(r))
    rows = _sample_rows(2560, seed=4)
    yref, mag = oracle.qgemv(oracle.Q4_K, wo, 2560, 4096, xo, residual=r, rows=rows)
    check_close(yo.float().cpu().numpy()[:, rows], yref, mag, fp16_out=True, what="wo+res")
    hg, wg, _, _ = mats["gate"]
    hu, wu, _, _ = mats["up"]
    yg, yu = qg.pair_run(hg, hu, xd)
    for h, w, y in ((hg, wg, yg), (hu, wu, yu)):
        rows = _sample_rows(h.M, seed=5)
        yref, mag = oracle.qgemv(oracle.Q4_K, w, h.M, K, x, rows=rows)
        check_close(y.float().cpu().numpy()[:, rows], yref, mag, fp16_out=True, what="pair")
    hd, wd, _, _ = mats["down"]
    xdn = synth.activations(N, 9728, seed=6)
    yd = hd.run(to_dev(xdn))
    rows = _sample_rows(2560, seed=7)
    yref, mag = oracle.qgemv(oracle.Q6_K, wd, 2560, 9728, xdn, rows=rows)
    check_close(yd.float().cpu().numpy()[:, rows], yref, mag, fp16_out=True, what="down")
    for role in mats:
        assert mats[role][0].device_status() == 0, role


@pytest.mark.parametrize("qtype,M,K", synth.SWEEP_SHAPES)
def test_skinny_sweep_full_size(qtype, M, K):
    h, w, _, _ = make_matrix(qtype, M, K, seed=8)
    x = synth.activations(32, K, seed=8, duplicate_rows=True)
    xd = to_dev(x)
    rows = _sample_rows(M, seed=9)
    one = None
    for N in synth.SWEEP_N:
        y = h.run(xd[:N], out_f32=True).cpu().numpy()
        yref, mag = oracle.qgemv(ORTYPE[qtype], w, M, K, x[:N], rows=rows)
        check_close(y[:, rows], yref, mag, what=f"sweep N={N}")
        if one is None:
            one = np.concatenate([h.run(xd[n:n + 1], out_f32=True).cpu().numpy()
                                  for n in range(32)])
        assert np.array_equal(y.view(np.uint32), one[:N].view(np.uint32))


@pytest.mark.parametrize("M,K", synth.NVFP4_SHAPES)
def test_nvfp4_full_size(M, K):
    h, w, sc, g = make_matrix(qg.NVFP4_W4A16, M, K, seed=10)
    x = synth.activations(32, K, seed=10)
    xd = to_dev(x)
    rows = _sample_rows(M, seed=11)
    for N in synth.NVFP4_N:
        y = h.run(xd[:N], out_f32=True).cpu().numpy()
        yref, mag = oracle.qgemv(oracle.NVFP4, w, M, K, x[:N], scales=sc, global_scale=g,
                                 rows=rows)
        check_close(y[:, rows], yref, mag, what=f"nvfp4 {M}x{K} N={N}")


@pytest.mark.parametrize("N", [1, 33, 128])
def test_36_layer_set_as_the_bench_runs_it(N):
    """The decode-layer set the bench times: 36 layers of device-generated
    weights (2.3 GB), each layer's four calls in the bench's form (at N = 1
    one qgemv_chain_run, at N = 33 and 128 the prefill chunks), with device-
    generated x.  Sampled rows of every matrix of every layer against the
    oracle (weights, x and residual copied back from the generators'
    buffers)."""
    t = torch()
    dev = t.device("cuda", 0)
    f16 = t.float16
    ORT = {qg.Q4_K: oracle.Q4_K, qg.Q6_K: oracle.Q6_K}
    xs = {k: synth.device_activations(N, K, 0, s, dev)
          for k, K, s in (("qkv", 2560, 1), ("o", 4096, 2), ("res", 2560, 3), ("ffn", 2560, 4),
                          ("dn", 9728, 5))}
    xh = {k: v.cpu().numpy() for k, v in xs.items()}
    M = {"q": 4096, "k": 1024, "v": 1024, "o": 2560, "g": 9728, "u": 9728, "d": 2560}
    ys = {k: t.empty((N, m), dtype=f16, device=dev) for k, m in M.items()}
    P = lambda v: v.data_ptr()
    chain = qg.Chain()
    out_of = {"wq": ("q", "qkv"), "wk": ("k", "qkv"), "wv": ("v", "qkv"), "wo": ("o", "o"),
              "gate": ("g", "ffn"), "up": ("u", "ffn"), "down": ("d", "dn")}
    rng = np.random.default_rng(36)
    worst = 0.0
    for L in range(36):
        hs, host = {}, {}
        for i, (role, qt, Mr, K) in enumerate(synth.LAYER):
            w, sc, g = synth.device_weights(qt, Mr, K, seed=0, stream=1000 * L + i, device=dev)
            hs[role] = qg.QGemv(qt, Mr, K, w, sc, g, max_tokens=128)
            host[role] = w
        h = {k: v.h for k, v in hs.items()}
        calls = qg.make_calls([
            (qg.CALL_TRIPLE, [h["wq"], h["wk"], h["wv"]], P(xs["qkv"]), N,
             [P(ys["q"]), P(ys["k"]), P(ys["v"])], qg.OUT_F16, None),
            (qg.CALL_RUN_ADD, [h["wo"]], P(xs["o"]), N, [P(ys["o"])], qg.OUT_F16, P(xs["res"])),
            (qg.CALL_PAIR, [h["gate"], h["up"]], P(xs["ffn"]), N, [P(ys["g"]), P(ys["u"])],
             qg.OUT_F16, None),
            (qg.CALL_RUN, [h["down"]], P(xs["dn"]), N, [P(ys["d"])], qg.OUT_F16, None)])
        chain.run(calls)
        t.cuda.synchronize()
        for role, qt, Mr, K in synth.LAYER:
            yk, xk = out_of[role]
            rows = np.unique(np.concatenate([[0, Mr - 1], rng.integers(0, Mr, 3)]))
            wrows = host[role][t.from_numpy(rows).to(dev)].cpu().numpy()
            yref, mag = oracle.qgemv(ORT[qt], wrows, len(rows), K, xh[xk],
                                     residual=xh["res"][:, rows] if role == "wo" else None)
            got = ys[yk].float().cpu().numpy()[:, rows]
            worst = max(worst, check_close(got, yref, mag, fp16_out=True,
                                           what=f"layer {L} {role} N={N}"))
        for v in hs.values():
            assert v.device_status() == 0
        del hs, host
    assert chain.status() == 0
    assert worst <= 1.0
