"""GPU parity of decode chains (qgemv_chain_run), in both forms (one
persistent launch, and one launch per call): every output has the bits of the
same calls issued one by one, each call reads its inputs only after the
earlier calls have written them, and the results agree with the oracle."""
import numpy as np
import pytest

import oracle
from gpu_util import check_close, make_matrix, to_dev, torch
from skinny_gemm_q4_gb300 import qgemv as qg
from skinny_gemm_q4_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from skinny_gemm_q4_gb300 import build
    build.build()
    assert torch().cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(params=[qg.CHAIN_PERSISTENT, 0], ids=["persistent", "launch_per_call"])
def chain_flags(request):
    return request.param


@pytest.fixture(scope="module")
def layer():
    """The decode layer's matrices (Qwen3-4B shapes): Q/K Q4_K, V Q6_K,
    Wo Q4_K, gate/up Q4_K, down Q6_K, with their host bytes."""
    shapes = {"wq": (qg.Q4_K, 4096, 2560), "wk": (qg.Q4_K, 1024, 2560),
              "wv": (qg.Q6_K, 1024, 2560), "wo": (qg.Q4_K, 2560, 4096),
              "gate": (qg.Q4_K, 9728, 2560), "up": (qg.Q4_K, 9728, 2560),
              "down": (qg.Q6_K, 2560, 9728)}
    out = {}
    for i, (name, (qt, M, K)) in enumerate(shapes.items()):
        h, w, _, _ = make_matrix(qt, M, K, seed=40, stream=i + 1)
        out[name] = (h, w)
    return out


def _empty(N, M, f32=False):
    t = torch()
    return t.empty((N, M), dtype=t.float32 if f32 else t.float16, device="cuda")


def _layer_calls(L, xs, ys, N, res, f32):
    odt = qg.OUT_F32 if f32 else qg.OUT_F16
    h = {k: v[0].h for k, v in L.items()}
    return qg.make_calls([
        (qg.CALL_TRIPLE, [h["wq"], h["wk"], h["wv"]], xs["qkv"].data_ptr(), N,
         [ys["q"].data_ptr(), ys["k"].data_ptr(), ys["v"].data_ptr()], odt, None),
        (qg.CALL_RUN_ADD, [h["wo"]], xs["o"].data_ptr(), N, [ys["o"].data_ptr()], qg.OUT_F16,
         res.data_ptr()),
        (qg.CALL_PAIR, [h["gate"], h["up"]], xs["ffn"].data_ptr(), N,
         [ys["g"].data_ptr(), ys["u"].data_ptr()], odt, None),
        (qg.CALL_RUN, [h["down"]], xs["dn"].data_ptr(), N, [ys["d"].data_ptr()], odt, None),
    ])


@pytest.mark.parametrize("N", [1, 3, 8])
def test_layer_chain_equals_separate_calls_and_oracle(layer, N, chain_flags):
    """The four layer calls with independent inputs: one persistent launch,
    each output bit-equal to its own entry point's, and (sampled rows) within
    the oracle tolerance."""
    t = torch()
    f32 = N != 3  # fp16 outputs at N = 3
    xh = {k: synth.activations(N, K, seed=41, stream=s)
          for k, K, s in (("qkv", 2560, 1), ("o", 4096, 2), ("ffn", 2560, 3), ("dn", 9728, 4))}
    xs = {k: to_dev(v) for k, v in xh.items()}
    resh = synth.residual(N, 2560, seed=41)
    res = to_dev(resh)
    M = {"q": 4096, "k": 1024, "v": 1024, "o": 2560, "g": 9728, "u": 9728, "d": 2560}
    ys = {k: _empty(N, m, f32 and k != "o") for k, m in M.items()}
    calls = _layer_calls(layer, xs, ys, N, res, f32)
    ch = qg.Chain(chain_flags)
    ch.run(calls)
    t.cuda.synchronize()
    assert ch.status() == 0

    L = {k: v[0] for k, v in layer.items()}
    sq, sk, sv = qg.triple_run(L["wq"], L["wk"], L["wv"], xs["qkv"], out_f32=f32)
    so = L["wo"].run_add(xs["o"], res)
    sg, su = qg.pair_run(L["gate"], L["up"], xs["ffn"], out_f32=f32)
    sd = L["down"].run(xs["dn"], out_f32=f32)
    t.cuda.synchronize()
    for k, sep in (("q", sq), ("k", sk), ("v", sv), ("o", so), ("g", sg), ("u", su), ("d", sd)):
        assert t.equal(ys[k], sep), k

    rows = {"q": np.arange(0, 4096, 37), "o": np.arange(0, 2560, 23), "g": np.arange(5, 9728, 91),
            "d": np.arange(3, 2560, 29), "v": np.arange(0, 1024, 11)}
    refs = (("q", "wq", oracle.Q4_K, "qkv", None), ("v", "wv", oracle.Q6_K, "qkv", None),
            ("o", "wo", oracle.Q4_K, "o", resh), ("g", "gate", oracle.Q4_K, "ffn", None),
            ("d", "down", oracle.Q6_K, "dn", None))
    for yk, wk, ot, xk, rr in refs:
        hnd, w = layer[wk]
        r = rows[yk]
        yref, mag = oracle.qgemv(ot, w, hnd.M, hnd.K, xh[xk], residual=rr, rows=r)
        got = ys[yk].float().cpu().numpy()[:, r]
        check_close(got, yref, mag, fp16_out=ys[yk].dtype == t.float16, what=f"chain {yk}")


@pytest.mark.parametrize("N", [1, 4])
def test_chain_reads_earlier_outputs(layer, N, chain_flags):
    """Each call consumes the previous call's output (Wo + residual -> gate/up
    pair -> down -> QKV triple).  The intermediate buffers hold NaN before
    every run, so a call that read its x before the earlier call had written
    it would give NaN or other bits; five runs in a row (the counters reset
    between launches) all equal the calls issued one by one."""
    t = torch()
    L = {k: v[0] for k, v in layer.items()}
    h = {k: v.h for k, v in L.items()}
    # tiny inputs keep the chained products finite in fp16 (each call here
    # multiplies magnitudes by 250-900; the last one peaks near 15,000)
    x0 = to_dev((synth.activations(N, 4096, seed=42) * 2.0 ** -23).astype(np.float16))
    res = to_dev((synth.residual(N, 2560, seed=42) * 2.0 ** -17).astype(np.float16))
    M = {"o": 2560, "g": 9728, "u": 9728, "d": 2560, "q": 4096, "k": 1024, "v": 1024}
    ys = {k: _empty(N, m) for k, m in M.items()}
    calls = qg.make_calls([
        (qg.CALL_RUN_ADD, [h["wo"]], x0.data_ptr(), N, [ys["o"].data_ptr()], qg.OUT_F16,
         res.data_ptr()),
        (qg.CALL_PAIR, [h["gate"], h["up"]], ys["o"].data_ptr(), N,
         [ys["g"].data_ptr(), ys["u"].data_ptr()], qg.OUT_F16, None),
        (qg.CALL_RUN, [h["down"]], ys["g"].data_ptr(), N, [ys["d"].data_ptr()], qg.OUT_F16, None),
        (qg.CALL_TRIPLE, [h["wq"], h["wk"], h["wv"]], ys["d"].data_ptr(), N,
         [ys["q"].data_ptr(), ys["k"].data_ptr(), ys["v"].data_ptr()], qg.OUT_F16, None),
    ])
    so = L["wo"].run_add(x0, res)
    sg, su = qg.pair_run(L["gate"], L["up"], so)
    sd = L["down"].run(sg)
    sq, sk, sv = qg.triple_run(L["wq"], L["wk"], L["wv"], sd)
    t.cuda.synchronize()
    for k, v in (("o", so), ("g", sg), ("d", sd), ("q", sq)):
        assert bool(t.isfinite(v).all()) and bool((v != 0).any()), k
    ch = qg.Chain(chain_flags)
    for _ in range(5):
        for v in ys.values():
            v.fill_(float("nan"))
        ch.run(calls)
        t.cuda.synchronize()
        for k, sep in (("o", so), ("g", sg), ("u", su), ("d", sd), ("q", sq), ("k", sk),
                       ("v", sv)):
            assert t.equal(ys[k], sep), k
    assert ch.status() == 0


def test_chain_segments_around_calls_it_does_not_serve(layer, chain_flags):
    """A Q5_K call and an N = 12 call in the middle of a chain run through
    their own entry points between persistent launches; the order and the
    bits stay those of the separate calls."""
    t = torch()
    L = {k: v[0] for k, v in layer.items()}
    q5, _, _, _ = make_matrix(qg.Q5_K, 2560, 2560, seed=43, stream=9)
    N = 2
    # (scaled so the three chained products stay finite in fp16)
    x = to_dev((synth.activations(N, 2560, seed=43) * 2.0 ** -14).astype(np.float16))
    x12 = to_dev(synth.activations(12, 2560, seed=44))
    y = {"g": _empty(N, 9728), "u": _empty(N, 9728), "f": _empty(N, 2560),
         "d": _empty(N, 2560), "w": _empty(12, 1024), "k": _empty(N, 1024), "v": _empty(N, 1024)}
    h = {k: v.h for k, v in L.items()}
    calls = qg.make_calls([
        (qg.CALL_PAIR, [h["gate"], h["up"]], x.data_ptr(), N,
         [y["g"].data_ptr(), y["u"].data_ptr()], qg.OUT_F16, None),
        (qg.CALL_RUN, [q5.h], x.data_ptr(), N, [y["f"].data_ptr()], qg.OUT_F16, None),
        (qg.CALL_RUN, [h["down"]], y["g"].data_ptr(), N, [y["d"].data_ptr()], qg.OUT_F16, None),
        (qg.CALL_RUN, [h["wk"]], x12.data_ptr(), 12, [y["w"].data_ptr()], qg.OUT_F16, None),
        (qg.CALL_RUN, [h["wk"]], y["d"].data_ptr(), N, [y["k"].data_ptr()], qg.OUT_F16, None),
        (qg.CALL_RUN, [h["wv"]], y["d"].data_ptr(), N, [y["v"].data_ptr()], qg.OUT_F16, None),
    ])
    ch = qg.Chain(chain_flags)
    ch.run(calls)
    sg, su = qg.pair_run(L["gate"], L["up"], x)
    sd = L["down"].run(sg)
    sw = L["wk"].run(x12)
    sk = L["wk"].run(sd)
    sv = L["wv"].run(sd)
    sf = q5.run(x)
    t.cuda.synchronize()
    for k, sep in (("g", sg), ("u", su), ("d", sd), ("w", sw), ("k", sk), ("v", sv), ("f", sf)):
        assert bool(t.isfinite(sep).all()), k
        assert t.equal(y[k], sep), k
    assert ch.status() == 0


def test_chain_in_a_graph(layer, chain_flags):
    """Captured once in a CUDA graph and replayed with new inputs copied in
    before each replay: every replay gives the separate calls' bits."""
    t = torch()
    L = {k: v[0] for k, v in layer.items()}
    N = 1
    xs = {k: _empty(N, K) for k, K in (("qkv", 2560), ("o", 4096), ("ffn", 2560), ("dn", 9728))}
    res = _empty(N, 2560)
    M = {"q": 4096, "k": 1024, "v": 1024, "o": 2560, "g": 9728, "u": 9728, "d": 2560}
    ys = {k: _empty(N, m) for k, m in M.items()}
    calls = _layer_calls(layer, xs, ys, N, res, False)
    ch = qg.Chain(chain_flags)
    for k, v in xs.items():
        v.copy_(to_dev(synth.activations(N, v.shape[1], seed=45, stream=len(k))))
    res.copy_(to_dev(synth.residual(N, 2560, seed=45)))
    ch.run(calls)  # warm-up outside the capture
    t.cuda.synchronize()
    side = t.cuda.Stream()
    g = t.cuda.CUDAGraph()
    with t.cuda.stream(side):
        with t.cuda.graph(g, stream=side):
            ch.run(calls)
    for rep in range(3):
        for k, v in xs.items():
            v.copy_(to_dev(synth.activations(N, v.shape[1], seed=46 + rep, stream=len(k))))
        g.replay()
        t.cuda.synchronize()
        sq, sk, sv = qg.triple_run(L["wq"], L["wk"], L["wv"], xs["qkv"])
        so = L["wo"].run_add(xs["o"], res)
        sg, su = qg.pair_run(L["gate"], L["up"], xs["ffn"])
        sd = L["down"].run(xs["dn"])
        t.cuda.synchronize()
        for k, sep in (("q", sq), ("k", sk), ("v", sv), ("o", so), ("g", sg), ("u", su),
                       ("d", sd)):
            assert t.equal(ys[k], sep), (rep, k)
    assert ch.status() == 0


def test_persistent_chain_reports_a_wait_that_runs_out(layer, monkeypatch):
    """Failure detection without a GPU fault: with QGEMV_FAULT_INJECT=
    chain_publish one side of the persistent launch never publishes its
    outputs, so every other side's wait for the earlier calls runs out (about
    half a second each) and sets bit 4 of the chain's error word instead of
    hanging; the next launches are correct and report nothing."""
    t = torch()
    N = 1
    xs = {k: to_dev(synth.activations(N, K, seed=47, stream=s))
          for k, K, s in (("qkv", 2560, 1), ("o", 4096, 2), ("ffn", 2560, 3), ("dn", 9728, 4))}
    res = to_dev(synth.residual(N, 2560, seed=47))
    M = {"q": 4096, "k": 1024, "v": 1024, "o": 2560, "g": 9728, "u": 9728, "d": 2560}
    ys = {k: _empty(N, m) for k, m in M.items()}
    calls = _layer_calls(layer, xs, ys, N, res, False)
    ch = qg.Chain(qg.CHAIN_PERSISTENT)
    monkeypatch.setenv("QGEMV_FAULT_INJECT", "chain_publish")
    ch.run(calls)
    t.cuda.synchronize()
    monkeypatch.delenv("QGEMV_FAULT_INJECT")
    assert ch.status(clear=True) & 4
    assert ch.status() == 0
    ch.run(calls)
    L = {k: v[0] for k, v in layer.items()}
    sq, sk, sv = qg.triple_run(L["wq"], L["wk"], L["wv"], xs["qkv"])
    so = L["wo"].run_add(xs["o"], res)
    sg, su = qg.pair_run(L["gate"], L["up"], xs["ffn"])
    sd = L["down"].run(xs["dn"])
    t.cuda.synchronize()
    for k, sep in (("q", sq), ("k", sk), ("v", sv), ("o", so), ("g", sg), ("u", su), ("d", sd)):
        assert t.equal(ys[k], sep), k
    assert ch.status() == 0


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_chain_run_host_round_trip(layer, pinned):
    """qgemv_chain_run_host: the step's inputs from host memory, the layer's
    calls, every output back to host memory, synchronized.  Page-locked
    buffers go through the SMs' copy kernel, pageable ones through the copy
    engine; both give the device path's bytes."""
    t = torch()
    N = 2
    kin = {"qkv": 2560, "o": 4096, "res": 2560, "ffn": 2560, "dn": 9728}
    kout = {"q": 4096, "k": 1024, "v": 1024, "o": 2560, "g": 9728, "u": 9728, "d": 2560}
    nin, nout = N * sum(kin.values()), N * sum(kout.values())
    hin = t.from_numpy(synth.activations(1, nin, seed=48).reshape(-1))
    hout = t.empty(nout, dtype=t.float16)
    if pinned:
        hin, hout = hin.pin_memory(), hout.pin_memory()
    din = t.empty(nin, dtype=t.float16, device="cuda")
    dout = t.empty(nout, dtype=t.float16, device="cuda")

    def views(buf, sizes):
        out, o = {}, 0
        for k, n in sizes.items():
            out[k] = buf[o:o + N * n].view(N, n)
            o += N * n
        return out
    xs, ys = views(din, kin), views(dout, kout)
    calls = _layer_calls(layer, xs, ys, N, xs["res"], False)
    ch = qg.Chain()
    s = t.cuda.current_stream().cuda_stream
    qg.qgemv_chain_run_host(ch.c, calls, hin.data_ptr(), din.data_ptr(), nin * 2, dout.data_ptr(),
                            hout.data_ptr(), nout * 2, s)
    ref_in = hin.cuda()
    assert t.equal(din, ref_in)
    xr, yr = views(ref_in, kin), views(t.empty_like(dout), kout)
    qg.qgemv_chain_run(ch.c, _layer_calls(layer, xr, yr, N, xr["res"], False), s)
    t.cuda.synchronize()
    ref_out = t.cat([yr[k].reshape(-1) for k in kout])
    assert t.equal(hout, ref_out.cpu())
    assert ch.status() == 0
